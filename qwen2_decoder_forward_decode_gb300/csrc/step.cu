// Persistent decode step: one kernel runs a whole greedy decode step of one sequence of a
// bf16 model ("LLM Speedrun: Architecture", Transformer architecture and Implementing Qwen;
// "augur", Features: greedy generation with a preallocated KV cache).
//
// One CTA per SM, all resident (cooperative launch). Warp 8 of each CTA is a producer: its
// lane 0 walks the step's whole weight schedule (per layer: q/k/v rows, o_proj rows,
// gate/up rows, down rows; then the LM head) and bulk-copies (TMA, 1-D) the CTA's share
// into a ring of shared-memory slots, never waiting for data dependencies, only for free
// slots. Warps 0..7 are consumers: per phase they stage the phase's input vector in shared
// memory, multiply it with the weight units arriving in the ring, write the outputs, and
// meet all other CTAs at a grid barrier before the next phase. The HBM weight stream thus
// keeps running across the 5 dependent phases of every layer.
//
// Phases of a layer: QKV (RMSNorm, projections + bias, split-half RoPE, KV append);
// ATTN (split-context GQA attention partials); OPROJ (merge of the partials, x += Wo o);
// GATEUP (RMSNorm, silu(gate) * up); DOWN (x += Wd a). Then LM (final RMSNorm, logits,
// greedy argmax) and the bookkeeping of token, position and history.
//
// Every wait (ring slots, grid barriers) is bounded; on expiry the kernel raises an abort
// flag that every other wait observes, flags ERR_TIMEOUT, lets its bulk copies land and
// returns.
#include "common.cuh"
#include "internal.h"

#include <math.h>

namespace qw {
namespace step {

constexpr int NCW = 8;                    // consumer warps
constexpr int NPW = 2;                    // producer warps (each issues every NPW-th unit)
constexpr int PF_WARP = NCW + NPW;        // L2 prefetch warp
constexpr int THREADS = (NCW + NPW + 1) * 32;
constexpr int MAXQ = 64;                  // QKV items per CTA whose epilogue inputs are staged
constexpr int NCT = NCW * 32;             // consumer threads
constexpr int SLOT_DEFAULT = 24 * 1024;   // bytes per ring slot (a unit of whole rows)
constexpr int MAX_SLOTS = 16;
constexpr int GMAX = 8;

enum : int { P_QKV = 0, P_ATTN = 1, P_OPROJ = 2, P_GATEUP = 3, P_DOWN = 4, P_LM = 5 };

typedef StepLayer Layer;

struct Params {
  const Layer* layers;
  int L, H, nq, nkv, hd, I, V, cap;
  float eps;
  const bf16 *embed, *final_norm, *head;
  const float2* rope;
  f16* kv;          // this sequence's cache: [L][2][nkv][cap][hd]
  float *x, *q, *act, *logits;
  float* part;      // attention partials [nq][MAX_SPLIT][hd + 2]
  int* tok;
  int* pos;
  unsigned long long* key;
  int *hist, *hist_n;
  int hist_cap;
  unsigned long long* bar;   // monotonic arrival counter (never reset)
  unsigned long long bar_base;  // its value when this launch started
  int* abort;
  int* err;
  int nslots;
  int slot;         // bytes per ring slot (multiple of 16)
  int pf_units;     // L2 prefetch distance ahead of the producers, in units (0: off)
  int xs_floats;    // floats of the staged input vector region
  unsigned long long* tl;  // timeline: per phase [start, end, producer issued] (CTA 0), or null
  int* diag;               // [0..3] first expired wait (site, CTA, warp, detail); then per CTA
                           // the first wait that gave up: [4 + 4c ..] (site, warp, detail, phase)
};

constexpr int MAX_SPLIT = 16;

// A phase's items (one or two weight rows each) are split in contiguous blocks over the
// CTAs. A CTA groups consecutive items of its block into units of whole rows that fit one
// ring slot (one bulk copy per row segment); an item whose rows alone exceed a slot is
// split along K into U chunk units instead.
struct Geo {
  int n_items, rows, K;
  bool paired;   // the two rows of an item come from two segments (RoPE pair, gate/up)
  int cut;       // units never cross multiples of this item index (0: no constraint)
  int ipu;       // items per unit
  int chunk;     // K elements per unit
  int U;         // chunk units per item (1 unless a row exceeds a slot)
};

__device__ __forceinline__ Geo geo(const Params& p, int ph) {
  Geo g;
  g.paired = false;
  g.cut = 0;
  switch (ph) {
    case P_QKV: g.n_items = (p.nq + 2 * p.nkv) * (p.hd / 2); g.rows = 2; g.K = p.H; g.paired = true; g.cut = p.hd / 2; break;
    case P_OPROJ: g.n_items = (p.H + 1) / 2; g.rows = 2; g.K = p.nq * p.hd; break;
    case P_GATEUP: g.n_items = p.I; g.rows = 2; g.K = p.H; g.paired = true; break;
    case P_DOWN: g.n_items = p.H; g.rows = 1; g.K = p.I; break;
    default: g.n_items = (p.V + 1) / 2; g.rows = 2; g.K = p.H; break;
  }
  const int SLOT = p.slot;
  const int item_bytes = g.rows * g.K * 2;
  if (item_bytes <= SLOT) {
    g.ipu = SLOT / item_bytes;
    if (g.ipu > 16) g.ipu = 16;
    g.chunk = g.K;
    g.U = 1;
  } else {
    g.ipu = 1;
    g.chunk = (SLOT / (g.rows * 2)) & ~7;
    g.U = (g.K + g.chunk - 1) / g.chunk;
  }
  return g;
}

// first row of item `item` in segment `seg` (paired ops), else the item's first row
__device__ __forceinline__ const bf16* item_row(const Params& p, const Layer* lw, int ph, int item, int seg) {
  switch (ph) {
    case P_QKV: {
      const int half = p.hd >> 1;
      int head = item / half;
      const int i = item - head * half + seg * half;
      const bf16* m = lw->wq;
      if (head >= p.nq) { head -= p.nq; m = lw->wk; if (head >= p.nkv) { head -= p.nkv; m = lw->wv; } }
      return m + (size_t)(head * p.hd + i) * p.H;
    }
    case P_OPROJ: return lw->wo + (size_t)(2 * item) * p.nq * p.hd;
    case P_GATEUP: return (seg == 0 ? lw->wg : lw->wu) + (size_t)item * p.H;
    case P_DOWN: return lw->wd + (size_t)item * p.I;
    default: return p.head + (size_t)(2 * item) * p.H;
  }
}

// The weight tensor an item row lives in (base, elements), for the copy checks.
__device__ __forceinline__ void item_tensor(const Params& p, const Layer* lw, int ph, int item, int seg,
                                            const bf16*& base, size_t& elems) {
  switch (ph) {
    case P_QKV: {
      const int head = item / (p.hd >> 1);
      if (head < p.nq) { base = lw->wq; elems = (size_t)p.nq * p.hd * p.H; }
      else if (head < p.nq + p.nkv) { base = lw->wk; elems = (size_t)p.nkv * p.hd * p.H; }
      else { base = lw->wv; elems = (size_t)p.nkv * p.hd * p.H; }
      return;
    }
    case P_OPROJ: base = lw->wo; elems = (size_t)p.H * p.nq * p.hd; return;
    case P_GATEUP: base = seg == 0 ? lw->wg : lw->wu; elems = (size_t)p.I * p.H; return;
    case P_DOWN: base = lw->wd; elems = (size_t)p.H * p.I; return;
    default: base = p.head; elems = (size_t)p.V * p.H; return;
  }
}

// rows of the (non-paired) items [i, i + n) that exist: the last pair of an odd-sized
// matrix has one row
__device__ __forceinline__ int consecutive_rows(const Params& p, int ph, const Geo& g, int i, int n) {
  if (g.rows == 1) return n;
  const int N = ph == P_OPROJ ? p.H : p.V;
  return min(2 * n, N - 2 * i);
}

// contiguous item block [i0, i1) of this CTA
__device__ __forceinline__ void item_block(int n_items, int& i0, int& i1) {
  i0 = (int)((long long)blockIdx.x * n_items / gridDim.x);
  i1 = (int)((long long)(blockIdx.x + 1) * n_items / gridDim.x);
}

// length of the unit starting at item i of a block ending at i1
__device__ __forceinline__ int unit_len(const Geo& g, int i, int i1) {
  int len = min(g.ipu, i1 - i);
  if (g.cut) len = min(len, g.cut - i % g.cut);
  return len;
}

// Calls fn(seq, phase, layer weights, geometry, first item, items, chunk) for every unit
// of this CTA in stream order (per layer: QKV, OPROJ, GATEUP, DOWN; then LM) until fn
// returns false.
template <class Fn>
__device__ __forceinline__ void walk_units(const Params& p, Fn&& fn) {
  long long seq = 0;
  for (int l = 0; l <= p.L; ++l) {
    for (int ph = 0; ph < 5; ++ph) {
      int phase = ph;
      if (l == p.L) {
        if (ph > 0) break;
        phase = P_LM;
      } else if (ph == P_ATTN) {
        continue;
      }
      const Geo g = geo(p, phase);
      const Layer* lw = p.layers + (l < p.L ? l : 0);
      int i0, i1;
      item_block(g.n_items, i0, i1);
      for (int i = i0; i < i1;) {
        const int len = unit_len(g, i, i1);
        for (int u = 0; u < g.U; ++u, ++seq)
          if (!fn(seq, l, phase, lw, g, i, len, u)) return;
        i += len;
      }
    }
  }
}

__device__ __forceinline__ bool aborted(const Params& p) { return *(volatile int*)p.abort != 0; }

enum : int {
  SITE_SLOT_FULL = 1,
  SITE_SLOT_EMPTY = 2,
  SITE_GRID = 3,
  SITE_COPY = 4,
  SITE_SMEM = 5,
  SITE_STORE = 6,
  SITE_SLOT_REUSE = 7
};

// Per CTA, the first wait that gave up (expired, or saw another CTA's abort).
__device__ __forceinline__ void note_giveup(const Params& p, int site, long long detail) {
  if (!p.diag) return;
  int* d = p.diag + 4 + 4 * blockIdx.x;
  if (atomicCAS(d, 0, site) == 0) {
    d[1] = threadIdx.x >> 5;
    d[2] = (int)detail;
  }
}
// First expiry wins the global record; every later wait sees the abort flag.
__device__ __forceinline__ void raise_abort(const Params& p, int site, long long detail) {
  if (atomicExch(p.abort, 1) == 0 && p.diag) {
    p.diag[0] = site;
    p.diag[1] = blockIdx.x;
    p.diag[2] = threadIdx.x >> 5;
    p.diag[3] = (int)detail;
  }
  note_giveup(p, site, detail);
  atomicOr(p.err, ERR_TIMEOUT);
}

// Bulk copy with its source checked against the weight tensor it must lie in and its
// destination against the ring; a violation is recorded, the copy skipped, and the launch
// aborted (so no wait is left hanging on the missing bytes).
__device__ __forceinline__ bool checked_copy(const Params& p, uint32_t dst, const bf16* src, uint32_t bytes,
                                             uint32_t bar, const bf16* tbase, size_t telems, uint32_t ring_lo,
                                             uint32_t ring_hi, long long detail) {
  const bool ok = bytes > 0 && (bytes & 15) == 0 && ((uintptr_t)src & 15) == 0 && (dst & 15) == 0 &&
                  src >= tbase && src + bytes / 2 <= tbase + telems && dst >= ring_lo && dst + bytes <= ring_hi;
  if (!ok) {
    raise_abort(p, SITE_COPY, detail);
    return false;
  }
  bulk_copy_g2s(dst, src, bytes, bar);
  return true;
}

// Bounded wait (non-blocking tests) that also gives up when another CTA has aborted.
__device__ __forceinline__ bool slot_wait(const Params& p, uint32_t bar, uint32_t parity, int site,
                                          long long detail) {
  if (mbar_test_now(bar, parity)) return true;
  const long long t0 = clock64();
  for (int it = 0;; ++it) {
    if (mbar_test_now(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (aborted(p)) {
        note_giveup(p, site + 10, detail);
        return false;
      }
      if (clock64() - t0 > WAIT_CYCLES) {
        raise_abort(p, site, detail);
        return false;
      }
    }
  }
}

// A consumer may test a slot's full barrier for unit seq only once the slot's previous unit
// (seq - NS) has been released: before that the barrier is still in the previous unit's
// phase, whose parity is the opposite one, and the parity test would pass at once. With
// fewer slots than consumer warps that previous unit belongs to another warp, so the
// releases are published per slot in shared memory (monotonic: a slot's units are
// released in order, each copy waiting for the previous release).
__device__ __forceinline__ bool reuse_wait(const Params& p, const volatile int* rel, int want, long long detail) {
  if (*rel >= want) return true;
  const long long t0 = clock64();
  for (int it = 0;; ++it) {
    if (*rel >= want) return true;
    if ((it & 63) == 0) {
      if (aborted(p)) {
        note_giveup(p, SITE_SLOT_REUSE + 10, detail);
        return false;
      }
      if (clock64() - t0 > WAIT_CYCLES) {
        raise_abort(p, SITE_SLOT_REUSE, detail);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void cbar() {  // consumer warps only (named barrier 1)
  asm volatile("bar.sync 1, %0;" ::"r"(NCT) : "memory");
}
// consumer barrier that also ANDs a predicate over all consumer threads
__device__ __forceinline__ bool cbar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\t"
      "setp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, 1, %2, a;\n\t"
      "selp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(NCT)
      : "memory");
  return r != 0;
}

// Grid barrier among the consumers of all CTAs: every CTA adds one to a monotonic 64-bit
// counter and waits until it reaches this barrier's target (launch base + (b + 1) * CTAs).
__device__ bool grid_barrier(const Params& p, int& b) {
  __shared__ int s_ok;
  cbar();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    atomicAdd(p.bar, 1ull);
    const unsigned long long target = p.bar_base + (unsigned long long)(b + 1) * gridDim.x;
    const long long t0 = clock64();
    for (int it = 0;; ++it) {
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p.bar) : "memory");
      if (v >= target) break;
      if ((it & 15) == 0 && (aborted(p) || clock64() - t0 > WAIT_CYCLES)) {
        if (!aborted(p)) raise_abort(p, SITE_GRID, b);
        else note_giveup(p, SITE_GRID + 10, (long long)b * 100000 + (long long)(v - p.bar_base));
        ok = 0;
        break;
      }
    }
    s_ok = ok && !aborted(p);
  }
  ++b;
  cbar();
  return s_ok != 0;
}

// xs = x * rsqrt(mean(x^2) + eps) * gain  (consumers; x from global, H % 4 == 0)
__device__ void stage_norm(const Params& p, float* xs, float* scratch, const float* x, const bf16* gain, int H) {
  const int ct = threadIdx.x;
  const int n4 = H >> 2;
  float ss = 0.f;
  for (int base = ct; base < n4; base += 4 * NCT) {
    float4 v[4];
    uint2 g[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = base + i * NCT;
      v[i] = j < n4 ? __ldcg(reinterpret_cast<const float4*>(x) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      g[i] = j < n4 ? __ldg(reinterpret_cast<const uint2*>(gain) + j) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = base + i * NCT;
      if (j < n4) {
        reinterpret_cast<float4*>(xs)[j] = v[i];
        reinterpret_cast<uint2*>(xs + H)[j] = g[i];  // gains parked behind x
        ss = fmaf(v[i].x, v[i].x, fmaf(v[i].y, v[i].y, fmaf(v[i].z, v[i].z, fmaf(v[i].w, v[i].w, ss))));
      }
    }
  }
  // block sum over consumer threads
  ss = warp_sum(ss);
  if ((ct & 31) == 0) scratch[ct >> 5] = ss;
  cbar();
  float t = 0.f;
  for (int i = 0; i < NCW; ++i) t += scratch[i];
  const float inv = rsqrtf(t / (float)H + p.eps);
  for (int j = ct; j < n4; j += NCT) {
    float4 v = reinterpret_cast<float4*>(xs)[j];
    const uint2 g = reinterpret_cast<const uint2*>(xs + H)[j];
    v.x = v.x * inv * bf_lo(g.x);
    v.y = v.y * inv * bf_hi(g.x);
    v.z = v.z * inv * bf_lo(g.y);
    v.w = v.w * inv * bf_hi(g.y);
    reinterpret_cast<float4*>(xs)[j] = v;
  }
  cbar();
}

__device__ void stage_copy(float* xs, const float* src, int n) {
  const int ct = threadIdx.x;
  const int n4 = n >> 2;
  for (int base = ct; base < n4; base += 8 * NCT) {
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = base + i * NCT;
      v[i] = j < n4 ? __ldcg(reinterpret_cast<const float4*>(src) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = base + i * NCT;
      if (j < n4) reinterpret_cast<float4*>(xs)[j] = v[i];
    }
  }
  cbar();
}

// x (fp32, global) = E[tok]; xs = norm(x) * gain. Every CTA builds xs itself; CTA 0 also
// writes the residual stream.
__device__ void stage_embed(const Params& p, float* xs, float* scratch, const bf16* gain) {
  const int ct = threadIdx.x;
  int t = __ldcg(p.tok);
  if (t < 0 || t >= p.V) {
    if (ct == 0 && blockIdx.x == 0) atomicOr(p.err, ERR_TOKEN);
    t = 0;
  }
  const uint4* row = reinterpret_cast<const uint4*>(p.embed + (size_t)t * p.H);
  float ss = 0.f;
  for (int v = ct; v < p.H / 8; v += NCT) {
    const uint4 w = __ldg(row + v);
    const float f[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y), bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      xs[v * 8 + e] = f[e];
      ss = fmaf(f[e], f[e], ss);
    }
    if (blockIdx.x == 0) {
      reinterpret_cast<float4*>(p.x)[2 * v] = make_float4(f[0], f[1], f[2], f[3]);
      reinterpret_cast<float4*>(p.x)[2 * v + 1] = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
  ss = warp_sum(ss);
  if ((ct & 31) == 0) scratch[ct >> 5] = ss;
  cbar();
  float tot = 0.f;
  for (int i = 0; i < NCW; ++i) tot += scratch[i];
  const float inv = rsqrtf(tot / (float)p.H + p.eps);
  for (int k = ct; k < p.H; k += NCT) xs[k] = xs[k] * inv * __bfloat162float(gain[k]);
  cbar();
}

// Softmax partial of one (KV head, context chunk) for the G query heads of the head, in
// tiles of 64 positions with running max / sum (online softmax); written to p.part.
__device__ void attention_partial(const Params& p, float* xs, const f16* kc, const f16* vc, int ctx,
                                  int nsplit) {
  const int ct = threadIdx.x, warp = ct >> 5, lane = ct & 31;
  const int G = p.nq / p.nkv, hd = p.hd;
  const int g = blockIdx.x / nsplit, sp = blockIdx.x - g * nsplit;
  const int chunk = (ctx + nsplit - 1) / nsplit;
  const int j0 = sp * chunk, j1 = min(ctx, j0 + chunk);
  // shared: q [G][hd] f32 | scores [G][64] | running (m, l) [G][2] | tile corr [G] |
  //         K, V tiles [64][hd] f16
  float* qs = xs;
  float* sc = qs + G * hd;
  float* run = sc + G * 64;
  float* corr = run + 2 * G;
  f16* ks = reinterpret_cast<f16*>(xs + ((G * hd + G * 64 + 3 * G + 3) & ~3));  // 16-byte aligned
  f16* vs = ks + 64 * hd;
  {
    const float4* qsrc = reinterpret_cast<const float4*>(p.q + (size_t)g * G * hd);
    float4 r[GMAX * 128 / 4 / NCT];
#pragma unroll
    for (int i = 0; i < GMAX * 128 / 4 / NCT; ++i) {
      const int jv = ct + i * NCT;
      r[i] = jv < G * hd / 4 ? __ldcg(qsrc + jv) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < GMAX * 128 / 4 / NCT; ++i) {
      const int jv = ct + i * NCT;
      if (jv < G * hd / 4) reinterpret_cast<float4*>(qs)[jv] = r[i];
    }
  }
  if (ct < G) {
    run[2 * ct] = -INFINITY;
    run[2 * ct + 1] = 0.f;
  }
  constexpr int EPT = GMAX * 128 / NCT;  // output elements of [G][hd] per consumer thread
  float o[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) o[e] = 0.f;
  const float scale = rsqrtf((float)hd);
  for (int t0 = j0; t0 < j1; t0 += 64) {
    const int n = min(64, j1 - t0);
    const int kvv = n * hd / 8;  // 16-byte vectors per tile of K (and of V)
    const uint4* ksrc = reinterpret_cast<const uint4*>(kc + ((size_t)g * p.cap + t0) * hd);
    const uint4* vsrc = reinterpret_cast<const uint4*>(vc + ((size_t)g * p.cap + t0) * hd);
    cbar();  // previous tile fully used (and q, run initialised)
    for (int b0 = ct; b0 < 2 * kvv; b0 += 8 * NCT) {
      uint4 r[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int jv = b0 + i * NCT;
        if (jv < kvv) r[i] = __ldcg(ksrc + jv);
        else if (jv < 2 * kvv) r[i] = __ldcg(vsrc + (jv - kvv));
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int jv = b0 + i * NCT;
        if (jv < kvv) reinterpret_cast<uint4*>(ks)[jv] = r[i];
        else if (jv < 2 * kvv) reinterpret_cast<uint4*>(vs)[jv - kvv] = r[i];
      }
    }
    cbar();
    for (int jj = warp; jj < n; jj += NCW) {  // scores: a warp per position
      float part[GMAX];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) part[h] = 0.f;
      for (int dd = lane; dd < hd; dd += 32) {
        const float kv = __half2float(ks[jj * hd + dd]);
#pragma unroll
        for (int h = 0; h < GMAX; ++h)
          if (h < G) part[h] = fmaf(qs[h * hd + dd], kv, part[h]);
      }
#pragma unroll
      for (int h = 0; h < GMAX; ++h)
        if (h < G) {
          const float sv = warp_sum(part[h]);
          if (lane == 0) sc[h * 64 + jj] = sv * scale;
        }
    }
    cbar();
    for (int h = warp; h < G; h += NCW) {  // running max and sum of head h
      float m = -INFINITY;
      for (int jj = lane; jj < n; jj += 32) m = fmaxf(m, sc[h * 64 + jj]);
      m = warp_max(m);
      const float m_old = run[2 * h];
      const float m_new = fmaxf(m_old, m);
      float ls = 0.f;
      for (int jj = lane; jj < n; jj += 32) {
        const float pr = expf(sc[h * 64 + jj] - m_new);
        sc[h * 64 + jj] = pr;
        ls += pr;
      }
      ls = warp_sum(ls);
      if (lane == 0) {
        const float c = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
        corr[h] = c;
        run[2 * h] = m_new;
        run[2 * h + 1] = run[2 * h + 1] * c + ls;
      }
    }
    cbar();
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int idx = ct + e * NCT;
      if (idx < G * hd) {
        const int h = idx / hd, dd = idx - h * hd;
        float acc = o[e] * corr[h];
        for (int jj = 0; jj < n; ++jj) acc = fmaf(sc[h * 64 + jj], __half2float(vs[jj * hd + dd]), acc);
        o[e] = acc;
      }
    }
  }
  cbar();
  const int pstride = hd + 2;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int idx = ct + e * NCT;
    if (idx < G * hd) {
      const int h = idx / hd, dd = idx - h * hd;
      p.part[((size_t)(g * G + h) * MAX_SPLIT + sp) * pstride + dd] = o[e];
    }
  }
  if (ct < G) {
    float* pp = p.part + ((size_t)(g * G + ct) * MAX_SPLIT + sp) * pstride;
    pp[hd] = run[2 * ct];
    pp[hd + 1] = run[2 * ct + 1];
  }
}

// xs[0, nq*hd) = attention output: per head, the chunk partials merged exactly
// (out = sum_s exp(m_s - M) O_s / sum_s exp(m_s - M) l_s).
__device__ void merge_partials(const Params& p, float* xs, int nsplit) {
  const int ct = threadIdx.x;
  const int hd = p.hd, nq = p.nq, pstride = hd + 2;
  float* wts = xs + nq * hd;  // [nq][MAX_SPLIT] merge weights
  for (int i = ct; i < nq * nsplit; i += NCT) {
    const int h = i / nsplit, s = i - h * nsplit;
    wts[h * MAX_SPLIT + s] = __ldcg(p.part + ((size_t)h * MAX_SPLIT + s) * pstride + hd);  // m_s
  }
  cbar();
  if (ct < nq) {
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, wts[ct * MAX_SPLIT + s]);
    float L = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float wv = expf(wts[ct * MAX_SPLIT + s] - M);
      wts[ct * MAX_SPLIT + s] = wv;
      L = fmaf(__ldcg(p.part + ((size_t)ct * MAX_SPLIT + s) * pstride + hd + 1), wv, L);
    }
    const float inv = 1.f / L;
    for (int s = 0; s < nsplit; ++s) wts[ct * MAX_SPLIT + s] *= inv;
  }
  cbar();
  for (int idx0 = ct; idx0 < nq * hd; idx0 += 4 * NCT) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < nsplit; s0 += 4) {
      float v[4][4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int idx = idx0 + k * NCT;
        const int h = idx / hd, dd = idx - h * hd;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          v[k][u] = (idx < nq * hd && s0 + u < nsplit)
                        ? __ldcg(p.part + ((size_t)h * MAX_SPLIT + s0 + u) * pstride + dd)
                        : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int idx = idx0 + k * NCT;
        const int h = idx / hd;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (idx < nq * hd && s0 + u < nsplit) acc[k] = fmaf(v[k][u], wts[h * MAX_SPLIT + s0 + u], acc[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = idx0 + k * NCT;
      if (idx < nq * hd) xs[idx] = acc[k];
    }
  }
  cbar();
}

// ---- the kernel ----------------------------------------------------------------------------

__global__ void __launch_bounds__(THREADS, 1) decode_step_kernel(const Params p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ __align__(8) unsigned long long full[MAX_SLOTS], empty[MAX_SLOTS];
  __shared__ float scratch[32];
  __shared__ unsigned long long s_key[NCW];
  __shared__ int s_bad[NCW];
  __shared__ int rel[MAX_SLOTS];  // per slot: sequence number of the last released unit
  __shared__ long long s_issued;  // last unit producer 0 issued (paces the prefetch warp)
  __shared__ float4 s_qkv_epi[MAXQ];  // QKV items of this CTA: (bias a, bias b, cos, sin)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = p.nslots;
  const int SLOT = p.slot;
  float* xs = reinterpret_cast<float*>(dsm + (size_t)NS * SLOT);
  const uint32_t ring = smem_addr(dsm);
  const uint32_t full0 = smem_addr(full), empty0 = smem_addr(empty);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
      rel[s] = -1;
    }
    s_issued = -1;
    mbar_fence_init();
  }
  __syncthreads();
  const int pos = __ldcg(p.pos);  // the token of this step sits at position pos

  // ---------------- L2 prefetch warp ----------------
  if (warp == PF_WARP) {
    // Walks the same schedule up to pf_units units ahead of producer 0 and asks L2 for
    // each unit's rows, so the HBM stream runs on while the consumers are in phases that
    // move little data (attention, barriers). Advisory: it gives up silently.
    if (lane != 0 || p.pf_units <= 0) return;
    walk_units(p, [&](long long seq, int, int phase, const Layer* lw, const Geo& g, int i, int len, int u) {
      if (seq > *(volatile long long*)&s_issued + p.pf_units) {
        const long long t0 = clock64();
        while (seq > *(volatile long long*)&s_issued + p.pf_units) {
          if (aborted(p) || clock64() - t0 > WAIT_CYCLES) return false;
        }
      }
      const uint32_t rb = (uint32_t)g.K * 2;
      if (g.U == 1) {
        if (g.paired) {
          prefetch_l2_bulk(item_row(p, lw, phase, i, 0), (uint32_t)len * rb);
          prefetch_l2_bulk(item_row(p, lw, phase, i, 1), (uint32_t)len * rb);
        } else {
          prefetch_l2_bulk(item_row(p, lw, phase, i, 0), (uint32_t)consecutive_rows(p, phase, g, i, len) * rb);
        }
      } else {
        const int k0 = u * g.chunk;
        const uint32_t b = (uint32_t)min(g.chunk, g.K - k0) * 2;
        prefetch_l2_bulk(item_row(p, lw, phase, i, 0) + k0, b);
        if (g.paired) prefetch_l2_bulk(item_row(p, lw, phase, i, 1) + k0, b);
        else if (g.rows == 2 && consecutive_rows(p, phase, g, i, 1) == 2)
          prefetch_l2_bulk(item_row(p, lw, phase, i, 0) + (size_t)g.K + k0, b);
      }
      return true;
    });
    return;
  }

  // ---------------- producers ----------------
  if (warp >= NCW) {
    // Producer warp pw issues the units whose sequence number is pw mod NPW (NS is a
    // multiple of NPW, so its units always land in its own slots). Copies from one thread
    // are processed one after another, so whole-row units (up to 24 KB) and two issuing
    // warps keep the stream at full bandwidth.
    if (lane != 0) return;
    const int pw = warp - NCW;
    long long last = -1;
    bool ok = !aborted(p);
    if (ok) walk_units(p, [&](long long seq, int l, int phase, const Layer* lw, const Geo& g, int i, int len, int u) {
      if ((int)(seq % NPW) != pw) return true;
      const int s = (int)(seq % NS);
      if (p.tl && blockIdx.x == 0 && pw == 0) {  // ring occupancy statistics (profiling)
        p.tl[3 * (5 * p.L + 1) + 0] += 1;
        if (seq >= NS && !mbar_test_now(empty0 + 8 * s, (uint32_t)(((seq / NS) - 1) & 1)))
          p.tl[3 * (5 * p.L + 1) + 1] += 1;
      }
      if (seq >= NS && !slot_wait(p, empty0 + 8 * s, (uint32_t)(((seq / NS) - 1) & 1), SITE_SLOT_EMPTY, seq)) {
        ok = false;
        return false;
      }
      const uint32_t rb = (uint32_t)g.K * 2;  // bytes of a full row
      const uint32_t bar = full0 + 8 * s;
      const uint32_t dst = ring + s * SLOT;
      const uint32_t rlo = ring, rhi = ring + (uint32_t)NS * SLOT;
      const bf16* tb0;
      const bf16* tb1;
      size_t te0, te1;
      item_tensor(p, lw, phase, i, 0, tb0, te0);
      item_tensor(p, lw, phase, i, 1, tb1, te1);
      const long long dt = seq * 1000 + phase;
      bool cok = true;
      if (g.U == 1) {
        if (g.paired) {
          const uint32_t b = (uint32_t)len * rb;
          mbar_expect_tx(bar, 2 * b);
          cok = checked_copy(p, dst, item_row(p, lw, phase, i, 0), b, bar, tb0, te0, rlo, rhi, dt) &&
                checked_copy(p, dst + (uint32_t)g.ipu * rb, item_row(p, lw, phase, i, 1), b, bar, tb1, te1,
                             rlo, rhi, dt);
        } else {
          const uint32_t b = (uint32_t)consecutive_rows(p, phase, g, i, len) * rb;
          mbar_expect_tx(bar, b);
          cok = checked_copy(p, dst, item_row(p, lw, phase, i, 0), b, bar, tb0, te0, rlo, rhi, dt);
        }
      } else {  // one item, K chunk u
        const int k0 = u * g.chunk;
        const uint32_t b = (uint32_t)min(g.chunk, g.K - k0) * 2;
        const bf16* r0 = item_row(p, lw, phase, i, 0) + k0;
        const bf16* r1 = nullptr;
        if (g.paired) r1 = item_row(p, lw, phase, i, 1) + k0;
        else if (g.rows == 2 && consecutive_rows(p, phase, g, i, 1) == 2) r1 = r0 + g.K;
        mbar_expect_tx(bar, b * (r1 ? 2u : 1u));
        cok = checked_copy(p, dst, r0, b, bar, tb0, te0, rlo, rhi, dt);
        if (cok && r1)
          cok = checked_copy(p, dst + (uint32_t)g.chunk * 2, r1, b, bar, g.paired ? tb1 : tb0, g.paired ? te1 : te0,
                             rlo, rhi, dt);
      }
      if (!cok) {
        ok = false;
        return false;
      }
      last = seq;
      if (pw == 0) *(volatile long long*)&s_issued = seq;
      if (p.tl && blockIdx.x == 0 && pw == 0) p.tl[3 * (l == p.L ? 5 * p.L : 5 * l + phase) + 2] = gtime();
      return true;
    });
    // let every copy this warp issued land before the CTA may finish
    for (long long k = last - NS + 1 > 0 ? last - NS + 1 : 0; k <= last; ++k) {
      if ((int)(k % NPW) != pw) continue;
      const int s = (int)(k % NS);
      const long long t0 = clock64();
      while (!mbar_test_now(full0 + 8 * s, (uint32_t)((k / NS) & 1)) && clock64() - t0 < WAIT_CYCLES) {
      }
    }
    if (pw == 0 && ok) *(volatile long long*)&s_issued = 1ll << 60;  // release the prefetch warp
    return;
  }

  // ---------------- consumers ----------------
  const int ct = threadIdx.x;
  int gen = 0;  // barriers passed in this launch
  long long base = 0;  // ring sequence number of the current phase's first unit
  const int half = p.hd >> 1;
  const int G = p.nq / p.nkv;
  float best_v = -INFINITY;
  int best_i = -1;
  bool nonfinite = false;

  int phase_no = 0;
  auto stamp = [&](int which) {  // CTA 0: [start, end] of consumer phase phase_no
    if (p.tl && blockIdx.x == 0 && ct == 0) p.tl[3 * phase_no + which] = gtime();
  };
  auto substamp = [&](int which) {  // CTA 0: [input staged, first unit ready, units done]
    if (p.tl && blockIdx.x == 0 && ct == 0) p.tl[3 * (5 * p.L + 2 + phase_no) + which] = gtime();
  };
  // consume one weight phase: warp w takes every NCW-th unit of this CTA's block; per item
  // it reduces the rows (over the chunk units of the item when K was split) and runs the
  // epilogue
  auto run_phase = [&](int phase, int l, auto&& epilogue) -> bool {
    const Geo g = geo(p, phase);
    int i0, i1;
    item_block(g.n_items, i0, i1);
    const size_t rb = (size_t)g.K * 2;
    bool ok = true;
    long long seq = base;
    int unit = 0;
    for (int i = i0; i < i1; ++unit) {
      const int len = unit_len(g, i, i1);
      if (unit % NCW == warp && ok) {
        float a0 = 0.f, a1 = 0.f;
        for (int u = 0; u < g.U; ++u) {
          const long long sq = seq + u;
          const int s = (int)(sq % NS);
          if (p.tl && blockIdx.x == 0 && threadIdx.x == 0 &&
              !mbar_test_now(full0 + 8 * s, (uint32_t)((sq / NS) & 1)))
            p.tl[3 * (5 * p.L + 1) + 2] += 1;
          if (sq >= NS && !__all_sync(0xffffffffu, reuse_wait(p, rel + s, (int)(sq - NS), sq))) {
            ok = false;
            break;
          }
          if (!__all_sync(0xffffffffu, slot_wait(p, full0 + 8 * s, (uint32_t)((sq / NS) & 1), SITE_SLOT_FULL, sq))) {
            ok = false;
            break;
          }
          if (unit == 0 && u == 0) substamp(1);
          const unsigned char* slot = dsm + (size_t)s * SLOT;
          {  // the rows this unit reads must lie inside its slot, x inside the staged vector
            const size_t need = g.U == 1 ? (g.paired ? (size_t)(g.ipu + len) * rb : (size_t)g.rows * len * rb)
                                         : (size_t)g.rows * g.chunk * 2;
            const int xneed = g.U == 1 ? g.K : u * g.chunk + min(g.chunk, g.K - u * g.chunk);
            if (need > (size_t)SLOT || xneed > p.xs_floats) {
              if (lane == 0) raise_abort(p, SITE_SMEM, sq * 1000 + phase);
              ok = false;
              break;
            }
          }
          float e0 = 0.f, e1 = 0.f;
          if (g.U == 1) {  // whole rows of len items
            const int nv = g.K >> 3;
            const float4* x4 = reinterpret_cast<const float4*>(xs);
            for (int t = 0; t < len; ++t) {
              const uint4* w0;
              const uint4* w1;
              if (g.paired) {
                w0 = reinterpret_cast<const uint4*>(slot + t * rb);
                w1 = reinterpret_cast<const uint4*>(slot + g.ipu * rb + t * rb);
              } else {
                w0 = reinterpret_cast<const uint4*>(slot + (size_t)g.rows * t * rb);
                w1 = reinterpret_cast<const uint4*>(slot + ((size_t)g.rows * t + 1) * rb);
              }
              float b0 = 0.f, b1 = 0.f;
#pragma unroll 4
              for (int v = lane; v < nv; v += 32) {
                const float4 xa = x4[2 * v], xb = x4[2 * v + 1];
                const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
                b0 = dotv(w0[v], xv, b0, bf16());
                if (g.rows == 2) b1 = dotv(w1[v], xv, b1, bf16());
              }
              b0 = warp_sum(b0);
              if (g.rows == 2) b1 = warp_sum(b1);
              if (lane == t) {  // lane t keeps item t; the epilogues run side by side below
                e0 = b0;
                e1 = b1;
              }
            }
          } else {  // chunk u of one item
            const int k0 = u * g.chunk;
            const int nv = min(g.chunk, g.K - k0) >> 3;
            const uint4* w0 = reinterpret_cast<const uint4*>(slot);
            const uint4* w1 = reinterpret_cast<const uint4*>(slot + (size_t)g.chunk * 2);
            const float4* x4 = reinterpret_cast<const float4*>(xs + k0);
#pragma unroll 4
            for (int v = lane; v < nv; v += 32) {
              const float4 xa = x4[2 * v], xb = x4[2 * v + 1];
              const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
              a0 = dotv(w0[v], xv, a0, bf16());
              if (g.rows == 2) a1 = dotv(w1[v], xv, a1, bf16());
            }
          }
          __syncwarp();
          if (lane == 0) {
            *(volatile int*)(rel + s) = (int)sq;
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty0 + 8 * s) : "memory");
          }
          if (g.U == 1 && lane < len) epilogue(i + lane, e0, e1);
        }
        if (ok && g.U > 1) {
          a0 = warp_sum(a0);
          if (g.rows == 2) a1 = warp_sum(a1);
          if (lane == 0) epilogue(i, a0, a1);
        }
      }
      seq += g.U;
      i += len;
    }
    base = seq;
    substamp(2);  // warp 0 done with its units
    return ok;
  };

  bool ok = !aborted(p);  // a failed earlier launch leaves the model unusable: return fast
  for (int l = 0; l < p.L && ok; ++l) {
    const Layer& w = p.layers[l];
    f16* kc = p.kv + (size_t)l * 2 * p.nkv * p.cap * p.hd;
    f16* vc = kc + (size_t)p.nkv * p.cap * p.hd;
    // ---- QKV
    stamp(0);
    int q0, q1;  // this CTA's QKV items; their bias pairs and rotations are staged first
    item_block((p.nq + 2 * p.nkv) * half, q0, q1);
    auto qkv_epi = [&](int item) -> float4 {
      const int head = item / half, i = item - head * half;
      const bf16* bias;
      int h;
      if (head < p.nq) { bias = w.bq; h = head; }
      else if (head < p.nq + p.nkv) { bias = w.bk; h = head - p.nq; }
      else { bias = w.bv; h = head - p.nq - p.nkv; }
      float4 e = make_float4(0.f, 0.f, 1.f, 0.f);
      if (bias) {
        e.x = __bfloat162float(bias[h * p.hd + i]);
        e.y = __bfloat162float(bias[h * p.hd + i + half]);
      }
      if (head < p.nq + p.nkv && pos >= 0 && pos < p.cap) {
        const float2 cs = p.rope[(size_t)pos * half + i];
        e.z = cs.x;
        e.w = cs.y;
      }
      return e;
    };
    if (ct < q1 - q0 && ct < MAXQ) s_qkv_epi[ct] = qkv_epi(q0 + ct);  // published by the norm's barriers
    if (l == 0) stage_embed(p, xs, scratch, w.in_norm);
    else stage_norm(p, xs, scratch, p.x, w.in_norm, p.H);
    substamp(0);
    ok = run_phase(P_QKV, l, [&](int item, float a, float b) {
      int head = item / half;
      const int i = item - head * half;
      int h;
      if (head < p.nq) h = head;
      else if (head < p.nq + p.nkv) h = head - p.nq;
      else h = head - p.nq - p.nkv;
      if (item < q0 || item >= q1 || pos < 0 || pos >= p.cap) {
        raise_abort(p, SITE_STORE, item);
        return;
      }
      const float4 e = item - q0 < MAXQ ? s_qkv_epi[item - q0] : qkv_epi(item);
      a += e.x;
      b += e.y;
      if (head < p.nq + p.nkv) {
        const float ra = a * e.z - b * e.w, rb = b * e.z + a * e.w;
        a = ra;
        b = rb;
      }
      if (head < p.nq) {
        p.q[h * p.hd + i] = a;
        p.q[h * p.hd + i + half] = b;
      } else {
        f16* dst = (head < p.nq + p.nkv ? kc : vc) + ((size_t)h * p.cap + pos) * p.hd;
        dst[i] = __float2half_rn(a);
        dst[i + half] = __float2half_rn(b);
      }
    }) && ok;
    ok = cbar_and(ok);
    stamp(1);
    ++phase_no;
    if (!(ok = ok && grid_barrier(p, gen))) break;

    // ---- ATTN: CTA (g, sp) holds the softmax partial of KV head g over positions
    //      [sp * chunk, (sp + 1) * chunk) for its G query heads
    const int ctx = pos + 1;
    int nsplit = (ctx + 63) / 64;
    if (nsplit > MAX_SPLIT) nsplit = MAX_SPLIT;
    stamp(0);
    if ((int)blockIdx.x < p.nkv * nsplit) attention_partial(p, xs, kc, vc, ctx, nsplit);
    stamp(1);
    ++phase_no;
    if (!(ok = grid_barrier(p, gen))) break;

    // ---- OPROJ: merge the partials into xs = attention output, then x += Wo . xs
    stamp(0);
    merge_partials(p, xs, nsplit);
    substamp(0);
    ok = cbar_and(run_phase(P_OPROJ, l, [&](int item, float a, float b) {
      if (item < 0 || 2 * item >= p.H) { raise_abort(p, SITE_STORE, 100000 + item); return; }
      atomicAdd(p.x + 2 * item, a);
      if (2 * item + 1 < p.H) atomicAdd(p.x + 2 * item + 1, b);
    }));
    stamp(1);
    ++phase_no;
    if (!(ok = ok && grid_barrier(p, gen))) break;

    // ---- GATEUP
    stamp(0);
    stage_norm(p, xs, scratch, p.x, w.post_norm, p.H);
    substamp(0);
    ok = cbar_and(run_phase(P_GATEUP, l, [&](int item, float gt, float up) {
      if (item < 0 || item >= p.I) { raise_abort(p, SITE_STORE, 200000 + item); return; }
      p.act[item] = (gt / (1.f + expf(-gt))) * up;
    }));
    stamp(1);
    ++phase_no;
    if (!(ok = ok && grid_barrier(p, gen))) break;

    // ---- DOWN
    stamp(0);
    stage_copy(xs, p.act, p.I);
    substamp(0);
    ok = cbar_and(run_phase(P_DOWN, l, [&](int item, float a, float) {
      if (item < 0 || item >= p.H) { raise_abort(p, SITE_STORE, 300000 + item); return; }
      atomicAdd(p.x + item, a);
    }));
    stamp(1);
    ++phase_no;
    if (!(ok = ok && grid_barrier(p, gen))) break;
  }

  // ---- LM head: logits and the greedy argmax (lowest index among equal maxima)
  if (ok) {
    stamp(0);
    stage_norm(p, xs, scratch, p.x, p.final_norm, p.H);
    substamp(0);
    auto take = [&](int r, float v) {
      if (r < 0 || r >= p.V) { raise_abort(p, SITE_STORE, 400000 + r); return; }
      p.logits[r] = v;
      if (!isfinite(v)) nonfinite = true;
      if (v > best_v || best_i < 0) {  // a lane sees its rows in increasing order
        best_v = v;
        best_i = r;
      }
    };
    ok = cbar_and(run_phase(P_LM, p.L, [&](int item, float a, float b) {
      take(2 * item, a);
      if (2 * item + 1 < p.V) take(2 * item + 1, b);
    }));
    {  // every lane kept the best of its own rows (seen in increasing order): warp maximum
      unsigned long long k = best_i >= 0 ? argmax_key(best_v, best_i) : 0ull;
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, k, o);
        k = other > k ? other : k;
      }
      const bool bad = __any_sync(0xffffffffu, nonfinite);
      if (lane == 0) {
        s_key[warp] = k;
        s_bad[warp] = bad;
      }
    }
    cbar();
    if (ct == 0) {
      unsigned long long k = 0;
      int bad = 0;
      for (int i = 0; i < NCW; ++i) {
        k = s_key[i] > k ? s_key[i] : k;
        bad |= s_bad[i];
      }
      if (k) atomicMax(p.key, k);
      if (bad) atomicOr(p.err, ERR_NONFINITE);
    }
    stamp(1);
    ok = ok && grid_barrier(p, gen);
    if (ok && blockIdx.x == 0 && ct == 0) {
      const unsigned long long k = atomicAdd(p.key, 0ull);
      const int idx = argmax_key_index(k);
      *p.tok = idx;
      if (p.hist) {
        const int n = __ldcg(p.hist_n);
        if (n < p.hist_cap) p.hist[n] = idx;
        *p.hist_n = n + 1;
      }
      *p.pos = pos + 1;
      *p.key = 0ull;
    }
  }
}

}  // namespace step

// ---- host ----------------------------------------------------------------------------------

int step_xs_floats(const Dims& d) {
  const int G = d.nq / d.nkv;
  int n = d.I;                                        // down projection input
  if (2 * d.H > n) n = 2 * d.H;                       // normalised x + parked gains
  if (d.nq * d.hd > n) n = d.nq * d.hd;
  const int attn = ((G * d.hd + G * 64 + 3 * G + 3) & ~3) + 64 * d.hd;  // attention tile
  if (attn > n) n = attn;
  const int merge = d.nq * d.hd + d.nq * step::MAX_SPLIT;
  if (merge > n) n = merge;
  return (n + 31) & ~31;
}

int step_barriers_per_launch(const Dims& d) { return 5 * d.L + 1; }

bool step_kernel_supported(const Dims& d) {
  return d.dtype == 1 && d.hd <= 128 && d.hd % 8 == 0 && d.nq / d.nkv <= step::GMAX &&
         d.H % 8 == 0 && d.I % 8 == 0 && (size_t)step_xs_floats(d) * 4 + 4 * step::SLOT_DEFAULT <= 224 * 1024;
}

size_t step_part_bytes(const Dims& d) {
  return (size_t)d.nq * step::MAX_SPLIT * (d.hd + 2) * sizeof(float);
}

// Ring geometry: slots of slot_bytes (0: the default) filling the shared memory left
// beside the staged vector, an even number of them (one half per producer warp).
cudaError_t step_set_attributes(const Dims& d, int slot_bytes, int* slot_out, int* nslots_out, size_t* smem_out) {
  const size_t xs = (size_t)step_xs_floats(d) * 4;
  int slot = slot_bytes > 0 ? slot_bytes & ~15 : step::SLOT_DEFAULT;
  if (slot < 4096) slot = 4096;
  int ns = (int)((224 * 1024 - xs) / slot);
  if (ns > step::MAX_SLOTS) ns = step::MAX_SLOTS;
  ns -= ns % step::NPW;
  if (ns < 2) return cudaErrorInvalidValue;
  const size_t smem = (size_t)ns * slot + xs;
  *slot_out = slot;
  *nslots_out = ns;
  *smem_out = smem;
  return cudaFuncSetAttribute(step::decode_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_step(const StepLaunch& a, cudaStream_t s) {
  step::Params p{};
  p.layers = (const step::Layer*)a.layers_dev;
  p.L = a.d.L; p.H = a.d.H; p.nq = a.d.nq; p.nkv = a.d.nkv; p.hd = a.d.hd; p.I = a.d.I; p.V = a.d.V;
  p.cap = a.d.cap; p.eps = a.d.eps;
  p.embed = (const bf16*)a.embed; p.final_norm = (const bf16*)a.final_norm; p.head = (const bf16*)a.head;
  p.rope = a.rope; p.kv = (f16*)a.kv_seq;
  p.x = a.x; p.q = a.q; p.act = a.act; p.logits = a.logits; p.part = a.part;
  p.tok = a.tok; p.pos = a.pos; p.key = a.key; p.hist = a.hist; p.hist_n = a.hist_n; p.hist_cap = a.hist_cap;
  p.bar = a.bar; p.bar_base = a.bar_base; p.abort = a.abort; p.err = a.err;
  p.nslots = a.nslots; p.slot = a.slot; p.pf_units = a.pf_units; p.xs_floats = step_xs_floats(a.d);
  p.tl = a.tl;
  p.diag = a.diag;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(step::THREADS);
  cfg.dynamicSmemBytes = a.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step::decode_step_kernel, p);
}

}  // namespace qw
