// Persistent decode step of one sequence of a bf16 model: one cooperative launch runs the
// whole greedy decode step ("LLM Speedrun: Architecture", Transformer architecture and
// Implementing Qwen: embedding, per layer RMSNorm -> q/k/v with bias -> split-half RoPE ->
// KV append -> GQA attention -> o_proj + residual -> RMSNorm -> gate/up -> SwiGLU -> down +
// residual, then the final RMSNorm, the LM head and the greedy argmax; "augur", Features:
// preallocated KV cache, greedy generation).
//
// Why one kernel: a decode token streams every weight once (HBM-bound) through five
// dependent phases per layer. Launched as separate kernels, the HBM stream stops at every
// phase boundary and ramps up again. Here every CTA (one per SM) owns a ring of shared-memory
// slots that its producer warps keep filling with the weights of the phases ahead, in the
// order they will be used, without waiting for any data dependency; only the consumer warps
// wait for the phase inputs (grid barriers). So the HBM stream keeps running while the
// consumers go through the latency-bound q/k/v -> attention -> o_proj chain.
//
// Work split, per phase, in contiguous blocks over the CTAs (block b of n items is
// [b n / G, (b + 1) n / G)):
//   QKV     RoPE pairs (rows i and i + hd/2 of a head)     units: up to R/2 pairs of a head
//   ATTN    (KV head, context chunk) per CTA               no weights
//   OPROJ   rows of Wo                                     units: up to R rows
//   GATEUP  items i (gate row i, up row i)                 units: up to R/2 items
//   DOWN    rows of Wd (K = intermediate)                  units: one row, K split 8 ways
//   LM      rows of the LM head                            units: up to R rows
// R = rows of hidden elements per ring slot (8 for hidden 1536). Each unit is one or two
// 1-D bulk copies (TMA) into a slot. All eight consumer warps read every unit: in the row
// phases warp w takes row w of the unit (the input vector in registers), in DOWN warp w
// takes the w-th eighth of the row. Row results go to shared memory; after the phase each
// CTA applies its epilogue (bias + RoPE + KV append, residual adds, SwiGLU, logits and
// argmax) and meets the other CTAs at a grid barrier.
//
// Every wait is bounded: on expiry the kernel raises an abort flag that every other wait
// observes, sets ERR_TIMEOUT, lets its own copies land and returns.
#include "common.cuh"
#include "internal.h"

#include <math.h>

#include <algorithm>
#include <cstring>

namespace qw {
namespace mk {

constexpr int NCW = 8;                     // consumer warps
constexpr int NPW = 4;                     // producer warps (lane 0 of each issues copies)
constexpr int NCT = NCW * 32;              // consumer threads
constexpr int THREADS = (NCW + NPW) * 32;
constexpr int NS = 8;                      // ring slots (a multiple of NPW)
constexpr int SLOT = 24 * 1024;            // bytes per slot
constexpr int MAXV = 8;                    // 16-byte vectors per lane of the register tile, at most
constexpr int MAX_LOCAL = 128;             // items of one phase per CTA
constexpr int NSPLIT = 16;                 // most chunks per KV head merged by every o_proj CTA
constexpr int NSPLIT_MAX = 64;             // most attention chunks per KV head
constexpr int MAX_KV_GROUPS = 16;          // KV heads with an attention arrival counter
constexpr int CHUNK_MIN = 32;              // fewest positions per chunk
constexpr int AT_K = 32;                   // positions per attention tile
constexpr int GMAX = 8;                    // most query heads per KV head
constexpr int XS_FLOATS = 2048;            // staged input vector (hidden <= 2048)


enum : int { P_QKV = 0, P_ATTN = 1, P_OPROJ = 2, P_GATEUP = 3, P_DOWN = 4, P_LM = 5 };

struct LayerW {
  const bf16 *in_norm, *wq, *wk, *wv, *bq, *bk, *bv, *wo, *post_norm, *wg, *wu, *wd;
};

// Shared-memory layout (byte offsets from the 1024-aligned base), sized for the model.
struct Layout {
  uint32_t att, xs, da, db, dp, qe, xo, lt, bar, scr, total;
};
__host__ __device__ inline uint32_t align16(uint32_t v) { return (v + 15u) & ~15u; }
inline Layout make_layout(int hd, int H, int nq, int L) {
  Layout o;
  uint32_t off = (uint32_t)NS * SLOT;  // the ring
  o.att = off; off += align16(2u * AT_K * (hd + 8) * 2);  // K and V tiles (the combine reuses them)
  o.xs = off; off += align16((uint32_t)H * 4);
  o.da = off; off += MAX_LOCAL * 4;
  o.db = off; off += MAX_LOCAL * 4;
  o.dp = off; off += 64 * NCW * 4;                       // DOWN partials [rows][warps]
  o.qe = off; off += MAX_LOCAL * 4 * 4;                  // per q/k/v pair: bias a, bias b, cos, sin
  o.xo = off; off += 64 * 4;                             // this CTA's residual rows
  o.lt = off; off += align16((uint32_t)L * sizeof(LayerW));  // the layer pointer table
  o.bar = off; off += 2 * NS * 8;
  o.scr = off; off += 64 * 4;
  o.total = off + 1024;  // base alignment
  return o;
}

struct Params {
  const LayerW* layers;      // device array [L]
  int L, H, nq, nkv, I, V, cap;
  float eps;
  const bf16 *embed, *final_norm, *head;
  const float2* rope;        // [cap][hd/2] (cos, sin)
  f16* kv;                   // this sequence's cache [L][2][nkv][cap][hd]
  float *x, *q, *act, *logits, *part;  // x [H], act [I], part [nq][nsplit][hd + 4]
  float* att_o;              // [nq * hd] attention output merged by the attention CTAs (ns > NSPLIT)
  int nsplit;                // most chunks per KV head (<= NSPLIT_MAX, nkv * nsplit <= CTAs)
  unsigned long long* att_cnt;   // [nkv] monotonic arrival counters of the attention CTAs
  unsigned long long* att_base;  // [nkv] their values when a step starts (updated by CTA 0)
  int *tok, *pos;
  unsigned long long* key;   // packed argmax key (zero between steps)
  int *hist, *hist_n;
  int hist_cap;
  unsigned long long* bar;   // monotonic arrival counter
  unsigned long long* bar_base;  // its value when a step starts (updated by CTA 0 at the end)
  int* abort;                // nonzero: a wait gave up somewhere
  int* err;
  unsigned long long* tl;    // timeline: per phase [start, units done, end] (CTA 0), or null
  int pf_mode;               // when the MLP rows are asked into L2: 0 never, 1 attention start,
                             // 2 o_proj start, 3 when the producers reach them
  Layout lay;
};


__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"r"(NCT) : "memory"); }
// consumer barrier that also ANDs a predicate over every consumer thread
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

__device__ __forceinline__ bool aborted(const Params& p) { return *(volatile int*)p.abort != 0; }

__device__ __forceinline__ void raise_abort(const Params& p) {
  atomicExch(p.abort, 1);
  atomicOr(p.err, ERR_TIMEOUT);
}

// Bounded wait on an mbarrier phase that also gives up once the launch has aborted.
__device__ __forceinline__ bool slot_wait(const Params& p, uint32_t bar, uint32_t parity) {
  if (mbar_test_now(bar, parity)) return true;
  const long long t0 = clock64();
  for (int it = 0;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 31) == 31) {
      if (aborted(p)) return false;
      if (clock64() - t0 > WAIT_CYCLES) {
        raise_abort(p);
        return false;
      }
    }
  }
}

// block [i0, i1) of n items for this CTA
__device__ __forceinline__ void block_of(int n, int& i0, int& i1) {
  i0 = (int)((long long)blockIdx.x * n / gridDim.x);
  i1 = (int)((long long)(blockIdx.x + 1) * n / gridDim.x);
}

// rows of hidden (K = H) elements per slot, even, at most one per consumer warp
__device__ __forceinline__ int rows_per_slot(int H) {
  int r = SLOT / (2 * H);
  r &= ~1;
  return r > NCW ? NCW : r;
}

struct Unit {
  const unsigned char* src[2];
  uint32_t bytes[2];
  uint32_t off2;  // slot offset of the second copy
  int a, n;       // first item (pair, row) and count
};

// Calls f(unit) for each unit of phase ph of layer l for this CTA, in stream order, until f
// returns false; returns false in that case.
template <class F>
__device__ __forceinline__ bool phase_units(const Params& p, const LayerW* lt, int hd, int l, int ph, F&& f) {
  const int R = rows_per_slot(p.H);
  const size_t rowH = (size_t)p.H * 2;  // bytes of a row of K = H
  const LayerW& w = lt[l < p.L ? l : 0];
  int i0, i1;
  Unit u;
  u.bytes[1] = 0;
  u.src[1] = nullptr;
  u.off2 = 0;
  switch (ph) {
    case P_QKV: {
      const int half = hd >> 1;
      block_of((p.nq + 2 * p.nkv) * half, i0, i1);
      for (int a = i0; a < i1;) {
        const int head = a / half, i = a - head * half;
        int n = min(min(R / 2, i1 - a), half - i);
        const bf16* m;
        int hrow;
        if (head < p.nq) { m = w.wq; hrow = head * hd; }
        else if (head < p.nq + p.nkv) { m = w.wk; hrow = (head - p.nq) * hd; }
        else { m = w.wv; hrow = (head - p.nq - p.nkv) * hd; }
        u.src[0] = reinterpret_cast<const unsigned char*>(m + (size_t)(hrow + i) * p.H);
        u.src[1] = reinterpret_cast<const unsigned char*>(m + (size_t)(hrow + half + i) * p.H);
        u.bytes[0] = u.bytes[1] = (uint32_t)(n * rowH);
        u.off2 = (uint32_t)((R / 2) * rowH);
        u.a = a;
        u.n = n;
        if (!f(u)) return false;
        a += n;
      }
      return true;
    }
    case P_OPROJ:
    case P_LM: {
      const int N = ph == P_OPROJ ? p.H : p.V;
      const bf16* m = ph == P_OPROJ ? w.wo : p.head;
      block_of(N, i0, i1);
      for (int a = i0; a < i1;) {
        const int n = min(R, i1 - a);
        u.src[0] = reinterpret_cast<const unsigned char*>(m + (size_t)a * p.H);
        u.bytes[0] = (uint32_t)(n * rowH);
        u.bytes[1] = 0;
        u.a = a;
        u.n = n;
        if (!f(u)) return false;
        a += n;
      }
      return true;
    }
    case P_GATEUP: {
      block_of(p.I, i0, i1);
      for (int a = i0; a < i1;) {
        const int n = min(R / 2, i1 - a);
        u.src[0] = reinterpret_cast<const unsigned char*>(w.wg + (size_t)a * p.H);
        u.src[1] = reinterpret_cast<const unsigned char*>(w.wu + (size_t)a * p.H);
        u.bytes[0] = u.bytes[1] = (uint32_t)(n * rowH);
        u.off2 = (uint32_t)((R / 2) * rowH);
        u.a = a;
        u.n = n;
        if (!f(u)) return false;
        a += n;
      }
      return true;
    }
    case P_DOWN: {
      block_of(p.H, i0, i1);
      for (int a = i0; a < i1; ++a) {
        u.src[0] = reinterpret_cast<const unsigned char*>(w.wd + (size_t)a * p.I);
        u.bytes[0] = (uint32_t)p.I * 2;
        u.bytes[1] = 0;
        u.a = a;
        u.n = 1;
        if (!f(u)) return false;
      }
      return true;
    }
    default: return true;
  }
}

// attention chunking for a context of ctx positions: at most nsplit chunks per KV head of at
// least CHUNK_MIN positions. Up to NSPLIT chunks the o_proj CTAs merge them while staging
// their input; beyond, the attention CTAs of a KV head merge them (below).
__device__ __forceinline__ void att_chunks(int ctx, int nsplit, int& chunk, int& ns) {
  chunk = max(CHUNK_MIN, (ctx + nsplit - 1) / nsplit);
  ns = (ctx + chunk - 1) / chunk;
}

// SM clock stamp idx (< 8) of phase k (CTA 0, thread 0), a plain store
__device__ __forceinline__ void ck(const Params& p, int k, int idx) {
  if (p.tl && blockIdx.x == 0 && threadIdx.x == 0) p.tl[9 * (5 * p.L + 1) + 5 * gridDim.x + 8 * k + idx] = clock64();
}

// L2 requests of this CTA's gate, up and down rows of layer l (they are read by the ring
// later; asking early keeps HBM streaming while the consumers are in the attention chain)
__device__ __forceinline__ void mlp_l2_ahead(const Params& p, const LayerW& w) {
  int a0, a1;
  block_of(p.I, a0, a1);
  if (a1 > a0) {
    const uint32_t gb = (uint32_t)(a1 - a0) * p.H * 2;
    prefetch_l2_bulk(w.wg + (size_t)a0 * p.H, gb);
    prefetch_l2_bulk(w.wu + (size_t)a0 * p.H, gb);
  }
  block_of(p.H, a0, a1);
  if (a1 > a0) prefetch_l2_bulk(w.wd + (size_t)a0 * p.I, (uint32_t)(a1 - a0) * p.I * 2);
}

// ---- producers -----------------------------------------------------------------------

template <int HD>
__device__ void producer(const Params& p, const LayerW* lt, unsigned char* smem, uint32_t full0, uint32_t empty0,
                         int pw, int ctx) {
  long long u = 0;                 // unit counter (same sequence as the consumers')
  long long last_mine[NS / NPW];   // most recent unit issued into each of my slots
  for (int i = 0; i < NS / NPW; ++i) last_mine[i] = -1;
  bool ok = true;
  const uint32_t ring = smem_addr(smem);
  int chunk, ns;
  att_chunks(ctx, p.nsplit, chunk, ns);
  auto issue = [&](const Unit& un) -> bool {
    const long long my = u++;
    if ((int)(my % NPW) != pw) return true;
    const int s = (int)(my % NS);
    if (my >= NS) {  // the slot's previous unit (also mine) has been read by every consumer
      if (!slot_wait(p, empty0 + 8 * s, (uint32_t)(((my / NS) - 1) & 1))) return false;
      fence_proxy_async();
    }
    const uint32_t total = un.bytes[0] + un.bytes[1];
    // copies stay inside the slot, start 16-byte aligned and move multiples of 16 bytes
    if (total == 0 || total > SLOT || (un.bytes[0] & 15) || (un.bytes[1] & 15) ||
        un.off2 + un.bytes[1] > SLOT || (un.bytes[1] && un.off2 < un.bytes[0])) {
      raise_abort(p);
      return false;
    }
    const uint32_t dst = ring + (uint32_t)s * SLOT;
    mbar_expect_tx(full0 + 8 * s, total);
    bulk_copy_g2s(dst, un.src[0], un.bytes[0], full0 + 8 * s);
    if (un.bytes[1]) bulk_copy_g2s(dst + un.off2, un.src[1], un.bytes[1], full0 + 8 * s);
    last_mine[s / NPW] = my;
    return true;
  };
  for (int l = 0; l <= p.L && ok; ++l) {
    if (l < p.L) {
      // this CTA's attention chunk of layer l: its rows written by earlier steps into L2
      if (pw == 0 && (int)blockIdx.x < p.nkv * ns) {
        const int g = blockIdx.x / ns, c = blockIdx.x - g * ns;
        const int j0 = c * chunk, j1 = min(ctx - 1, j0 + chunk);  // the newest row is written this step
        if (j1 > j0) {
          const f16* kc = p.kv + (size_t)l * 2 * p.nkv * p.cap * HD;
          const size_t off = ((size_t)g * p.cap + j0) * HD;
          const uint32_t bytes = (uint32_t)(j1 - j0) * HD * 2;
          prefetch_l2_bulk(kc + off, bytes);
          prefetch_l2_bulk(kc + (size_t)p.nkv * p.cap * HD + off, bytes);
        }
      }
      const LayerW& w = lt[l];
      if (pw == 0) {  // small per-layer vectors every CTA reads (a few CTAs ask for them)
        const uint32_t hb = (uint32_t)p.H * 2;
        switch (blockIdx.x) {
          case 0: prefetch_l2_bulk(w.in_norm, hb); break;
          case 1: prefetch_l2_bulk(w.post_norm, hb); break;
          case 2: if (w.bq) prefetch_l2_bulk(w.bq, (uint32_t)p.nq * HD * 2); break;
          case 3: if (w.bk) prefetch_l2_bulk(w.bk, (uint32_t)p.nkv * HD * 2); break;
          case 4: if (w.bv) prefetch_l2_bulk(w.bv, (uint32_t)p.nkv * HD * 2); break;
          case 5: if (l == 0) prefetch_l2_bulk(p.rope + (size_t)(ctx - 1) * (HD / 2), HD * 4); break;
          default: break;
        }
      }
      const int phs[4] = {P_QKV, P_OPROJ, P_GATEUP, P_DOWN};
      for (int k = 0; k < 4 && ok; ++k) {
        if (phs[k] == P_GATEUP && pw == 0 && p.pf_mode == 3) mlp_l2_ahead(p, w);
        ok = phase_units(p, lt, HD, l, phs[k], issue);
        if (ok && aborted(p)) ok = false;
      }
    } else {
      if (pw == 0 && blockIdx.x == 0) prefetch_l2_bulk(p.final_norm, (uint32_t)p.H * 2);
      ok = phase_units(p, lt, HD, l, P_LM, issue);
    }
  }
  // copies in flight land before the CTA may exit (they were all consumed unless aborted)
  for (int i = 0; i < NS / NPW; ++i) {
    const long long m = last_mine[i];
    if (m >= 0) slot_wait(p, full0 + 8 * (int)(m % NS), (uint32_t)((m / NS) & 1));
  }
}

// ---- consumer helpers ----------------------------------------------------------------

// dot of this warp's vectors of a row held in a slot (16-byte vectors of bf16) with the input
// vector in registers: lane l takes vectors v_lo + l + 32 q < v_hi; one independent 8-term
// chain per vector, added pairwise, then the warp reduction
template <int NV>
__device__ __forceinline__ float row_dot(const uint4* r, const float (&xr)[NV][8], int v_lo, int v_hi, int lane) {
  float part[NV];
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    const int v = v_lo + lane + 32 * q;
    part[q] = v < v_hi ? dotv(r[v], xr[q], 0.f, bf16()) : 0.f;
  }
#pragma unroll
  for (int st = 1; st < NV; st *= 2)
#pragma unroll
    for (int q = 0; q + st < NV; q += 2 * st) part[q] += part[q + st];
  return warp_sum(part[0]);
}

// input vector of the row phases from the staged xs (floats) into registers: lane l holds
// vectors l, l + 32, ... (8 floats each); two 16-byte shared loads per vector, lanes with bit
// 2 set taking the halves in the other order (conflict-free)
template <int NV>
__device__ __forceinline__ void load_xr(float (&xr)[NV][8], const float* xs, int nvec, int lane) {
  const bool sw = (lane & 4) != 0;
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    const int v = lane + 32 * q;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (v < nvec) {
      const float4* s = reinterpret_cast<const float4*>(xs) + 2 * v;
      a = s[sw ? 1 : 0];
      b = s[sw ? 0 : 1];
    }
    const float4 lo = sw ? b : a, hi = sw ? a : b;
    xr[q][0] = lo.x; xr[q][1] = lo.y; xr[q][2] = lo.z; xr[q][3] = lo.w;
    xr[q][4] = hi.x; xr[q][5] = hi.y; xr[q][6] = hi.z; xr[q][7] = hi.w;
  }
}

// xs = gain * src over H elements (consumer threads, each element once per CTA), src the
// residual (written by other CTAs: read through L2) or, when erow is given, the bf16 embedding
// row; each warp's sum of squares goes to scr. After the one consumer barrier every thread
// can take its slice of xs into registers and norm_scale(scr) gives 1 / sqrt(mean(src^2) +
// eps), by which the row results are scaled.
__device__ void stage_gain(const Params& p, float* xs, float* scr, const float* src, const bf16* erow,
                           const bf16* gain, float4* extra_dst = nullptr, float4 extra = float4{}) {
  const int t = threadIdx.x;
  const int n4 = p.H >> 2;
  float4 v[2];
  uint2 g[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {  // every load first
    const int j = t + i * NCT;
    v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    g[i] = make_uint2(0u, 0u);
    if (j < n4) {
      if (erow) {
        const uint2 e = __ldg(reinterpret_cast<const uint2*>(erow) + j);
        v[i] = make_float4(bf_lo(e.x), bf_hi(e.x), bf_lo(e.y), bf_hi(e.y));
      } else {
        v[i] = __ldcg(reinterpret_cast<const float4*>(src) + j);
      }
      g[i] = __ldg(reinterpret_cast<const uint2*>(gain) + j);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int j = t + i * NCT;
    ss = fmaf(v[i].x, v[i].x, fmaf(v[i].y, v[i].y, fmaf(v[i].z, v[i].z, fmaf(v[i].w, v[i].w, ss))));
    if (j < n4)
      reinterpret_cast<float4*>(xs)[j] = make_float4(v[i].x * bf_lo(g[i].x), v[i].y * bf_hi(g[i].x),
                                                     v[i].z * bf_lo(g[i].y), v[i].w * bf_hi(g[i].y));
  }
  ss = warp_sum(ss);
  if ((t & 31) == 0) scr[t >> 5] = ss;
  if (extra_dst) *extra_dst = extra;  // (a value loaded earlier, published by the same barrier)
  cbar();
}
__device__ __forceinline__ float norm_scale(const Params& p, const float* scr) {
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < NCW; ++i) tot += scr[i];  // fixed order: deterministic
  return rsqrtf(tot / (float)p.H + p.eps);
}

// Grid barrier of the consumers of all CTAs: each CTA adds one to a monotonic counter and
// waits until it reaches base + nb * CTAs. ok is this thread's status; the result (the same
// for every consumer thread of the CTA) is false if any consumer thread of the CTA, or any
// CTA's wait, gave up.
__device__ bool grid_sync(const Params& p, unsigned long long base, int& nb, int* s_flag, int k, bool ok) {
  const bool all_ok = cbar_and(ok);
  ++nb;
  if (threadIdx.x == 0) {
    int res = 0;
    if (all_ok && !aborted(p)) {
      // release: this CTA's writes of the phase (ordered before by the consumer barrier)
      asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p.bar), "l"(1ull) : "memory");
      if (p.tl) {
        const unsigned long long now = gtime();
        atomicMax(p.tl + 3 * (5 * p.L + 1 + k) + 2, now);  // the last CTA's arrival
        if (k >= 5 && k < 10)  // every CTA's arrival after the phases of layer 1
          p.tl[9 * (5 * p.L + 1) + (k - 5) * gridDim.x + blockIdx.x] = now;
      }
      const unsigned long long target = base + (unsigned long long)nb * gridDim.x;
      const long long t0 = clock64();
      res = 1;
      for (int it = 0;; ++it) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p.bar) : "memory");
        if (v >= target) break;
        if ((it & 15) == 15) {
          if (aborted(p)) { res = 0; break; }
          if (clock64() - t0 > WAIT_CYCLES) { raise_abort(p); res = 0; break; }
        }
      }
    }
    *s_flag = res;
    if (p.tl && blockIdx.x == 0) p.tl[3 * (5 * p.L + 1 + k) + 1] = gtime();
  }
  cbar();
  return *(volatile int*)s_flag != 0;
}

__device__ __forceinline__ void tl_mark(const Params& p, int k, int which) {
  if (p.tl && blockIdx.x == 0 && threadIdx.x == 0) p.tl[3 * k + which] = gtime();
}
// second timeline record of phase k: [0] input staged, [1] barrier passed (CTA 0), [2] the
// last CTA's arrival at the barrier after the phase
__device__ __forceinline__ void tl_mark2(const Params& p, int k) {
  if (p.tl && blockIdx.x == 0 && threadIdx.x == 0) p.tl[3 * (5 * p.L + 1 + k)] = gtime();
}
// third record of phase k: [0] first unit consumed, [1] epilogue start, [2] epilogue end
__device__ __forceinline__ void tl_mark3(const Params& p, int k, int which) {
  if (p.tl && blockIdx.x == 0 && threadIdx.x == 0) p.tl[3 * (2 * (5 * p.L + 1) + k) + which] = gtime();
}


// ---- attention of one (KV head, chunk) -----------------------------------------------------
//
// Tiles of AT_K positions: all consumer threads copy the K and V rows (cp.async, rows padded
// by 16 bytes); warps 0 and 1 each take 16 positions with mma.sync m16n8k16 (the G query
// heads of the KV head are the rows of the A operand, fp16 q scaled by 1/sqrt(hd)), keeping a
// running maximum and sum per row; the two warps' states are combined into the chunk's
// partial (unnormalised output, maximum, sum), which the o_proj phase merges.
// Copies of tile tt's K and V rows into the tile buffers (cp.async; rows past the chunk are
// zero). With skip_newest the newest position of the context (written by this step's q/k/v
// phase) is left out: the first tile's other rows were written by earlier steps and are
// requested before the grid barrier.
template <int HD>
__device__ __forceinline__ void att_tile_load(f16* Ks, f16* Vs, const f16* kc, const f16* vc, int tt, int n,
                                              int newest, bool skip_newest) {
  constexpr int KS = HD + 8;
  constexpr int NV = AT_K * HD / 8;  // 16-byte vectors of a K (or V) tile
  for (int i = threadIdx.x; i < 2 * NV; i += NCT) {
    const int which = i >= NV, idx = i - which * NV;
    const int j = idx / (HD / 8), c8 = idx - j * (HD / 8);
    f16* dst = (which ? Vs : Ks) + j * KS + c8 * 8;
    const int key = tt * AT_K + j;
    if (key >= n) *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    else if (!(skip_newest && key == newest)) cp_async16(dst, (which ? vc : kc) + (size_t)key * HD + c8 * 8);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int HD>
__device__ __forceinline__ void att_rows(const Params& p, int l, int g, int c, int chunk, int ctx, const f16*& kc,
                                         const f16*& vc, int& n, int& newest) {
  const int j0 = c * chunk, j1 = min(ctx, j0 + chunk);
  n = j1 - j0;
  newest = j1 == ctx ? n - 1 : -1;  // chunk-relative position of the newest row, if in this chunk
  kc = p.kv + (size_t)l * 2 * p.nkv * p.cap * HD + ((size_t)g * p.cap + j0) * HD;
  vc = kc + (size_t)p.nkv * p.cap * HD;
}

// the first tile's rows written by earlier steps, before the grid barrier
template <int HD>
__device__ void attention_preload(const Params& p, unsigned char* att, int l, int g, int c, int chunk, int ctx) {
  f16* Ks = reinterpret_cast<f16*>(att);
  f16* Vs = Ks + AT_K * (HD + 8);
  const f16 *kc, *vc;
  int n, newest;
  att_rows<HD>(p, l, g, c, chunk, ctx, kc, vc, n, newest);
  att_tile_load<HD>(Ks, Vs, kc, vc, 0, n, newest, true);
}

template <int HD>
__device__ void attention_chunk(const Params& p, unsigned char* att, int l, int g, int c, int chunk, int ctx) {
  constexpr int KS = HD + 8, NKK = HD / 16, NNT = HD / 8;
  static_assert(2 * 16 * HD * 4 + 4 * 16 * 4 <= 2 * AT_K * KS * 2, "the combine must fit the tile area");
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, gid = lane >> 2, tig = lane & 3;
  const int G = p.nq / p.nkv;
  f16* Ks = reinterpret_cast<f16*>(att);
  f16* Vs = Ks + AT_K * KS;
  const f16 *kc, *vc;
  int n, newest;
  att_rows<HD>(p, l, g, c, chunk, ctx, kc, vc, n, newest);
  // the first tile's newest row (the rest was requested before the barrier)
  if (newest >= 0 && newest < AT_K) {
    for (int i = t; i < 2 * (HD / 8); i += NCT) {
      const int which = i >= HD / 8, c8 = i - which * (HD / 8);
      cp_async16((which ? Vs : Ks) + newest * KS + c8 * 8, (which ? vc : kc) + (size_t)newest * HD + c8 * 8);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  const float scale = rsqrtf((float)HD);
  uint32_t qa[NKK][4];
  if (warp < 2) {
    const float* qz = p.q + (size_t)g * G * HD;
#pragma unroll
    for (int kk = 0; kk < NKK; ++kk)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = (r & 1) ? gid + 8 : gid;
        const int col = 16 * kk + ((r & 2) ? 8 : 0) + 2 * tig;
        float2 v = make_float2(0.f, 0.f);
        if (row < G) v = __ldcg(reinterpret_cast<const float2*>(qz + (size_t)row * HD + col));
        qa[kk][r] = pack_half2(v.x * scale, v.y * scale);
      }
  }
  float o[NNT][4];
#pragma unroll
  for (int nt = 0; nt < NNT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  const int ntiles = (n + AT_K - 1) / AT_K;
  const int kw = 16 * warp;
  for (int tt = 0; tt < ntiles; ++tt) {
    if (tt > 0) att_tile_load<HD>(Ks, Vs, kc, vc, tt, n, newest, false);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    cbar();
    if (warp < 2 && tt * AT_K + kw < n) {
      float sc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        const f16* krow = Ks + (size_t)(kw + 8 * nt + gid) * KS + 2 * tig;
#pragma unroll
        for (int kk = 0; kk < NKK; ++kk)
          mma16816(sc[nt], qa[kk], *reinterpret_cast<const uint32_t*>(krow + 16 * kk),
                   *reinterpret_cast<const uint32_t*>(krow + 16 * kk + 8));
        const int key = tt * AT_K + kw + 8 * nt + 2 * tig;  // positions past the chunk: masked
        if (key >= n) sc[nt][0] = sc[nt][2] = -INFINITY;
        if (key + 1 >= n) sc[nt][1] = sc[nt][3] = -INFINITY;
      }
      float mx_lo = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx_hi = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float c_lo = m_lo == -INFINITY ? 0.f : expf(m_lo - mn_lo);
      const float c_hi = m_hi == -INFINITY ? 0.f : expf(m_hi - mn_hi);
      float pr[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        pr[nt][0] = mn_lo == -INFINITY ? 0.f : expf(sc[nt][0] - mn_lo);
        pr[nt][1] = mn_lo == -INFINITY ? 0.f : expf(sc[nt][1] - mn_lo);
        pr[nt][2] = mn_hi == -INFINITY ? 0.f : expf(sc[nt][2] - mn_hi);
        pr[nt][3] = mn_hi == -INFINITY ? 0.f : expf(sc[nt][3] - mn_hi);
      }
      float s_lo = pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1], s_hi = pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
      s_lo += __shfl_xor_sync(0xffffffffu, s_lo, 1);
      s_lo += __shfl_xor_sync(0xffffffffu, s_lo, 2);
      s_hi += __shfl_xor_sync(0xffffffffu, s_hi, 1);
      s_hi += __shfl_xor_sync(0xffffffffu, s_hi, 2);
      l_lo = l_lo * c_lo + s_lo;
      l_hi = l_hi * c_hi + s_hi;
      m_lo = mn_lo;
      m_hi = mn_hi;
      const uint32_t pa[4] = {pack_half2(pr[0][0], pr[0][1]), pack_half2(pr[0][2], pr[0][3]),
                              pack_half2(pr[1][0], pr[1][1]), pack_half2(pr[1][2], pr[1][3])};
      // value rows kw + (lane % 8) + 8 ((lane / 8) % 2), columns of n-tile pair nt, nt + 1
      const f16* vrow = Vs + (size_t)(kw + (lane & 7) + ((lane >> 3) & 1) * 8) * KS + (lane >> 4) * 8;
#pragma unroll
      for (int nt = 0; nt < NNT; nt += 2) {
        o[nt][0] *= c_lo; o[nt][1] *= c_lo; o[nt][2] *= c_hi; o[nt][3] *= c_hi;
        o[nt + 1][0] *= c_lo; o[nt + 1][1] *= c_lo; o[nt + 1][2] *= c_hi; o[nt + 1][3] *= c_hi;
        uint32_t b[4];
        ldmatrix_x4_trans(b, vrow + nt * 8);
        mma16816(o[nt], pa, b[0], b[1]);
        mma16816(o[nt + 1], pa, b[2], b[3]);
      }
    }
    cbar();  // the tile buffers are free again
  }
  // combine warps 0 and 1 (rows < G) in the tile area
  float* cO = reinterpret_cast<float*>(att);  // [2][16][HD]
  float* cM = cO + 2 * 16 * HD;               // [2][16]
  float* cL = cM + 2 * 16;
  if (warp < 2) {
#pragma unroll
    for (int nt = 0; nt < NNT; ++nt) {
      const int col = 8 * nt + 2 * tig;
      *reinterpret_cast<float2*>(cO + (size_t)(warp * 16 + gid) * HD + col) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(cO + (size_t)(warp * 16 + gid + 8) * HD + col) = make_float2(o[nt][2], o[nt][3]);
    }
    if (tig == 0) {
      cM[warp * 16 + gid] = m_lo;
      cM[warp * 16 + gid + 8] = m_hi;
      cL[warp * 16 + gid] = l_lo;
      cL[warp * 16 + gid + 8] = l_hi;
    }
  }
  cbar();
  const int ps = attn_part_stride(HD);
  for (int idx = t; idx < G * HD; idx += NCT) {
    const int r = idx / HD, d = idx - r * HD;
    const float M = fmaxf(cM[r], cM[16 + r]);
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const float mw = cM[w * 16 + r];
      if (mw != -INFINITY) acc = fmaf(expf(mw - M), cO[(size_t)(w * 16 + r) * HD + d], acc);
    }
    p.part[((size_t)(g * G + r) * p.nsplit + c) * ps + d] = acc;
  }
  if (t < G) {
    const float M = fmaxf(cM[t], cM[16 + t]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const float mw = cM[w * 16 + t];
      if (mw != -INFINITY) L = fmaf(expf(mw - M), cL[w * 16 + t], L);
    }
    float* pp = p.part + ((size_t)(g * G + t) * p.nsplit + c) * ps;
    pp[HD] = M;
    pp[HD + 1] = L;
  }
}

// o (the attention output of all heads) merged from the chunk partials into xs:
// o_h = sum_c w_c O_c / sum_c w_c l_c, w_c = exp(m_c - M), M = max_c m_c (chunk order).
// Thread t merges the 4-element groups t and t + NCT, computing its heads' weights itself,
// so the partials, maxima and sums it needs are requested together (one round trip for up to
// MB chunks; a running maximum carries across batches).
template <int HD>
__device__ void stage_merge(const Params& p, float* xs, int ns) {
  const int t = threadIdx.x;
  const int ps = attn_part_stride(HD), groups = p.nq * HD / 4;
  constexpr int MB = 8;
  float4 acc[2];
  float M[2], L[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    M[e] = -INFINITY;
    L[e] = 0.f;
  }
  for (int c0 = 0; c0 < ns; c0 += MB) {
    float4 v[2][MB];
    float2 ml[2][MB];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int gi = t + e * NCT;
      const int h = (4 * gi) / HD, d = 4 * gi - h * HD;
      const float* base = p.part + (size_t)h * p.nsplit * ps;
#pragma unroll
      for (int u = 0; u < MB; ++u) {
        const bool in = gi < groups && c0 + u < ns;
        v[e][u] = in ? __ldcg(reinterpret_cast<const float4*>(base + (size_t)(c0 + u) * ps + d))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        ml[e][u] = in ? __ldcg(reinterpret_cast<const float2*>(base + (size_t)(c0 + u) * ps + HD))
                      : make_float2(-INFINITY, 0.f);
      }
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float mb = M[e];
#pragma unroll
      for (int u = 0; u < MB; ++u) mb = fmaxf(mb, ml[e][u].x);
      if (mb == -INFINITY) continue;  // (groups past the vector)
      const float r = M[e] == -INFINITY ? 0.f : expf(M[e] - mb);  // rescale the earlier batches
      acc[e].x *= r; acc[e].y *= r; acc[e].z *= r; acc[e].w *= r;
      L[e] *= r;
#pragma unroll
      for (int u = 0; u < MB; ++u) {
        if (ml[e][u].x == -INFINITY) continue;
        const float wgt = expf(ml[e][u].x - mb);
        L[e] = fmaf(ml[e][u].y, wgt, L[e]);
        acc[e].x = fmaf(v[e][u].x, wgt, acc[e].x);
        acc[e].y = fmaf(v[e][u].y, wgt, acc[e].y);
        acc[e].z = fmaf(v[e][u].z, wgt, acc[e].z);
        acc[e].w = fmaf(v[e][u].w, wgt, acc[e].w);
      }
      M[e] = mb;
    }
  }
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int gi = t + e * NCT;
    if (gi < groups) {
      const float inv = 1.f / L[e];
      reinterpret_cast<float4*>(xs)[gi] = make_float4(acc[e].x * inv, acc[e].y * inv, acc[e].z * inv, acc[e].w * inv);
    }
  }
  cbar();
}

// Attention output of KV head g merged by the group's own ns attention CTAs (ns > NSPLIT, long
// contexts): each CTA publishes its chunk partials (release on the group's monotonic counter),
// waits (bounded) until the group's ns chunks of layer l are in, then merges a contiguous share
// of the group's G * HD outputs into att_o: o = sum_c w_c O_c / sum_c w_c l_c with
// w_c = exp(m_c - M), M = max_c m_c, in chunk order (deterministic). gbase: the counter's value
// when the step started. False if a wait gave up.
template <int HD>
__device__ bool group_merge(const Params& p, int l, int g, int c, int ns, unsigned long long gbase, int* s_flag) {
  const int t = threadIdx.x, G = p.nq / p.nkv, ps = attn_part_stride(HD);
  cbar();  // this CTA's partials are written
  if (t == 0) {
    int res = 0;
    if (!aborted(p)) {
      asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p.att_cnt + g), "l"(1ull) : "memory");
      const unsigned long long target = gbase + (unsigned long long)(l + 1) * ns;
      const long long t0 = clock64();
      res = 1;
      for (int it = 0;; ++it) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p.att_cnt + g) : "memory");
        if (v >= target) break;
        if ((it & 15) == 15) {
          if (aborted(p)) { res = 0; break; }
          if (clock64() - t0 > WAIT_CYCLES) { raise_abort(p); res = 0; break; }
        }
      }
    }
    *s_flag = res;
  }
  cbar();
  if (!*(volatile int*)s_flag) return false;
  // warp w merges outputs o0 + w + 8k, lane j reads chunks j and j + 32 (ns <= 64): every
  // load of the share first, then warp reductions in a fixed order
  constexpr int KM = 8;  // outputs per warp: G * HD / ns <= 8 * HD / 17 < 8 * NCW
  const int n_out = G * HD, per = (n_out + ns - 1) / ns;
  const int o0 = c * per, o1 = min(n_out, o0 + per);
  const int warp = t >> 5, lane = t & 31;
  float2 ml[KM][2];
  float ov[KM][2];
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    const int i = o0 + warp + NCW * k;
    const int h = g * G + i / HD, d = i - (i / HD) * HD;
    const float* base = p.part + (size_t)h * p.nsplit * ps;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int cc = lane + 32 * j;
      const bool in = i < o1 && cc < ns;
      ml[k][j] = in ? __ldcg(reinterpret_cast<const float2*>(base + (size_t)cc * ps + HD)) : make_float2(-INFINITY, 0.f);
      ov[k][j] = in ? __ldcg(base + (size_t)cc * ps + d) : 0.f;
    }
  }
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    const int i = o0 + warp + NCW * k;
    float M = fmaxf(ml[k][0].x, ml[k][1].x);
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float w = ml[k][j].x == -INFINITY ? 0.f : expf(ml[k][j].x - M);
      L = fmaf(ml[k][j].y, w, L);
      acc = fmaf(ov[k][j], w, acc);
    }
    L = warp_sum(L);
    acc = warp_sum(acc);
    if (lane == 0 && i < o1) {
      const int h = g * G + i / HD, d = i - (i / HD) * HD;
      p.att_o[(size_t)h * HD + d] = acc / L;
    }
  }
  return true;
}

// xs = src[0 .. n) (the merged attention output), one barrier
__device__ void stage_vec(float* xs, const float* src, int n) {
  for (int i = threadIdx.x; i < (n >> 2); i += NCT)
    reinterpret_cast<float4*>(xs)[i] = __ldcg(reinterpret_cast<const float4*>(src) + i);
  cbar();
}

// ---- the kernel ------------------------------------------------------------------------

// NV: 16-byte vectors per lane of the register tile of the input vector (a row of hidden
// elements, or a warp's eighth of a down-projection row)
template <int HD, int NV>
__global__ void __launch_bounds__(THREADS, 1) decode_step_kernel(const Params p) {
  extern __shared__ unsigned char mk_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)mk_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* att = smem + p.lay.att;
  float* xs = reinterpret_cast<float*>(smem + p.lay.xs);
  float* dA = reinterpret_cast<float*>(smem + p.lay.da);
  float* dB = reinterpret_cast<float*>(smem + p.lay.db);
  float* dP = reinterpret_cast<float*>(smem + p.lay.dp);
  float* qe = reinterpret_cast<float*>(smem + p.lay.qe);
  float* xo = reinterpret_cast<float*>(smem + p.lay.xo);
  LayerW* lt = reinterpret_cast<LayerW*>(smem + p.lay.lt);
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(smem + p.lay.bar);
  float* scr = reinterpret_cast<float*>(smem + p.lay.scr);
  int* s_flag = reinterpret_cast<int*>(scr + 48);
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + NS);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int half = HD >> 1;
  const int npairs = (p.nq + 2 * p.nkv) * half;

  // the position and the token were written by the previous step (or the prefill), before
  // this launch; the key is zero between steps
  const int pos = __ldcg(p.pos);
  const int ctx = pos + 1;
  int tok = __ldcg(p.tok);
  if (tok < 0 || tok >= p.V) {
    if (t == 0 && blockIdx.x == 0) atomicOr(p.err, ERR_TOKEN);
    tok = 0;
  }
  const bf16* erow = p.embed + (size_t)tok * p.H;
  int r0, r1;  // this CTA's residual rows (the o_proj and down rows)
  block_of(p.H, r0, r1);
  int q0, q1;  // this CTA's q/k/v pairs
  block_of(npairs, q0, q1);
  // pair t (t < q1 - q0): the rotation at pos (the same in every layer) and the bias of both
  // rows, requested well before the q/k/v phase that uses them (weights and the position only)
  float4 qv = make_float4(0.f, 0.f, 1.f, 0.f);
  const int qhead = (q0 + t) / half, qe_i = q0 + t - qhead * half;
  if (t < q1 - q0 && qhead < p.nq + p.nkv) {
    const float2 cs = p.rope[(size_t)pos * half + qe_i];
    qv.z = cs.x;
    qv.w = cs.y;
  }
  auto load_bias = [&](const LayerW& w) {
    if (t < q1 - q0) {
      const bf16* bias;
      int hh;
      if (qhead < p.nq) { bias = w.bq; hh = qhead; }
      else if (qhead < p.nq + p.nkv) { bias = w.bk; hh = qhead - p.nq; }
      else { bias = w.bv; hh = qhead - p.nq - p.nkv; }
      if (bias) {
        qv.x = __bfloat162float(bias[hh * HD + qe_i]);
        qv.y = __bfloat162float(bias[hh * HD + qe_i + half]);
      }
    }
  };
  load_bias(reinterpret_cast<const LayerW*>(p.layers)[0]);
  if (t == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, NCW);
    }
    mbar_fence_init();
  }
  {  // the layer pointer table, read at every phase, lives in shared memory
    const int n8 = p.L * (int)(sizeof(LayerW) / 8);
    const unsigned long long* src = reinterpret_cast<const unsigned long long*>(p.layers);
    unsigned long long* dst = reinterpret_cast<unsigned long long*>(lt);
    for (int i = t; i < n8; i += THREADS) dst[i] = __ldg(src + i);
  }
  if (t < NCT) {
    // the residual stream starts as the embedding row (this CTA's rows)
    for (int i = t; i < r1 - r0; i += NCT) {
      xo[i] = __bfloat162float(erow[r0 + i]);
      p.x[r0 + i] = xo[i];
    }
  }
  __syncthreads();  // the only block-wide barrier: producers and consumers part here

  if (warp >= NCW) {
    if (lane == 0) producer<HD>(p, lt, smem, full0, empty0, warp - NCW, ctx);
    return;
  }

  // ---------------- consumers ----------------
  const unsigned long long base = __ldcg(p.bar_base);
  int nb = 0;        // grid barriers passed
  long long u = 0;   // unit counter
  const int nvecH = p.H >> 3;
  const size_t rowH = (size_t)p.H * 2;
  int chunk, ns;
  att_chunks(ctx, p.nsplit, chunk, ns);
  float xr[NV][8];
  bool alive = true;
  int ph_idx = 0;  // timeline index

  // wait for unit u, apply fn to it (fn sees the unit's index in its phase), release the slot
  int phase_u = 0;  // units consumed in the current phase
  auto consume = [&](const Unit& un, auto&& fn) -> bool {
    const long long my = u++;
    const int s = (int)(my % NS);
    const bool ok = __all_sync(0xffffffffu, slot_wait(p, full0 + 8 * s, (uint32_t)((my / NS) & 1)));
    if (!ok) return false;
    fn(smem + (size_t)s * SLOT, un);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    if (phase_u++ == 0) {
      tl_mark3(p, ph_idx, 0);
      ck(p, ph_idx, 4);
    }
    return true;
  };
  // In the paired phases (q/k/v: rows i, i + hd/2 of a RoPE pair; gate/up: gate row i, up row
  // i) a unit holds up to 4 pairs: pair j in row j of the first and of the second copy. The
  // units of a phase alternate between warps 0-3 and 4-7; warp w takes pair w % 4 of its
  // units, both rows, and finishes the pair itself.
  const int pj = warp & 3, pgroup = warp >> 2;

  for (int l = 0; l < p.L && alive; ++l) {
    const LayerW& w = lt[l];
    // ===== QKV: RMSNorm -> q/k/v rows (+ bias) -> RoPE -> q out, K/V append
    tl_mark(p, ph_idx, 0);
    phase_u = 0;
    if ((int)blockIdx.x < p.nkv * ns) {  // the first attention tile's rows of earlier steps
      const int g = blockIdx.x / ns, c = blockIdx.x - g * ns;
      attention_preload<HD>(p, att, l, g, c, chunk, ctx);
    }
    ck(p, ph_idx, 0);
    stage_gain(p, xs, scr, p.x, l == 0 ? erow : nullptr, w.in_norm,
               t < q1 - q0 ? reinterpret_cast<float4*>(qe) + t : nullptr, qv);
    load_xr(xr, xs, nvecH, lane);
    float inv = norm_scale(p, scr);
    tl_mark2(p, ph_idx);
    ck(p, ph_idx, 3);
    alive = phase_units(p, lt, HD, l, P_QKV, [&](const Unit& un) {
      return consume(un, [&](const unsigned char* slot, const Unit& v) {
        if (pgroup != (phase_u & 1) || pj >= v.n) return;
        float a = row_dot<NV>(reinterpret_cast<const uint4*>(slot + pj * rowH), xr, 0, nvecH, lane) * inv;
        float b = row_dot<NV>(reinterpret_cast<const uint4*>(slot + v.off2 + pj * rowH), xr, 0, nvecH, lane) * inv;
        if (lane == 0) {
          const int pi = v.a + pj - q0, item = v.a + pj, head = item / half, e = item - head * half;
          a += qe[4 * pi + 0];
          b += qe[4 * pi + 1];
          if (head < p.nq + p.nkv) {  // rotate the pair (e, e + hd/2)
            const float c = qe[4 * pi + 2], sn = qe[4 * pi + 3];
            const float ra = a * c - b * sn, rb = b * c + a * sn;
            a = ra;
            b = rb;
          }
          if (head < p.nq) {
            p.q[head * HD + e] = a;
            p.q[head * HD + e + half] = b;
          } else {
            const bool is_k = head < p.nq + p.nkv;
            const int hh = is_k ? head - p.nq : head - p.nq - p.nkv;
            f16* dst = p.kv + (size_t)l * 2 * p.nkv * p.cap * HD + (is_k ? 0 : (size_t)p.nkv * p.cap * HD) +
                       ((size_t)hh * p.cap + pos) * HD;
            store_kv(dst + e, a, p.err);
            store_kv(dst + e + half, b, p.err);
          }
        }
      });
    });
    tl_mark(p, ph_idx, 1);
    ck(p, ph_idx, 5);
    tl_mark3(p, ph_idx, 2);
    ck(p, ph_idx, 7);
    tl_mark(p, ph_idx++, 2);
    alive = grid_sync(p, base, nb, s_flag, ph_idx - 1, alive);
    if (!alive) break;

    // ===== ATTN: (KV head, chunk) partials
    tl_mark(p, ph_idx, 0);
    phase_u = 0;
    bool att_ok = true;
    if ((int)blockIdx.x < p.nkv * ns) {
      const int g = blockIdx.x / ns, c = blockIdx.x - g * ns;
      attention_chunk<HD>(p, att, l, g, c, chunk, ctx);
      if (ns > NSPLIT) att_ok = group_merge<HD>(p, l, g, c, ns, __ldcg(p.att_base + g), s_flag);
    }
    tl_mark3(p, ph_idx, 2);
    tl_mark(p, ph_idx++, 2);
    alive = grid_sync(p, base, nb, s_flag, ph_idx - 1, att_ok);
    if (!alive) break;

    // ===== OPROJ: merge -> x += Wo o (each row's warp updates the CTA's residual row)
    tl_mark(p, ph_idx, 0);
    phase_u = 0;
    ck(p, ph_idx, 0);
    if (ns > NSPLIT)
      stage_vec(xs, p.att_o, p.nq * HD);
    else
      stage_merge<HD>(p, xs, ns);
    load_xr(xr, xs, (p.nq * HD) >> 3, lane);
    tl_mark2(p, ph_idx);
    ck(p, ph_idx, 3);
    {
      const int R = rows_per_slot(p.H);
      alive = phase_units(p, lt, HD, l, P_OPROJ, [&](const Unit& un) {
        return consume(un, [&](const unsigned char* slot, const Unit& v) {
          if (warp >= R || warp >= v.n) return;
          const float d = row_dot<NV>(reinterpret_cast<const uint4*>(slot + (size_t)warp * rowH), xr, 0,
                                      (p.nq * HD) >> 3, lane);
          if (lane == 0) {
            const int r = v.a + warp;
            xo[r - r0] += d;
            p.x[r] = xo[r - r0];
          }
        });
      });
    }
    tl_mark(p, ph_idx, 1);
    ck(p, ph_idx, 5);
    tl_mark3(p, ph_idx, 2);
    ck(p, ph_idx, 7);
    tl_mark(p, ph_idx++, 2);
    alive = grid_sync(p, base, nb, s_flag, ph_idx - 1, alive);
    if (!alive) break;

    // ===== GATEUP: RMSNorm -> gate/up rows -> SwiGLU (each pair's warp writes its output)
    tl_mark(p, ph_idx, 0);
    phase_u = 0;
    ck(p, ph_idx, 0);
    stage_gain(p, xs, scr, p.x, nullptr, w.post_norm);
    load_xr(xr, xs, nvecH, lane);
    inv = norm_scale(p, scr);
    tl_mark2(p, ph_idx);
    ck(p, ph_idx, 3);
    alive = phase_units(p, lt, HD, l, P_GATEUP, [&](const Unit& un) {
      return consume(un, [&](const unsigned char* slot, const Unit& v) {
        if (pgroup != (phase_u & 1) || pj >= v.n) return;
        const float gv = row_dot<NV>(reinterpret_cast<const uint4*>(slot + pj * rowH), xr, 0, nvecH, lane) * inv;
        const float uv = row_dot<NV>(reinterpret_cast<const uint4*>(slot + v.off2 + pj * rowH), xr, 0, nvecH, lane) * inv;
        if (lane == 0) p.act[v.a + pj] = (gv / (1.f + expf(-gv))) * uv;
      });
    });
    tl_mark(p, ph_idx, 1);
    ck(p, ph_idx, 5);
    tl_mark3(p, ph_idx, 2);
    ck(p, ph_idx, 7);
    tl_mark(p, ph_idx++, 2);
    alive = grid_sync(p, base, nb, s_flag, ph_idx - 1, alive);
    if (!alive) break;

    // ===== DOWN: x += Wd act, each row's K split over the eight warps
    tl_mark(p, ph_idx, 0);
    phase_u = 0;
    ck(p, ph_idx, 0);
    if (l + 1 < p.L) load_bias(lt[l + 1]);  // (used by the next layer's q/k/v phase)
    {
      const int nvecI = p.I >> 3;
      const int segv = (nvecI + NCW - 1) / NCW;
      const int v0 = warp * segv, v1 = min(nvecI, v0 + segv);
#pragma unroll
      for (int qd = 0; qd < NV; ++qd) {
        const int v = v0 + lane + 32 * qd;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (v < v1) {
          a = __ldcg(reinterpret_cast<const float4*>(p.act) + 2 * v);
          b = __ldcg(reinterpret_cast<const float4*>(p.act) + 2 * v + 1);
        }
        xr[qd][0] = a.x; xr[qd][1] = a.y; xr[qd][2] = a.z; xr[qd][3] = a.w;
        xr[qd][4] = b.x; xr[qd][5] = b.y; xr[qd][6] = b.z; xr[qd][7] = b.w;
      }
      tl_mark2(p, ph_idx);
      ck(p, ph_idx, 3);
      alive = phase_units(p, lt, HD, l, P_DOWN, [&](const Unit& un) {
        return consume(un, [&](const unsigned char* slot, const Unit& v) {
          const float acc = row_dot<NV>(reinterpret_cast<const uint4*>(slot), xr, v0, v1, lane);
          if (lane == 0) dP[(v.a - r0) * NCW + warp] = acc;
        });
      });
    }
    tl_mark(p, ph_idx, 1);
    ck(p, ph_idx, 5);
    alive = cbar_and(alive);
    tl_mark3(p, ph_idx, 1);
    ck(p, ph_idx, 6);
    if (alive)
      for (int i = t; i < r1 - r0; i += NCT) {
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < NCW; ++k) sum += dP[i * NCW + k];  // warp order
        xo[i] += sum;
        p.x[r0 + i] = xo[i];
      }
    tl_mark3(p, ph_idx, 2);
    ck(p, ph_idx, 7);
    tl_mark(p, ph_idx++, 2);
    alive = grid_sync(p, base, nb, s_flag, ph_idx - 1, alive);
  }

  // ===== LM head: final RMSNorm -> logits -> greedy argmax
  if (alive) {
    tl_mark(p, ph_idx, 0);
    phase_u = 0;
    ck(p, ph_idx, 0);
    stage_gain(p, xs, scr, p.x, nullptr, p.final_norm);
    load_xr(xr, xs, nvecH, lane);
    const float inv = norm_scale(p, scr);
    tl_mark2(p, ph_idx);
    ck(p, ph_idx, 3);
    float best_v = -INFINITY;
    int best_i = -1;
    bool bad = false;
    {
      const int R = rows_per_slot(p.H);
      alive = phase_units(p, lt, HD, p.L, P_LM, [&](const Unit& un) {
        return consume(un, [&](const unsigned char* slot, const Unit& v) {
          if (warp >= R || warp >= v.n) return;
          const float z = row_dot<NV>(reinterpret_cast<const uint4*>(slot + (size_t)warp * rowH), xr, 0, nvecH, lane) * inv;
          const int r = v.a + warp;
          if (lane == 0) p.logits[r] = z;
          if (!isfinite(z)) bad = true;
          if (z > best_v || best_i < 0) { best_v = z; best_i = r; }  // rows arrive in increasing order
        });
      });
    }
    tl_mark(p, ph_idx, 1);
    ck(p, ph_idx, 5);
    if (lane == 0) {
      reinterpret_cast<unsigned long long*>(dP)[warp] = best_i >= 0 ? argmax_key(best_v, best_i) : 0ull;
      reinterpret_cast<int*>(dA)[warp] = bad;
    }
    alive = cbar_and(alive);
    tl_mark3(p, ph_idx, 1);
    ck(p, ph_idx, 6);
    if (alive && t == 0) {
      unsigned long long k = 0;
      int anybad = 0;
      for (int i = 0; i < NCW; ++i) {
        const unsigned long long ki = reinterpret_cast<unsigned long long*>(dP)[i];
        k = ki > k ? ki : k;
        anybad |= reinterpret_cast<int*>(dA)[i];
      }
      if (k) atomicMax(p.key, k);
      if (anybad) atomicOr(p.err, ERR_NONFINITE);
    }
    tl_mark3(p, ph_idx, 2);
    ck(p, ph_idx, 7);
    tl_mark(p, ph_idx++, 2);
    alive = grid_sync(p, base, nb, s_flag, ph_idx - 1, alive);
    if (alive && blockIdx.x == 0 && t == 0) {
      const unsigned long long k = atomicAdd(p.key, 0ull);
      const int idx = argmax_key_index(k);
      *p.tok = idx;
      const int hn = __ldcg(p.hist_n);
      if (hn < p.hist_cap) p.hist[hn] = idx;
      *p.hist_n = hn + 1;
      *p.pos = pos + 1;
      *p.key = 0ull;
      *p.bar_base = base + (unsigned long long)nb * gridDim.x;  // every CTA has arrived nb times
      if (ns > NSPLIT)  // every attention CTA of each KV head has arrived once per layer
        for (int g = 0; g < p.nkv; ++g) p.att_base[g] += (unsigned long long)p.L * ns;
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // (copies are only left after an abort)
}

}  // namespace mk

// ---- host side ---------------------------------------------------------------------------

// 16-byte vectors per lane the register tile needs: a row of hidden elements, or a warp's
// eighth of a down-projection row
static int megastep_nv(const Dims& d) {
  const int row = (d.H / 8 + 31) / 32;
  const int seg = ((d.I / 8 + mk::NCW - 1) / mk::NCW + 31) / 32;
  const int need = std::max(row, seg);
  return need <= 4 ? 4 : need <= 6 ? 6 : need <= 8 ? 8 : 0;
}

bool megastep_supported(const Dims& d, int nsm) {
  if (d.dtype != 1) return false;
  if (d.hd != 64 && d.hd != 128) return false;
  if (d.nq / d.nkv > mk::GMAX || d.nq * d.hd != d.H) return false;
  if (d.H % 8 || d.H > mk::XS_FLOATS) return false;
  if (d.nq > 32) return false;  // merge weights [2][nq][NSPLIT] of 32 heads at most
  if (d.I % 8 || (size_t)d.I * 2 > (size_t)mk::SLOT) return false;
  if (megastep_nv(d) == 0) return false;
  const int R = std::min(mk::NCW, (mk::SLOT / (2 * d.H)) & ~1);
  if (R < 2) return false;
  const int pairs = (d.nq + 2 * d.nkv) * d.hd / 2;
  auto per_cta = [&](int n) { return (n + nsm - 1) / nsm; };
  if (per_cta(pairs) > mk::MAX_LOCAL || per_cta(d.I) > mk::MAX_LOCAL || per_cta(d.H) > 64) return false;
  if (d.nkv * mk::NSPLIT > nsm) return false;
  if (d.nkv > mk::MAX_KV_GROUPS) return false;
  if (megastep_smem(d) > 227 * 1024) return false;
  return true;
}

size_t megastep_smem(const Dims& d) { return mk::make_layout(d.hd, d.H, d.nq, d.L).total; }

static const void* megastep_fn(const Dims& d) {
  const int nv = megastep_nv(d);
  if (d.hd == 128)
    return nv == 4 ? (const void*)mk::decode_step_kernel<128, 4>
                   : nv == 6 ? (const void*)mk::decode_step_kernel<128, 6> : (const void*)mk::decode_step_kernel<128, 8>;
  return nv == 4 ? (const void*)mk::decode_step_kernel<64, 4>
                 : nv == 6 ? (const void*)mk::decode_step_kernel<64, 6> : (const void*)mk::decode_step_kernel<64, 8>;
}

// most attention chunks per KV head: every (KV head, chunk) pair has its own CTA
int megastep_nsplit(const Dims& d, int nsm) { return std::min(mk::NSPLIT_MAX, nsm / d.nkv); }

size_t megastep_work_floats(const Dims& d) {  // x, act, the attention partials, the merged output
  return (size_t)d.H + d.I + (size_t)d.nq * megastep_nsplit(d, d.nsm) * attn_part_stride(d.hd) + (size_t)d.nq * d.hd;
}


cudaError_t megastep_set_attributes(const Dims& d) {
  return cudaFuncSetAttribute(megastep_fn(d), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)megastep_smem(d));
}

int megastep_threads() { return mk::THREADS; }

cudaError_t megastep_occupancy(const Dims& d, int* per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, megastep_fn(d), mk::THREADS, megastep_smem(d));
}

size_t megastep_layer_bytes() { return sizeof(mk::LayerW); }

void megastep_fill_layer(void* dst, const LayerPtrs& w) {
  mk::LayerW lw{(const bf16*)w.in_norm, (const bf16*)w.wq, (const bf16*)w.wk, (const bf16*)w.wv,
                (const bf16*)w.bq, (const bf16*)w.bk, (const bf16*)w.bv, (const bf16*)w.wo,
                (const bf16*)w.post_norm, (const bf16*)w.w_gate, (const bf16*)w.w_up, (const bf16*)w.w_down};
  std::memcpy(dst, &lw, sizeof(lw));
}

cudaError_t launch_megastep(const MegaLaunch& a, cudaStream_t s) {
  mk::Params p{};
  p.layers = (const mk::LayerW*)a.layers_dev;
  p.L = a.d.L; p.H = a.d.H; p.nq = a.d.nq; p.nkv = a.d.nkv; p.I = a.d.I; p.V = a.d.V; p.cap = a.d.cap;
  p.eps = a.d.eps;
  p.embed = (const bf16*)a.embed; p.final_norm = (const bf16*)a.final_norm; p.head = (const bf16*)a.head;
  p.rope = a.rope; p.kv = (f16*)a.kv_seq;
  p.x = a.work;
  p.act = a.work + a.d.H;
  p.part = a.work + a.d.H + a.d.I;
  p.nsplit = megastep_nsplit(a.d, a.d.nsm);
  p.att_o = p.part + (size_t)a.d.nq * p.nsplit * attn_part_stride(a.d.hd);
  p.att_cnt = a.bar + 2;
  p.att_base = a.bar + 2 + mk::MAX_KV_GROUPS;
  p.q = a.q; p.logits = a.logits;
  p.tok = a.tok; p.pos = a.pos; p.key = a.key; p.hist = a.hist; p.hist_n = a.hist_n; p.hist_cap = a.hist_cap;
  p.bar = a.bar; p.bar_base = a.bar_base; p.abort = a.abort; p.err = a.err; p.tl = a.tl;
  p.pf_mode = a.pf_mode;
  p.lay = mk::make_layout(a.d.hd, a.d.H, a.d.nq, a.d.L);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(mk::THREADS);
  cfg.dynamicSmemBytes = p.lay.total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&p};
  return cudaLaunchKernelExC(&cfg, megastep_fn(a.d), args);
}

}  // namespace qw
