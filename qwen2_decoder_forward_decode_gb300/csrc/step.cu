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
constexpr int THREADS = (NCW + 1) * 32;   // + one producer warp
constexpr int NCT = NCW * 32;             // consumer threads
constexpr int SLOT = 6 * 1024;            // bytes per ring slot
constexpr int MAX_SLOTS = 28;
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
  int xs_floats;    // floats of the staged input vector region
  unsigned long long* tl;  // timeline: per phase [start, end, producer issued] (CTA 0), or null
  int* diag;               // first expired wait: [site, CTA, warp, detail]
};

constexpr int MAX_SPLIT = 16;

struct Geo {
  int n_items, rows, K, chunk, U;
};

__device__ __forceinline__ Geo geo(const Params& p, int ph) {
  Geo g;
  switch (ph) {
    case P_QKV: g.n_items = (p.nq + 2 * p.nkv) * (p.hd / 2); g.rows = 2; g.K = p.H; break;
    case P_OPROJ: g.n_items = (p.H + 1) / 2; g.rows = 2; g.K = p.nq * p.hd; break;
    case P_GATEUP: g.n_items = p.I; g.rows = 2; g.K = p.H; break;
    case P_DOWN: g.n_items = p.H; g.rows = 1; g.K = p.I; break;
    default: g.n_items = (p.V + 1) / 2; g.rows = 2; g.K = p.H; break;
  }
  int chunk = SLOT / (g.rows * 2);
  chunk &= ~7;
  g.chunk = g.K < chunk ? g.K : chunk;
  g.U = (g.K + g.chunk - 1) / g.chunk;
  return g;
}

// row r of item `item` in phase ph of layer l (null when the row does not exist)
__device__ __forceinline__ const bf16* row_ptr(const Params& p, int ph, int l, int item, int r) {
  const Layer& w = p.layers[l < p.L ? l : 0];
  switch (ph) {
    case P_QKV: {
      const int half = p.hd >> 1;
      int head = item / half;
      const int rr = item - head * half + r * half;
      if (head < p.nq) return w.wq + (size_t)(head * p.hd + rr) * p.H;
      head -= p.nq;
      if (head < p.nkv) return w.wk + (size_t)(head * p.hd + rr) * p.H;
      head -= p.nkv;
      return w.wv + (size_t)(head * p.hd + rr) * p.H;
    }
    case P_OPROJ: {
      const int rr = 2 * item + r;
      return rr < p.H ? w.wo + (size_t)rr * p.nq * p.hd : nullptr;
    }
    case P_GATEUP: return (r == 0 ? w.wg : w.wu) + (size_t)item * p.H;
    case P_DOWN: return w.wd + (size_t)item * p.I;
    default: {
      const int rr = 2 * item + r;
      return rr < p.V ? p.head + (size_t)rr * p.H : nullptr;
    }
  }
}

__device__ __forceinline__ int n_local(int n_items) {
  const int c = blockIdx.x, G = gridDim.x;
  return c < n_items ? (n_items - 1 - c) / G + 1 : 0;
}

__device__ __forceinline__ bool aborted(const Params& p) { return *(volatile int*)p.abort != 0; }

enum : int { SITE_SLOT_FULL = 1, SITE_SLOT_EMPTY = 2, SITE_GRID = 3 };

// First expiry wins the diagnostic record; every later wait sees the abort flag.
__device__ __forceinline__ void raise_abort(const Params& p, int site, long long detail) {
  if (atomicExch(p.abort, 1) == 0 && p.diag) {
    p.diag[0] = site;
    p.diag[1] = blockIdx.x;
    p.diag[2] = threadIdx.x >> 5;
    p.diag[3] = (int)detail;
  }
  atomicOr(p.err, ERR_TIMEOUT);
}

// Bounded wait (non-blocking tests) that also gives up when another CTA has aborted.
__device__ __forceinline__ bool slot_wait(const Params& p, uint32_t bar, uint32_t parity, int site,
                                          long long detail) {
  if (mbar_test_now(bar, parity)) return true;
  const long long t0 = clock64();
  for (int it = 0;; ++it) {
    if (mbar_test_now(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (aborted(p)) return false;
      if (clock64() - t0 > WAIT_CYCLES) {
        raise_abort(p, site, detail);
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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = p.nslots;
  float* xs = reinterpret_cast<float*>(dsm + (size_t)NS * SLOT);
  const uint32_t ring = smem_addr(dsm);
  const uint32_t full0 = smem_addr(full), empty0 = smem_addr(empty);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_fence_init();
  }
  __syncthreads();
  const int pos = __ldcg(p.pos);  // the token of this step sits at position pos

  // ---------------- producer ----------------
  if (warp == NCW) {
    // Units of a phase are issued in batches: lane k of the warp computes the addresses of
    // unit (batch + k), waits for that unit's slot to be free and issues its copies. A batch
    // holds at most NS units, so no two lanes of a batch share a slot.
    const int NSB = NS < 32 ? NS : 32;
    long long seq = 0, issued = 0;  // units scheduled / actually issued
    bool ok = !aborted(p);
    for (int l = 0; l <= p.L && ok; ++l) {
      for (int ph = 0; ph < 5 && ok; ++ph) {
        int phase = ph;
        if (l == p.L) {
          if (ph > 0) break;
          phase = P_LM;
        } else if (ph == P_ATTN) {
          continue;
        }
        const Geo g = geo(p, phase);
        const int nl = n_local(g.n_items);
        const int total = nl * g.U;
        // this phase's matrices, once per phase
        const Layer* lw = p.layers + (l < p.L ? l : 0);
        const bf16* mq = lw->wq;
        const bf16* mk = lw->wk;
        const bf16* mv = lw->wv;
        const bf16* mo = lw->wo;
        const bf16* mg = lw->wg;
        const bf16* mu = lw->wu;
        const bf16* md = lw->wd;
        for (int b0 = 0; b0 < total && ok; b0 += NSB) {
          const int k = b0 + lane;
          const bf16* r0 = nullptr;
          const bf16* r1 = nullptr;
          uint32_t bytes = 0, dst_off = 0;
          if (lane < NSB && k < total) {
            const int j = k / g.U, u = k - j * g.U;
            const int item = blockIdx.x + j * gridDim.x;
            switch (phase) {
              case P_QKV: {
                const int half = p.hd >> 1;
                int head = item / half;
                const int i = item - head * half;
                const bf16* m = mq;
                if (head >= p.nq) { head -= p.nq; m = mk; if (head >= p.nkv) { head -= p.nkv; m = mv; } }
                r0 = m + (size_t)(head * p.hd + i) * p.H;
                r1 = r0 + (size_t)half * p.H;
                break;
              }
              case P_OPROJ:
                r0 = mo + (size_t)(2 * item) * g.K;
                r1 = 2 * item + 1 < p.H ? r0 + g.K : nullptr;
                break;
              case P_GATEUP:
                r0 = mg + (size_t)item * p.H;
                r1 = mu + (size_t)item * p.H;
                break;
              case P_DOWN:
                r0 = md + (size_t)item * p.I;
                break;
              default:
                r0 = p.head + (size_t)(2 * item) * p.H;
                r1 = 2 * item + 1 < p.V ? r0 + p.H : nullptr;
                break;
            }
            const int k0 = u * g.chunk;
            bytes = (uint32_t)min(g.chunk, g.K - k0) * 2;
            r0 += k0;
            if (r1) r1 += k0;
            dst_off = (uint32_t)g.chunk * 2;
          }
          // lane 0 waits for each unit's slot and issues its copies, in sequence order
          const int n = min(NSB, total - b0);
          for (int kk = 0; kk < n && ok; ++kk) {
            const bf16* a0 = (const bf16*)__shfl_sync(0xffffffffu, (unsigned long long)r0, kk);
            const bf16* a1 = (const bf16*)__shfl_sync(0xffffffffu, (unsigned long long)r1, kk);
            const uint32_t nb = __shfl_sync(0xffffffffu, bytes, kk);
            const uint32_t off1 = __shfl_sync(0xffffffffu, dst_off, kk);
            bool lane_ok = true;
            if (lane == 0) {
              const long long sq = seq + b0 + kk;
              const int s = (int)(sq % NS);
              if (sq >= NS) {
                const uint32_t par = (uint32_t)(((sq / NS) - 1) & 1);
                if (p.tl && blockIdx.x == 0) {  // occupancy statistics of the ring (profiling)
                  p.tl[3 * (5 * p.L + 1) + 0] += 1;
                  if (!mbar_test_now(empty0 + 8 * s, par)) p.tl[3 * (5 * p.L + 1) + 1] += 1;
                }
                lane_ok = slot_wait(p, empty0 + 8 * s, par, SITE_SLOT_EMPTY, sq);
              }
              if (lane_ok) {
                mbar_expect_tx(full0 + 8 * s, nb * (a1 ? 2u : 1u));
                const uint32_t dst = ring + s * SLOT;
                bulk_copy_g2s(dst, a0, nb, full0 + 8 * s);
                if (a1) bulk_copy_g2s(dst + off1, a1, nb, full0 + 8 * s);
                issued = sq + 1;
              }
            }
            ok = __shfl_sync(0xffffffffu, lane_ok ? 1 : 0, 0) != 0;
          }
        }
        seq += total;
        if (p.tl && blockIdx.x == 0 && lane == 0) {
          const int pi = l == p.L ? 5 * p.L : 5 * l + ph;
          p.tl[3 * pi + 2] = gtime();
        }
      }
    }
    // let every issued copy land before this warp (and, with it, the CTA) may finish
    if (lane == 0) {
      const long long first = issued > NS ? issued - NS : 0;
      for (long long k = first; k < issued; ++k) {
        const int s = (int)(k % NS);
        const long long t0 = clock64();
        while (!mbar_test_now(full0 + 8 * s, (uint32_t)((k / NS) & 1)) && clock64() - t0 < WAIT_CYCLES) {
        }
      }
    }
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

  // consume one weight phase: per item, accumulate over its U units, then the epilogue
  auto run_phase = [&](int phase, int l, auto&& epilogue) -> bool {
    const Geo g = geo(p, phase);
    const int nl = n_local(g.n_items);
    bool ok = true;
    for (int j = warp; j < nl; j += NCW) {
      const int item = blockIdx.x + j * gridDim.x;
      float a0 = 0.f, a1 = 0.f;
      for (int u = 0; u < g.U; ++u) {
        const long long seq = base + (long long)j * g.U + u;
        const int s = (int)(seq % NS);
        if (p.tl && blockIdx.x == 0 && threadIdx.x == 0 &&
            !mbar_test_now(full0 + 8 * s, (uint32_t)((seq / NS) & 1)))
          p.tl[3 * (5 * p.L + 1) + 2] += 1;
        if (!__all_sync(0xffffffffu, slot_wait(p, full0 + 8 * s, (uint32_t)((seq / NS) & 1), SITE_SLOT_FULL, seq))) {
          ok = false;
          break;
        }
        const int k0 = u * g.chunk;
        const int nv = min(g.chunk, g.K - k0) >> 3;
        const uint4* w0 = reinterpret_cast<const uint4*>(dsm + (size_t)s * SLOT);
        const uint4* w1 = reinterpret_cast<const uint4*>(dsm + (size_t)s * SLOT + g.chunk * 2);
        const float4* x4 = reinterpret_cast<const float4*>(xs + k0);
#pragma unroll 4
        for (int v = lane; v < nv; v += 32) {
          const float4 xa = x4[2 * v], xb = x4[2 * v + 1];
          const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
          a0 = dotv(w0[v], xv, a0, bf16());
          if (g.rows == 2) a1 = dotv(w1[v], xv, a1, bf16());
        }
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty0 + 8 * s) : "memory");
      }
      if (!ok) break;
      a0 = warp_sum(a0);
      if (g.rows == 2) a1 = warp_sum(a1);
      if (lane == 0) epilogue(item, a0, a1);
    }
    base += (long long)nl * g.U;
    return ok;
  };

  bool ok = !aborted(p);  // a failed earlier launch leaves the model unusable: return fast
  int phase_no = 0;
  auto stamp = [&](int which) {  // CTA 0: [start, end] of consumer phase phase_no
    if (p.tl && blockIdx.x == 0 && ct == 0) p.tl[3 * phase_no + which] = gtime();
  };
  for (int l = 0; l < p.L && ok; ++l) {
    const Layer& w = p.layers[l];
    f16* kc = p.kv + (size_t)l * 2 * p.nkv * p.cap * p.hd;
    f16* vc = kc + (size_t)p.nkv * p.cap * p.hd;
    // ---- QKV
    stamp(0);
    if (l == 0) stage_embed(p, xs, scratch, w.in_norm);
    else stage_norm(p, xs, scratch, p.x, w.in_norm, p.H);
    ok = run_phase(P_QKV, l, [&](int item, float a, float b) {
      int head = item / half;
      const int i = item - head * half;
      const bf16* bias;
      int h;
      if (head < p.nq) { bias = w.bq; h = head; }
      else if (head < p.nq + p.nkv) { bias = w.bk; h = head - p.nq; }
      else { bias = w.bv; h = head - p.nq - p.nkv; }
      if (bias) {
        a += __bfloat162float(bias[h * p.hd + i]);
        b += __bfloat162float(bias[h * p.hd + i + half]);
      }
      if (head < p.nq + p.nkv) {
        const float2 cs = p.rope[(size_t)pos * half + i];
        const float ra = a * cs.x - b * cs.y, rb = b * cs.x + a * cs.y;
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
    ok = cbar_and(run_phase(P_OPROJ, l, [&](int item, float a, float b) {
      atomicAdd(p.x + 2 * item, a);
      if (2 * item + 1 < p.H) atomicAdd(p.x + 2 * item + 1, b);
    }));
    stamp(1);
    ++phase_no;
    if (!(ok = ok && grid_barrier(p, gen))) break;

    // ---- GATEUP
    stamp(0);
    stage_norm(p, xs, scratch, p.x, w.post_norm, p.H);
    ok = cbar_and(run_phase(P_GATEUP, l, [&](int item, float gt, float up) {
      p.act[item] = (gt / (1.f + expf(-gt))) * up;
    }));
    stamp(1);
    ++phase_no;
    if (!(ok = ok && grid_barrier(p, gen))) break;

    // ---- DOWN
    stamp(0);
    stage_copy(xs, p.act, p.I);
    ok = cbar_and(run_phase(P_DOWN, l, [&](int item, float a, float) { atomicAdd(p.x + item, a); }));
    stamp(1);
    ++phase_no;
    if (!(ok = ok && grid_barrier(p, gen))) break;
  }

  // ---- LM head: logits and the greedy argmax (lowest index among equal maxima)
  if (ok) {
    stamp(0);
    stage_norm(p, xs, scratch, p.x, p.final_norm, p.H);
    auto take = [&](int r, float v) {
      p.logits[r] = v;
      if (!isfinite(v)) nonfinite = true;
      if (v > best_v || best_i < 0) {  // a warp sees its rows in increasing order
        best_v = v;
        best_i = r;
      }
    };
    ok = cbar_and(run_phase(P_LM, p.L, [&](int item, float a, float b) {
      take(2 * item, a);
      if (2 * item + 1 < p.V) take(2 * item + 1, b);
    }));
    if (lane == 0) {
      s_key[warp] = best_i >= 0 ? argmax_key(best_v, best_i) : 0ull;
      s_bad[warp] = nonfinite;
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
         d.H % 8 == 0 && d.I % 8 == 0 && (size_t)step_xs_floats(d) * 4 + 16 * step::SLOT <= 220 * 1024;
}

size_t step_part_bytes(const Dims& d) {
  return (size_t)d.nq * step::MAX_SPLIT * (d.hd + 2) * sizeof(float);
}

cudaError_t step_set_attributes(const Dims& d, int* nslots_out, size_t* smem_out) {
  const size_t xs = (size_t)step_xs_floats(d) * 4;
  int ns = (int)((220 * 1024 - xs) / step::SLOT);
  if (ns > step::MAX_SLOTS) ns = step::MAX_SLOTS;
  const size_t smem = (size_t)ns * step::SLOT + xs;
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
  p.nslots = a.nslots; p.xs_floats = step_xs_floats(a.d);
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
