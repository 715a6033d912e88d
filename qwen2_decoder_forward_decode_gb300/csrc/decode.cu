// Decode-step kernels of one sequence (batch 1): the HBM-bound path.
//
// Per layer, in launch order ("LLM Speedrun: Architecture", Transformer architecture and
// Implementing Qwen; "augur", Features):
//   qkv    : RMSNorm(x) -> q/k/v projections + bias -> split-half RoPE -> KV append
//   attn   : GQA attention of the new token over the cache, context split into chunks
//            that leave softmax partials (maximum, sum, unnormalised output)
//   oproj  : merge of those partials in the prologue, then x += Wo . attn
//   resid  : the down projection, x += Wd . act
//   gateup : RMSNorm(x) -> gate/up projections -> SwiGLU
// then the LM head: final RMSNorm -> logits = E . h -> greedy argmax.
//
// Every projection is a GEMV whose weight rows stream once from HBM through per-warp rings
// of shared-memory slots filled by 1-D bulk copies (TMA); see the GEMV kernel below.
#include "common.cuh"
#include "internal.h"

#include <math.h>
#include <stdlib.h>

namespace qw {

constexpr int GEMV_WARPS = 8;

// ---- input-vector prologues ------------------------------------------------------------

// Four consecutive gains as fp32 (weights: read-only path).
__device__ __forceinline__ float4 load_gain4(const float* g, int j) {
  return __ldg(reinterpret_cast<const float4*>(g) + j);
}
__device__ __forceinline__ float4 load_gain4(const bf16* g, int j) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(g) + j);
  return make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
}

constexpr int PRO_BATCH = 4;  // float4 loads per thread kept in flight by the prologues

// xs = x / sqrt(mean(x^2) + eps) * gain, K % 4 == 0. The loads of x and of the gains are
// issued in batches of PRO_BATCH per thread before any is used, so the prologue costs one
// memory round trip per 4 * 4 * blockDim elements instead of one per loop iteration.
template <typename T>
__device__ __forceinline__ void prologue_norm(float* xs, float* gs, float* scratch, const float* x,
                                              const T* gain, int K, float eps) {
  const int n4 = K >> 2;
  float4* xs4 = reinterpret_cast<float4*>(xs);
  float4* gs4 = reinterpret_cast<float4*>(gs);
  float ss = 0.f;
  for (int base = threadIdx.x; base < n4; base += PRO_BATCH * blockDim.x) {
    float4 v[PRO_BATCH], g[PRO_BATCH];
#pragma unroll
    for (int i = 0; i < PRO_BATCH; ++i) {
      const int j = base + i * blockDim.x;
      v[i] = j < n4 ? __ldcg(reinterpret_cast<const float4*>(x) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      g[i] = j < n4 ? load_gain4(gain, j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < PRO_BATCH; ++i) {
      const int j = base + i * blockDim.x;
      if (j < n4) {
        xs4[j] = v[i];
        gs4[j] = g[i];
        ss = fmaf(v[i].x, v[i].x, fmaf(v[i].y, v[i].y, fmaf(v[i].z, v[i].z, fmaf(v[i].w, v[i].w, ss))));
      }
    }
  }
  ss = block_sum(ss, scratch);
  const float inv = rsqrtf(ss / (float)K + eps);
  for (int j = threadIdx.x; j < n4; j += blockDim.x) {
    float4 v = xs4[j];
    const float4 g = gs4[j];
    v.x = v.x * inv * g.x;
    v.y = v.y * inv * g.y;
    v.z = v.z * inv * g.z;
    v.w = v.w * inv * g.w;
    xs4[j] = v;
  }
}

__device__ __forceinline__ void prologue_copy(float* xs, const float* x, int K) {
  const int n4 = K >> 2;
  float4* xs4 = reinterpret_cast<float4*>(xs);
  for (int base = threadIdx.x; base < n4; base += PRO_BATCH * blockDim.x) {
    float4 v[PRO_BATCH];
#pragma unroll
    for (int i = 0; i < PRO_BATCH; ++i) {
      const int j = base + i * blockDim.x;
      v[i] = j < n4 ? __ldcg(reinterpret_cast<const float4*>(x) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < PRO_BATCH; ++i) {
      const int j = base + i * blockDim.x;
      if (j < n4) xs4[j] = v[i];
    }
  }
}

// ---- GEMV ops ----------------------------------------------------------------------------
//
// An item is RPI weight rows that one warp (or KS warps, splitting K) reduces together:
// the RoPE pair (i, i + hd/2) of a head, gate row i with up row i, or consecutive rows.

// q/k/v rows in RoPE pairs (i, i + hd/2) of one head; items run over q heads, k heads,
// v heads, hd/2 pairs each. T: weight type, KV: cache element type.
template <typename T, typename KV>
struct OpQKV {
  static constexpr bool PAIRED = true, NORM = true;
  static constexpr bool L2_PREWAIT = false;
  static constexpr bool LANE_EPI = true;
  static constexpr int SLOT_KNOB = 0;
  static constexpr int XS_MULT = 2;         // staged floats per K (input, gains)
  static constexpr bool DIRECT_OK = false;  // may read its input straight into registers
  __host__ __device__ int xs_extra() const { return 0; }
  static constexpr int RPI = 2;
  int K, n_items, hd, nq, nkv, cap;
  const T *wq, *wk, *wv, *bq, *bk, *bv, *gain;
  const float* x;
  float eps;
  const int* d_pos;
  const float2* rope;  // [cap][hd/2] (cos, sin)
  float* q_out;
  KV *kc, *vc;  // [nkv][cap][hd] of this layer and sequence
  int* err;     // ERR_RANGE: a key or value outside the fp16 range of the cache
  int pos;

  // the position is set by the previous step's LM head, finished before this step began
  __device__ void pre() { pos = __ldcg(d_pos); }
  __device__ void prologue(float* xs, float* gs, float* scratch) { prologue_norm(xs, gs, scratch, x, gain, K, eps); }
  // row r (0: i, 1: i + hd/2) of item (head, i)
  __device__ const T* row(int item, int r) const {
    const int half = hd >> 1;
    int head = item / half;
    const int rr = item - head * half + r * half;
    if (head < nq) return wq + (size_t)(head * hd + rr) * K;
    head -= nq;
    if (head < nkv) return wk + (size_t)(head * hd + rr) * K;
    head -= nkv;
    return wv + (size_t)(head * hd + rr) * K;
  }
  __device__ const float* xin() const { return x; }
  // bias pair and (cos, sin) of the item, loaded before its weights are waited for
  struct Epi {
    float ba, bb;
    float2 cs;
  };
  __device__ Epi epi_load(int item) const {
    const int half = hd >> 1;
    int head = item / half;
    const int i = item - head * half;
    const T* bias;
    int h;
    if (head < nq) { bias = bq; h = head; }
    else if (head < nq + nkv) { bias = bk; h = head - nq; }
    else { bias = bv; h = head - nq - nkv; }
    Epi e;
    e.ba = bias ? to_f32(bias[h * hd + i]) : 0.f;
    e.bb = bias ? to_f32(bias[h * hd + i + half]) : 0.f;
    e.cs = head < nq + nkv ? rope[(size_t)pos * half + i] : make_float2(1.f, 0.f);
    return e;
  }
  __device__ void epilogue(int item, float a, float b, const Epi& e) {
    const int half = hd >> 1;
    int head = item / half;
    const int i = item - head * half;
    int h;
    if (head < nq) h = head;
    else if (head < nq + nkv) h = head - nq;
    else h = head - nq - nkv;
    a += e.ba;
    b += e.bb;
    if (head < nq + nkv) {  // rotate (split-half RoPE): pair (i, i + hd/2)
      const float2 cs = e.cs;
      const float ra = a * cs.x - b * cs.y;
      const float rb = b * cs.x + a * cs.y;
      a = ra;
      b = rb;
    }
    if (head < nq) {
      q_out[h * hd + i] = a;
      q_out[h * hd + i + half] = b;
    } else {
      KV* c = head < nq + nkv ? kc : vc;
      KV* dst = c + ((size_t)h * cap + pos) * hd;
      store_kv(dst + i, a, err);
      store_kv(dst + i + half, b, err);
    }
  }
  __device__ void finish() {}
};

// gate row i and up row i -> act[i] = silu(gate) * up
template <typename T>
struct OpGateUp {
  static constexpr bool PAIRED = true, NORM = true;
  static constexpr bool L2_PREWAIT = true;  // resident during attention, when HBM is idle
  static constexpr bool LANE_EPI = true;    // epilogues of different items may run on any lanes
  static constexpr int SLOT_KNOB = 1;
  static constexpr int XS_MULT = 2;         // staged floats per K (input, gains)
  static constexpr bool DIRECT_OK = false;  // may read its input straight into registers
  __host__ __device__ int xs_extra() const { return 0; }
  static constexpr int RPI = 2;
  int K, n_items;
  const T *wg, *wu, *gain;
  const float* x;
  float eps;
  float* act;
  __device__ void pre() {}
  __device__ void prologue(float* xs, float* gs, float* scratch) { prologue_norm(xs, gs, scratch, x, gain, K, eps); }
  __device__ const T* row(int item, int r) const { return (r == 0 ? wg : wu) + (size_t)item * K; }
  __device__ const float* xin() const { return x; }
  struct Epi {};
  __device__ Epi epi_load(int) const { return Epi{}; }
  __device__ void epilogue(int item, float g, float u, const Epi&) { act[item] = (g / (1.f + expf(-g))) * u; }
  __device__ void finish() {}
};

// y[r] += W[r, :] . in, RPI consecutive rows per item
template <typename T, int RPI_>
struct OpResid {
  static constexpr bool PAIRED = false, NORM = false;
  static constexpr bool L2_PREWAIT = false;
  static constexpr bool LANE_EPI = true;
  static constexpr int SLOT_KNOB = 0;
  static constexpr int XS_MULT = 1;         // staged floats per K (input, gains)
  static constexpr bool DIRECT_OK = true;  // may read its input straight into registers
  __host__ __device__ int xs_extra() const { return 0; }
  static constexpr int RPI = RPI_;
  int K, n_items, N;
  const T* W;
  const float* in;
  float* y;
  __device__ void pre() {}
  __device__ void prologue(float* xs, float*, float*) { prologue_copy(xs, in, K); }
  __device__ const T* row(int item, int r) const {
    const int rr = RPI * item + r;
    return rr < N ? W + (size_t)rr * K : nullptr;
  }
  __device__ const float* xin() const { return in; }
  struct Epi {};
  __device__ Epi epi_load(int) const { return Epi{}; }
  // y += a as one reduction without a return value (each row has exactly one writer, so
  // the sum is the same single rounding as a load-add-store, without the load latency)
  __device__ void epilogue(int item, float a, float b, const Epi&) {
    const int r0 = RPI * item;
    atomicAdd(y + r0, a);
    if (RPI == 2 && r0 + 1 < N) atomicAdd(y + r0 + 1, b);
  }
  __device__ void finish() {}
};

// x += Wo . o, where o (the attention output of all heads) is merged in the prologue from
// the attention kernel's per-chunk partials: per head h and chunk s the maximum m_s, the
// sum of exponentials l_s and the unnormalised output O_s; o_h = sum_s w_s O_s with
// w_s = exp(m_s - M) / sum_s' l_s' exp(m_s' - M) (exact log-sum-exp combine, chunk order).
template <typename T>
struct OpOProj {
  static constexpr bool PAIRED = false, NORM = false;
  static constexpr bool L2_PREWAIT = false;
  static constexpr bool LANE_EPI = true;
  static constexpr int SLOT_KNOB = 0;
  static constexpr int XS_MULT = 1;
  static constexpr bool DIRECT_OK = false;
  static constexpr int RPI = 2;
  static constexpr int MB = 8;    // chunks whose partials one batch of loads covers
  static constexpr int EPT4 = 2;  // 4-element vectors of the input per thread: K <= 8 * 256
  int K, n_items, N;            // K = nq * hd
  const T* W;
  const float* part;            // [nq][nsplit_max][attn_part_stride(hd)]
  int nq, hd, nsplit_max, chunk_min;
  const int* d_pos;
  int ctx;
  float* y;
  __host__ __device__ int xs_extra() const { return 2 * nq * nsplit_max; }  // (m, l), then weights
  // the position is set by the previous step's LM head, finished before this step began
  __device__ void pre() { ctx = __ldcg(d_pos) + 1; }
  // One round trip for up to MB chunks: the thread's partial outputs of the first MB
  // chunks (16-byte vectors, 4 consecutive outputs of one head) are requested together
  // with the (m, l) pairs, before any of them is used.
  __device__ void prologue(float* xs, float*, float*) {
    const int chunk = max(chunk_min, (ctx + nsplit_max - 1) / nsplit_max);
    const int ns = (ctx + chunk - 1) / chunk;
    const int ps = attn_part_stride(hd);
    float* mw = xs + K;  // [nq][nsplit_max] maxima, then weights; [nq][nsplit_max] sums
    const int nt = blockDim.x;
    const float* src[EPT4];  // partial row of (head, chunk 0) at this thread's 4 outputs
    int hw[EPT4];            // offset of the head's weights in mw
#pragma unroll
    for (int e = 0; e < EPT4; ++e) {
      const int idx = 4 * (threadIdx.x + e * nt);
      const int h = idx / hd;
      src[e] = idx < K ? part + (size_t)h * nsplit_max * ps + (idx - h * hd) : nullptr;
      hw[e] = h * nsplit_max;
    }
    float4 v[EPT4][MB];
    auto load = [&](int s0) {
#pragma unroll
      for (int e = 0; e < EPT4; ++e)
#pragma unroll
        for (int u = 0; u < MB; ++u)
          v[e][u] = src[e] && s0 + u < ns ? __ldcg(reinterpret_cast<const float4*>(src[e] + (size_t)(s0 + u) * ps))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    load(0);
    for (int i = threadIdx.x; i < nq * ns; i += nt) {
      const int h = i / ns, sp = i - h * ns;
      const float* pp = part + ((size_t)h * nsplit_max + sp) * ps + hd;
      const float m = __ldcg(pp), l = __ldcg(pp + 1);
      mw[h * nsplit_max + sp] = m;
      mw[(nq + h) * nsplit_max + sp] = l;
    }
    __syncthreads();
    for (int h = threadIdx.x; h < nq; h += nt) {
      float M = -INFINITY;
      for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, mw[h * nsplit_max + sp]);
      float L = 0.f;
      for (int sp = 0; sp < ns; ++sp) {
        const float w = expf(mw[h * nsplit_max + sp] - M);
        mw[h * nsplit_max + sp] = w;
        L = fmaf(mw[(nq + h) * nsplit_max + sp], w, L);
      }
      const float inv = 1.f / L;
      for (int sp = 0; sp < ns; ++sp) mw[h * nsplit_max + sp] *= inv;
    }
    __syncthreads();
    float4 acc[EPT4];
#pragma unroll
    for (int e = 0; e < EPT4; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < ns; s0 += MB) {
      if (s0) load(s0);
#pragma unroll
      for (int e = 0; e < EPT4; ++e)
#pragma unroll
        for (int u = 0; u < MB; ++u) {
          if (src[e] && s0 + u < ns) {  // threads past the input vector own no head
            const float w = mw[hw[e] + s0 + u];
            acc[e].x = fmaf(v[e][u].x, w, acc[e].x);
            acc[e].y = fmaf(v[e][u].y, w, acc[e].y);
            acc[e].z = fmaf(v[e][u].z, w, acc[e].z);
            acc[e].w = fmaf(v[e][u].w, w, acc[e].w);
          }
        }
    }
#pragma unroll
    for (int e = 0; e < EPT4; ++e)
      if (src[e]) reinterpret_cast<float4*>(xs)[threadIdx.x + e * nt] = acc[e];
  }
  __device__ const T* row(int item, int r) const {
    const int rr = 2 * item + r;
    return rr < N ? W + (size_t)rr * K : nullptr;
  }
  __device__ const float* xin() const { return nullptr; }
  struct Epi {};
  __device__ Epi epi_load(int) const { return Epi{}; }
  __device__ void epilogue(int item, float a, float b, const Epi&) {
    const int r0 = 2 * item;
    atomicAdd(y + r0, a);
    if (r0 + 1 < N) atomicAdd(y + r0 + 1, b);
  }
  __device__ void finish() {}
};

// logits[r] = W[r, :] . norm(x); greedy argmax over all rows
template <typename T>
struct OpLMHead {
  static constexpr bool PAIRED = false, NORM = true;
  static constexpr bool L2_PREWAIT = false;
  static constexpr bool LANE_EPI = false;  // the argmax state lives in lane 0
  static constexpr int SLOT_KNOB = 2;
  static constexpr int XS_MULT = 2;         // staged floats per K (input, gains)
  static constexpr bool DIRECT_OK = false;  // may read its input straight into registers
  __host__ __device__ int xs_extra() const { return 0; }
  static constexpr int RPI = 2;
  int K, n_items, N;
  const T *W, *gain;
  const float* x;
  float eps;
  float* logits;
  Finalize f;
  float best_v;
  int best_i;
  bool nonfinite;
  __device__ void pre() {}
  __device__ void prologue(float* xs, float* gs, float* scratch) {
    prologue_norm(xs, gs, scratch, x, gain, K, eps);
    best_v = -INFINITY;
    best_i = -1;
    nonfinite = false;
  }
  __device__ const T* row(int item, int r) const {
    const int rr = 2 * item + r;
    return rr < N ? W + (size_t)rr * K : nullptr;
  }
  __device__ const float* xin() const { return x; }
  __device__ void take(int r, float v) {
    logits[r] = v;
    if (!isfinite(v)) nonfinite = true;
    if (v > best_v || best_i < 0) { best_v = v; best_i = r; }  // a thread sees rows in increasing order
  }
  struct Epi {};
  __device__ Epi epi_load(int) const { return Epi{}; }
  __device__ void epilogue(int item, float a, float b, const Epi&) {
    take(2 * item, a);
    if (2 * item + 1 < N) take(2 * item + 1, b);
  }
  __device__ void finish() {
    __shared__ unsigned long long s_key[GEMV_WARPS];
    __shared__ int s_bad[GEMV_WARPS];
    __shared__ bool s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
      s_key[warp] = best_i >= 0 ? argmax_key(best_v, best_i) : 0ull;
      s_bad[warp] = nonfinite;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long k = 0;
      int bad = 0;
      for (int w = 0; w < GEMV_WARPS; ++w) {
        k = s_key[w] > k ? s_key[w] : k;
        bad |= s_bad[w];
      }
      if (k) atomicMax(f.key, k);
      if (bad) atomicOr(f.err, ERR_NONFINITE);
      __threadfence();
      const unsigned t = atomicAdd(f.counter, 1u);
      s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (s_last && threadIdx.x == 0) {
      __threadfence();
      const unsigned long long k = atomicAdd(f.key, 0ull);
      const int idx = argmax_key_index(k);
      *f.tok = idx;
      if (f.hist) {
        const int n = __ldcg(f.hist_n);
        if (n < f.hist_cap) f.hist[n] = idx;
        *f.hist_n = n + 1;
      }
      if (f.pos_set >= 0) *f.pos = f.pos_set;
      else *f.pos = __ldcg(f.pos) + 1;
      *f.key = 0ull;
      *f.counter = 0u;
    }
  }
};

// ---- the GEMV kernel ---------------------------------------------------------------------
//
// Each warp runs its own pipeline: it owns NS slots of shared memory and NS mbarriers, and
// lane 0 bulk-copies (TMA, 1-D) the rows of its next items into free slots while the warp
// multiplies earlier ones with the input-vector slice held in registers. Warps never wait
// for each other in the main loop (KS > 1 warps sharing an item meet at a named barrier).
// The first NS items are requested before griddepcontrol.wait, and a CTA stays under half
// an SM, so under programmatic dependent launch the next kernel's weights are in flight
// while this one finishes. Partial sums over K segments add in a fixed order.
// Regions of a later kernel's weights that every CTA asks L2 to fetch before its dependency
// wait (the HBM stream then keeps running while this kernel waits and computes). Each region
// is cut into pieces of `piece` bytes; CTA b requests pieces b, b + grid, ... in address
// order, interleaving the regions, so data arrives roughly in the order it is consumed.
struct L2Ahead {
  const char* ptr[3];
  unsigned long long bytes[3];
  int n;
  unsigned piece;
};

struct GemvCfg {
  int KS, NS, slot_bytes, x_direct, pf_dist;
  int prewait_bytes;  // per warp: weight bytes beyond the ring prefetched into L2 before the wait
  int cpasync;        // 1: every lane fills the ring with 16-byte cp.async (else lane 0, bulk copies)
  L2Ahead ahead;
  int* err;
  unsigned long long* tl;  // timeline slots or null
};
constexpr int MAX_SLOTS = 8;
constexpr int MAX_DEFER = 16;  // items per warp whose K-split partials wait in shared memory

template <typename T, int MAXV, class Op>
__global__ void __launch_bounds__(GEMV_WARPS * 32, 2)
gemv_kernel(const Op op_in, const GemvCfg c) {
  Op op = op_in;
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ __align__(8) unsigned long long bars[GEMV_WARPS][MAX_SLOTS];
  __shared__ float scratch[32];
  __shared__ float red[GEMV_WARPS][2];
  __shared__ float red_all[GEMV_WARPS][MAX_DEFER][2];
  __shared__ volatile int s_abort[GEMV_WARPS];
  constexpr int VN = Vec<T>::N;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int KS = c.KS, NS = c.NS, RG = GEMV_WARPS / KS;
  const int rg = warp / KS, ks = warp - rg * KS;
  const int nvec = op.K / VN;
  const int seg = (nvec + KS - 1) / KS;
  const int v0 = ks * seg, v1 = min(nvec, v0 + seg);
  const uint32_t seg_bytes = (uint32_t)(v1 > v0 ? v1 - v0 : 0) * 16u;
  // items of this warp: first + k * step
  const int first = (int)blockIdx.x * RG + rg, step = (int)gridDim.x * RG;
  const int my_items = first < op.n_items ? (op.n_items - 1 - first) / step + 1 : 0;
  unsigned char* wslots = dsm + (size_t)warp * NS * c.slot_bytes;
  const uint32_t wslot0 = smem_addr(wslots);
  const uint32_t bar0 = smem_addr(&bars[warp][0]);
  float* xs = reinterpret_cast<float*>(dsm + (size_t)GEMV_WARPS * NS * c.slot_bytes);

  auto prefetch = [&](int k) {  // lane 0: ask L2 for item k's row segments ahead of use
    const int item = first + k * step;
    const T* r0 = op.row(item, 0);
    const T* r1 = Op::RPI == 2 ? op.row(item, 1) : nullptr;
    if (seg_bytes) {
      prefetch_l2_bulk(reinterpret_cast<const unsigned char*>(r0) + (size_t)v0 * 16, seg_bytes);
      if (r1) prefetch_l2_bulk(reinterpret_cast<const unsigned char*>(r1) + (size_t)v0 * 16, seg_bytes);
    }
  };
  auto issue_cp = [&](int k) {  // every lane: its 16-byte vectors of item k's row segments
    const int slot = k % NS;
    const int item = first + k * step;
    const unsigned char* r0 = reinterpret_cast<const unsigned char*>(op.row(item, 0)) + (size_t)v0 * 16;
    const T* r1t = Op::RPI == 2 ? op.row(item, 1) : nullptr;
    const uint32_t dst = wslot0 + slot * c.slot_bytes;
    const int nv = (int)(seg_bytes >> 4);
    for (int v = lane; v < nv; v += 32) cp_async16_s(dst + 16 * v, r0 + 16 * v);
    if (r1t) {
      const unsigned char* r1 = reinterpret_cast<const unsigned char*>(r1t) + (size_t)v0 * 16;
      for (int v = lane; v < nv; v += 32) cp_async16_s(dst + seg_bytes + 16 * v, r1 + 16 * v);
    }
    cp_async_arrive_noinc(bar0 + 8 * slot);
  };
  auto issue = [&](int k) {  // lane 0: copy this warp's K segment of item k's rows
    const int slot = k % NS;
    const int item = first + k * step;
    const T* r0 = op.row(item, 0);
    const T* r1 = Op::RPI == 2 ? op.row(item, 1) : nullptr;
    const uint32_t bar = bar0 + 8 * slot;
    mbar_expect_tx(bar, seg_bytes * (r1 ? 2u : 1u));
    const uint32_t dst = wslot0 + slot * c.slot_bytes;
    if (seg_bytes) {
      bulk_copy_g2s(dst, reinterpret_cast<const unsigned char*>(r0) + (size_t)v0 * 16, seg_bytes, bar);
      if (r1) bulk_copy_g2s(dst + seg_bytes, reinterpret_cast<const unsigned char*>(r1) + (size_t)v0 * 16, seg_bytes, bar);
    }
  };

  tl_stamp(c.tl, 0);
  const int n0 = min(NS, my_items);  // weights do not depend on upstream kernels
  if (c.cpasync) {
    if (lane == 0) {
      s_abort[warp] = 0;
      for (int sl = 0; sl < NS; ++sl) mbar_init(bar0 + 8 * sl, 32);  // one arrival per lane
      mbar_fence_init();
    }
    __syncwarp();
    for (int k = 0; k < n0; ++k) issue_cp(k);
  }
  if (lane == 0) {
    if (!c.cpasync) {
      s_abort[warp] = 0;
      for (int sl = 0; sl < NS; ++sl) mbar_init(bar0 + 8 * sl, 1);
      mbar_fence_init();
      for (int k = 0; k < n0; ++k) issue(k);
    }
    // and while the upstream kernels finish, the next items stream into L2
    const uint32_t item_bytes = seg_bytes * (uint32_t)Op::RPI;
    int n_pf = c.pf_dist;
    if (Op::L2_PREWAIT && item_bytes && c.prewait_bytes > 0 && (int)(c.prewait_bytes / item_bytes) > n_pf)
      n_pf = (int)(c.prewait_bytes / item_bytes);
    for (int k = n0; k < min(NS + n_pf, my_items); ++k) prefetch(k);
    if (warp == GEMV_WARPS - 1 && c.ahead.n) {  // a later kernel's weights, into L2
      const unsigned long long np = (c.ahead.bytes[0] + c.ahead.piece - 1) / c.ahead.piece;
      for (unsigned long long j = blockIdx.x; j < np; j += gridDim.x)
        for (int r = 0; r < c.ahead.n; ++r) {
          const unsigned long long a = j * c.ahead.piece;
          if (a >= c.ahead.bytes[r]) continue;
          unsigned long long n = c.ahead.bytes[r] - a;
          if (n > c.ahead.piece) n = c.ahead.piece;
          prefetch_l2_bulk(c.ahead.ptr[r] + a, (uint32_t)(n & ~15ull));
        }
    }
  }
  // inputs of the epilogue that do not depend on upstream kernels (first two items)
  op.pre();
  typename Op::Epi pe[2];
  if (my_items > 0) pe[0] = op.epi_load(first);
  if (my_items > 1) pe[1] = op.epi_load(first + step);
  __syncwarp();
  pdl_trigger();  // the next kernel may become resident and start its own weight stream
  pdl_wait();
  tl_stamp(c.tl, 1);
  if (!c.x_direct) op.prologue(xs, xs + op.K, scratch);
  __syncthreads();

  float xr[MAXV][VN];
#pragma unroll
  for (int q = 0; q < MAXV; ++q) {
    const int v = v0 + lane + 32 * q;
    if (c.x_direct) {
#pragma unroll
      for (int e = 0; e < VN; e += 4) {
        const float4 t = v < v1 ? __ldcg(reinterpret_cast<const float4*>(op.xin()) + (v * VN + e) / 4)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        xr[q][e] = t.x; xr[q][e + 1] = t.y; xr[q][e + 2] = t.z; xr[q][e + 3] = t.w;
      }
    } else if constexpr (VN == 8) {
      // Two 16-byte shared loads per vector. Lane l's vector starts 32 bytes after lane
      // l-1's, so lanes l and l+4 would share banks; lanes with bit 2 set take the halves
      // in the other order, and each 8-lane phase of a 16-byte load hits all 32 banks once.
      const bool sw = (lane & 4) != 0;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
      if (v < v1) {
        const float4* p = reinterpret_cast<const float4*>(xs) + 2 * v;
        a = p[sw ? 1 : 0];
        b = p[sw ? 0 : 1];
      }
      const float4 lo = sw ? b : a, hi = sw ? a : b;
      xr[q][0] = lo.x; xr[q][1] = lo.y; xr[q][2] = lo.z; xr[q][3] = lo.w;
      xr[q][4] = hi.x; xr[q][5] = hi.y; xr[q][6] = hi.z; xr[q][7] = hi.w;
    } else {  // one 16-byte vector per lane, consecutive: conflict-free
      const float4 a = v < v1 ? reinterpret_cast<const float4*>(xs)[v] : make_float4(0.f, 0.f, 0.f, 0.f);
      xr[q][0] = a.x; xr[q][1] = a.y; xr[q][2] = a.z; xr[q][3] = a.w;
    }
  }

  bool timed_out = false;
  int issued = n0, consumed = 0;
  // K split over KS warps with at most MAX_DEFER items per warp: every warp streams its
  // own segments without waiting for the others, parks its partial sums in shared memory,
  // and the KS partials of each item are added (in warp order) once, after the loop.
  const bool deferred = Op::LANE_EPI && KS > 1 && (op.n_items + step - 1) / step <= MAX_DEFER;  // CTA-uniform
  if (deferred) {
    for (int k = 0; k < my_items; ++k) {
      const int slot = k % NS;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * slot, (uint32_t)((k / NS) & 1)))) {
        timed_out = true;
        if (lane == 0) s_abort[rg] = 1;
        break;
      }
      consumed = k + 1;
      const uint4* s0 = reinterpret_cast<const uint4*>(wslots + (size_t)slot * c.slot_bytes);
      const uint4* s1 = reinterpret_cast<const uint4*>(wslots + (size_t)slot * c.slot_bytes + seg_bytes);
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int q = 0; q < MAXV; ++q) {
        const int v = lane + 32 * q;
        if (v0 + v < v1) {
          a0 = dotv(s0[v], xr[q], a0, T());
          if (Op::RPI == 2) a1 = dotv(s1[v], xr[q], a1, T());
        }
      }
      __syncwarp();
      if (k + NS < my_items) {  // slot free: request item k + NS
        if (c.cpasync) {
          issue_cp(k + NS);
        } else if (lane == 0) {
          fence_proxy_async();
          issue(k + NS);
        }
        ++issued;
      }
      a0 = warp_sum(a0);
      if (Op::RPI == 2) a1 = warp_sum(a1);
      if (lane == 0) {
        red_all[warp][k][0] = a0;
        red_all[warp][k][1] = a1;
      }
    }
    __syncthreads();
    if (ks == 0 && !s_abort[rg]) {  // lane k finishes item k of this row group
      for (int k = lane; k < my_items; k += 32) {
        float a0 = 0.f, a1 = 0.f;
        for (int j = 0; j < KS; ++j) {
          a0 += red_all[warp + j][k][0];
          a1 += red_all[warp + j][k][1];
        }
        const int item = first + k * step;
        const typename Op::Epi epi = k == 0 ? pe[0] : k == 1 ? pe[1] : op.epi_load(item);
        op.epilogue(item, a0, a1, epi);
      }
    }
  }
  for (int k = 0; k < my_items && !deferred; ++k) {
    const int slot = k % NS;
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * slot, (uint32_t)((k / NS) & 1)));
    if (KS > 1) {  // the KS warps sharing these items give up together
      if (!ok && lane == 0) s_abort[rg] = 1;
      asm volatile("bar.sync %0, %1;" ::"r"(1 + rg), "r"(KS * 32) : "memory");
      ok = s_abort[rg] == 0;
    }
    if (!ok) { timed_out = true; break; }
    consumed = k + 1;
    const int item = first + k * step;
    const typename Op::Epi epi = k == 0 ? pe[0] : k == 1 ? pe[1] : op.epi_load(item);
    const uint4* s0 = reinterpret_cast<const uint4*>(wslots + (size_t)slot * c.slot_bytes);
    const uint4* s1 = reinterpret_cast<const uint4*>(wslots + (size_t)slot * c.slot_bytes + seg_bytes);
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
      const int v = lane + 32 * q;
      if (v0 + v < v1) {
        a0 = dotv(s0[v], xr[q], a0, T());
        if (Op::RPI == 2) a1 = dotv(s1[v], xr[q], a1, T());
      }
    }
    __syncwarp();
    if (k + NS < my_items) {  // slot free: request item k + NS
      if (c.cpasync) {
        issue_cp(k + NS);
      } else if (lane == 0) {
        fence_proxy_async();
        issue(k + NS);
      }
      ++issued;
      if (lane == 0 && c.pf_dist && k + NS + c.pf_dist < my_items) prefetch(k + NS + c.pf_dist);
    }
    a0 = warp_sum(a0);
    if (Op::RPI == 2) a1 = warp_sum(a1);
    if (KS > 1) {  // the KS warps of this item meet at named barrier 1 + rg
      if (lane == 0) {
        red[warp][0] = a0;
        red[warp][1] = a1;
      }
      asm volatile("bar.sync %0, %1;" ::"r"(1 + rg), "r"(KS * 32) : "memory");
      if (ks == 0 && lane == 0) {
        a0 = 0.f;
        a1 = 0.f;
        for (int j = 0; j < KS; ++j) {
          a0 += red[warp + j][0];
          a1 += red[warp + j][1];
        }
      }
      asm volatile("bar.sync %0, %1;" ::"r"(1 + rg), "r"(KS * 32) : "memory");
    }
    if (ks == 0 && lane == 0) op.epilogue(item, a0, a1, epi);
  }
  if (timed_out && lane == 0) {
    atomicOr(c.err, ERR_TIMEOUT);
    for (int j = consumed; j < issued; ++j)  // copies in flight must land before exit
      mbar_wait_bounded(bar0 + 8 * (j % NS), (uint32_t)((j / NS) & 1));
  }
  if (c.cpasync) asm volatile("cp.async.wait_all;" ::: "memory");  // (nothing left unless a wait gave up)
  op.finish();
  tl_stamp(c.tl, 2);
}

// dynamic shared memory: per-warp slot rings and, unless x is read straight into
// registers, the input vector (and the gains of a norm prologue)
static constexpr int X_SMEM_MAX = 16 * 1024;
// Tuning: bytes of slots per warp (per kernel kind, below), the
// in-loop L2 prefetch distance in items, and the bytes per warp prefetched into L2 before
// the dependency wait; QW_GEMV_SLOT_KB / QW_GEMV_PF / QW_GEMV_PREWAIT_KB override them.
static int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  return v && *v ? std::atoi(v) : dflt;
}
// per warp: 0 the default, 1 gate/up, 2 the LM head (the last kernel of a step: no next
// kernel has to fit beside it)
static int warp_budget(int knob) {
  // 8 KB keeps the down projection's CTAs (55 KB) resident beside gate/up's (156 KB), so
  // its first weights stream while gate/up finishes (measured: 8 -> 839, 12 -> 803,
  // 16 -> 837, 20 -> 818 tok/s on the 1.5B shape)
  static const int b0 = env_int("QW_GEMV_SLOT_KB", 8) * 1024;
  static const int b1 = env_int("QW_GEMV_SLOT_KB_GU", 18) * 1024;  // measured best of 12/18/24
  static const int b2 = env_int("QW_GEMV_SLOT_KB_LM", 24) * 1024;  // of 12/18/24 (26 fits at most)
  return knob == 1 ? b1 : knob == 2 ? b2 : b0;
}
static int pf_dist() {
  static const int p = env_int("QW_GEMV_PF", 0);
  return p;
}
static int prewait_bytes() {
  static const int b = env_int("QW_GEMV_PREWAIT_KB", 0) * 1024;
  return b;
}
// ring fill: 1 = per-lane cp.async, 0 = bulk copies issued by lane 0
static int gemv_cpasync() {
  static const int v = env_int("QW_GEMV_CPASYNC", 0);
  return v;
}
// which later weights are requested into L2 ahead of use (bit 0: the o_proj kernel asks for
// gate/up, bit 1: the o_proj kernel asks for down, bit 2: the gate/up kernel asks for down)
int l2_ahead_mask() {
  static const int v = env_int("QW_L2_AHEAD", 0);
  return v;
}
static unsigned l2_ahead_piece() {
  static const unsigned v = (unsigned)env_int("QW_L2_AHEAD_PIECE_KB", 32) * 1024u;
  return v;
}

static int maxv_for(int nvec, int KS) {
  const int need = (((nvec + KS - 1) / KS) + 31) / 32;
  return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : need <= 6 ? 6 : need <= 8 ? 8 : need <= 12 ? 12 : 99;
}

struct GemvPlan {
  GemvCfg c;
  int maxv, grid;
  size_t smem;
};

template <typename T, class Op>
static bool plan_gemv(const Op& op, int nsm, int* err, unsigned long long* tl, GemvPlan* p) {
  const int nvec = op.K / Vec<T>::N;
  const int x_direct = (Op::DIRECT_OK && (size_t)op.K * 4 > X_SMEM_MAX) ? 1 : 0;
  const size_t xs = x_direct ? 0 : ((size_t)Op::XS_MULT * op.K + op.xs_extra()) * 4;
  // smallest K split whose slot (RPI row segments) fits the warp budget twice and whose
  // register tile fits; then split further while too few items exist to fill every warp
  int KS = 1;
  auto slot_of = [&](int ks) { return (size_t)Op::RPI * ((nvec + ks - 1) / ks) * 16; };
  const int WARP_BUDGET = warp_budget(Op::SLOT_KNOB);
  while (KS < GEMV_WARPS && (maxv_for(nvec, KS) > 8 || 2 * slot_of(KS) > (size_t)WARP_BUDGET)) KS *= 2;
  if (maxv_for(nvec, KS) > 12) return false;
  while (KS < GEMV_WARPS && (long long)op.n_items * KS < (long long)nsm * GEMV_WARPS) KS *= 2;
  const size_t slot = (slot_of(KS) + 127) & ~(size_t)127;
  int NS = (int)(WARP_BUDGET / slot);
  if (NS > MAX_SLOTS) NS = MAX_SLOTS;
  if (NS < 2) NS = 2;
  const size_t smem = (size_t)GEMV_WARPS * NS * slot + xs;
  if (smem > 220 * 1024) return false;
  const int RG = GEMV_WARPS / KS;
  p->c.KS = KS;
  p->c.NS = NS;
  p->c.slot_bytes = (int)slot;
  p->c.x_direct = x_direct;
  p->c.pf_dist = pf_dist();
  p->c.prewait_bytes = prewait_bytes();
  p->c.cpasync = gemv_cpasync();
  p->c.ahead = L2Ahead{};
  p->c.err = err;
  p->c.tl = tl;
  p->maxv = maxv_for(nvec, KS);
  const int groups = (op.n_items + RG - 1) / RG;
  p->grid = groups < nsm ? groups : nsm;
  p->smem = smem;
  return true;
}

template <typename T, class Op>
static cudaError_t run_gemv(const Op& op, int nsm, int* err, unsigned long long* tl, cudaStream_t s, bool pdl,
                            const L2Ahead* ahead = nullptr) {
  GemvPlan p;
  if (!plan_gemv<T, Op>(op, nsm, err, tl, &p)) return cudaErrorInvalidValue;
  if (ahead) p.c.ahead = *ahead;
  const dim3 g(p.grid), b(GEMV_WARPS * 32);
  switch (p.maxv) {
    case 1: return launch_k(gemv_kernel<T, 1, Op>, g, b, p.smem, s, pdl, op, p.c);
    case 2: return launch_k(gemv_kernel<T, 2, Op>, g, b, p.smem, s, pdl, op, p.c);
    case 4: return launch_k(gemv_kernel<T, 4, Op>, g, b, p.smem, s, pdl, op, p.c);
    case 6: return launch_k(gemv_kernel<T, 6, Op>, g, b, p.smem, s, pdl, op, p.c);
    case 8: return launch_k(gemv_kernel<T, 8, Op>, g, b, p.smem, s, pdl, op, p.c);
    default: return launch_k(gemv_kernel<T, 12, Op>, g, b, p.smem, s, pdl, op, p.c);
  }
}

template <typename T, class Op>
static cudaError_t set_gemv_attrs() {
  void* fns[6] = {(void*)gemv_kernel<T, 1, Op>, (void*)gemv_kernel<T, 2, Op>, (void*)gemv_kernel<T, 4, Op>,
                  (void*)gemv_kernel<T, 6, Op>, (void*)gemv_kernel<T, 8, Op>, (void*)gemv_kernel<T, 12, Op>};
  for (void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    if (e) return e;
    e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e) return e;
  }
  return cudaSuccess;
}

// ---- embedding ---------------------------------------------------------------------------

template <typename T>
__global__ void embed_kernel(const T* E, int V, int H, const int* tok, float* x, int* err,
                             unsigned long long* tl) {
  constexpr int VN = Vec<T>::N;
  tl_stamp(tl, 0);
  pdl_wait();
  tl_stamp(tl, 1);
  int t = __ldcg(tok);
  if (t < 0 || t >= V) {
    if (threadIdx.x == 0) atomicOr(err, ERR_TOKEN);
    t = 0;
  }
  const uint4* row = reinterpret_cast<const uint4*>(E + (size_t)t * H);
  for (int v = threadIdx.x; v < H / VN; v += blockDim.x) {
    const uint4 w = __ldg(row + v);
    float f[8];
    if (VN == 8) {
      f[0] = bf_lo(w.x); f[1] = bf_hi(w.x); f[2] = bf_lo(w.y); f[3] = bf_hi(w.y);
      f[4] = bf_lo(w.z); f[5] = bf_hi(w.z); f[6] = bf_lo(w.w); f[7] = bf_hi(w.w);
    } else {
      f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
      f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
    }
#pragma unroll
    for (int e = 0; e < VN; ++e) x[v * VN + e] = f[e];
  }
  pdl_trigger();
  tl_stamp(tl, 2);
}

// ---- host launchers ---------------------------------------------------------------------

template <typename T>
static cudaError_t set_attrs_t() {
  cudaError_t e;
  if ((e = set_gemv_attrs<T, OpQKV<T, float>>())) return e;
  if ((e = set_gemv_attrs<T, OpQKV<T, f16>>())) return e;
  if ((e = set_gemv_attrs<T, OpGateUp<T>>())) return e;
  if ((e = set_gemv_attrs<T, OpResid<T, 1>>())) return e;
  if ((e = set_gemv_attrs<T, OpResid<T, 2>>())) return e;
  if ((e = set_gemv_attrs<T, OpOProj<T>>())) return e;
  return set_gemv_attrs<T, OpLMHead<T>>();
}

cudaError_t decode_set_attributes(const Dims& d) {
  return d.dtype == 1 ? set_attrs_t<bf16>() : set_attrs_t<float>();
}

cudaError_t launch_embed(const Dims& d, const void* E, const int* tok, float* x, int* err,
                         unsigned long long* tl, cudaStream_t s, bool pdl) {
  if (d.dtype == 1)
    return launch_k(embed_kernel<bf16>, dim3(1), dim3(256), 0, s, pdl, (const bf16*)E, d.V, d.H, tok, x, err, tl);
  return launch_k(embed_kernel<float>, dim3(1), dim3(256), 0, s, pdl, (const float*)E, d.V, d.H, tok, x, err, tl);
}

template <typename T, typename KV>
static cudaError_t qkv_t(const Dims& d, const LayerPtrs& w, const float* x, const int* d_pos,
                         const float2* rope, float* q, void* kc, void* vc, int* err,
                         unsigned long long* tl, cudaStream_t s, bool pdl) {
  OpQKV<T, KV> op{};
  op.K = d.H;
  op.n_items = (d.nq + 2 * d.nkv) * (d.hd / 2);
  op.hd = d.hd; op.nq = d.nq; op.nkv = d.nkv; op.cap = d.cap;
  op.wq = (const T*)w.wq; op.wk = (const T*)w.wk; op.wv = (const T*)w.wv;
  op.bq = (const T*)w.bq; op.bk = (const T*)w.bk; op.bv = (const T*)w.bv;
  op.gain = (const T*)w.in_norm;
  op.x = x; op.eps = d.eps; op.d_pos = d_pos; op.rope = rope; op.q_out = q;
  op.kc = (KV*)kc; op.vc = (KV*)vc;
  op.err = err;
  return run_gemv<T>(op, d.nsm, err, tl, s, pdl);
}
cudaError_t launch_qkv(const Dims& d, const LayerPtrs& w, const float* x, const int* d_pos,
                       const float2* rope, float* q, void* kc, void* vc, int* err,
                       unsigned long long* tl, cudaStream_t s, bool pdl) {
  return d.dtype == 1 ? qkv_t<bf16, f16>(d, w, x, d_pos, rope, q, kc, vc, err, tl, s, pdl)
                      : qkv_t<float, float>(d, w, x, d_pos, rope, q, kc, vc, err, tl, s, pdl);
}

template <typename T>
static cudaError_t resid_t(const Dims& d, const void* W, int N, int K, const float* in, float* y,
                           int* err, unsigned long long* tl, cudaStream_t s, bool pdl) {
  if ((size_t)K * 4 > X_SMEM_MAX) {  // long rows (the down projection): one row per item
    OpResid<T, 1> op{};
    op.K = K; op.N = N; op.n_items = N; op.W = (const T*)W; op.in = in; op.y = y;
    return run_gemv<T>(op, d.nsm, err, tl, s, pdl);
  }
  OpResid<T, 2> op{};
  op.K = K; op.N = N; op.n_items = (N + 1) / 2; op.W = (const T*)W; op.in = in; op.y = y;
  return run_gemv<T>(op, d.nsm, err, tl, s, pdl);
}
cudaError_t launch_resid(const Dims& d, const void* W, int N, int K, const float* in, float* y,
                         int* err, unsigned long long* tl, cudaStream_t s, bool pdl) {
  return d.dtype == 1 ? resid_t<bf16>(d, W, N, K, in, y, err, tl, s, pdl)
                      : resid_t<float>(d, W, N, K, in, y, err, tl, s, pdl);
}

// L2 requests of a layer's MLP weights (mask bits as l2_ahead_mask: 1 gate and up, 2 down)
static L2Ahead mlp_ahead(const Dims& d, const LayerPtrs* w, int bits) {
  L2Ahead a{};
  a.piece = l2_ahead_piece();
  if (!w) return a;
  const unsigned long long mat = (unsigned long long)d.I * d.H * (d.dtype == 1 ? 2 : 4);
  if (bits & 1) {
    a.ptr[a.n] = (const char*)w->w_gate; a.bytes[a.n++] = mat;
    a.ptr[a.n] = (const char*)w->w_up; a.bytes[a.n++] = mat;
  }
  if (bits & 2) { a.ptr[a.n] = (const char*)w->w_down; a.bytes[a.n++] = mat; }
  return a;
}

template <typename T>
static cudaError_t oproj_t(const Dims& d, const void* W, const float* part, const int* d_pos, float* y, int* err,
                          unsigned long long* tl, cudaStream_t s, bool pdl, const LayerPtrs* mlp) {
  if (d.nq * d.hd > 4 * OpOProj<T>::EPT4 * GEMV_WARPS * 32 || d.hd % 4) return cudaErrorInvalidValue;
  OpOProj<T> op{};
  op.K = d.nq * d.hd; op.N = d.H; op.n_items = (d.H + 1) / 2; op.W = (const T*)W;
  op.part = part; op.nq = d.nq; op.hd = d.hd; op.nsplit_max = d.attn_nsplit; op.chunk_min = d.attn_chunk_min;
  op.d_pos = d_pos; op.y = y;
  const L2Ahead a = mlp_ahead(d, mlp, l2_ahead_mask() & 3);
  return run_gemv<T>(op, d.nsm, err, tl, s, pdl, a.n ? &a : nullptr);
}
cudaError_t launch_oproj(const Dims& d, const void* W, const float* part, const int* d_pos, float* y, int* err,
                         unsigned long long* tl, cudaStream_t s, bool pdl, const LayerPtrs* mlp) {
  return d.dtype == 1 ? oproj_t<bf16>(d, W, part, d_pos, y, err, tl, s, pdl, mlp)
                      : oproj_t<float>(d, W, part, d_pos, y, err, tl, s, pdl, mlp);
}

template <typename T>
static cudaError_t gateup_t(const Dims& d, const LayerPtrs& w, const float* x, float* act, int* err,
                            unsigned long long* tl, cudaStream_t s, bool pdl) {
  OpGateUp<T> op{};
  op.K = d.H; op.n_items = d.I; op.wg = (const T*)w.w_gate; op.wu = (const T*)w.w_up;
  op.gain = (const T*)w.post_norm; op.x = x; op.eps = d.eps; op.act = act;
  const L2Ahead a = mlp_ahead(d, &w, (l2_ahead_mask() & 4) ? 2 : 0);
  return run_gemv<T>(op, d.nsm, err, tl, s, pdl, a.n ? &a : nullptr);
}
cudaError_t launch_gateup(const Dims& d, const LayerPtrs& w, const float* x, float* act, int* err,
                          unsigned long long* tl, cudaStream_t s, bool pdl) {
  return d.dtype == 1 ? gateup_t<bf16>(d, w, x, act, err, tl, s, pdl)
                      : gateup_t<float>(d, w, x, act, err, tl, s, pdl);
}

template <typename T>
static cudaError_t lmhead_t(const Dims& d, const void* W, const void* fn, const float* x,
                            float* logits, const Finalize& f, unsigned long long* tl, cudaStream_t s,
                            bool pdl) {
  OpLMHead<T> op{};
  op.K = d.H; op.N = d.V; op.n_items = (d.V + 1) / 2; op.W = (const T*)W; op.gain = (const T*)fn;
  op.x = x; op.eps = d.eps; op.logits = logits; op.f = f;
  return run_gemv<T>(op, d.nsm, f.err, tl, s, pdl);
}
cudaError_t launch_lmhead(const Dims& d, const void* W, const void* final_norm, const float* x,
                          float* logits, const Finalize& f, unsigned long long* tl, cudaStream_t s,
                          bool pdl) {
  return d.dtype == 1 ? lmhead_t<bf16>(d, W, final_norm, x, logits, f, tl, s, pdl)
                      : lmhead_t<float>(d, W, final_norm, x, logits, f, tl, s, pdl);
}

}  // namespace qw
