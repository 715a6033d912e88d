// Decode-step kernels of one sequence (batch 1): the HBM-bound path.
//
// Per layer, in launch order ("LLM Speedrun: Architecture", Transformer architecture and
// Implementing Qwen; "augur", Features):
//   qkv    : RMSNorm(x) -> q/k/v projections + bias -> split-half RoPE -> KV append
//   attn   : GQA attention of the new token over the cache, context split into chunks
//            whose softmax partials are merged by the last CTA of each KV head
//   resid  : o_proj, x += Wo . attn          (also the down projection, x += Wd . act)
//   gateup : RMSNorm(x) -> gate/up projections -> SwiGLU
// then the LM head: final RMSNorm -> logits = E . h -> greedy argmax.
//
// Every projection is a GEMV whose weight rows stream once from HBM with 16-byte
// non-allocating loads, two rows per warp, the input vector held in registers. Each
// kernel issues its first weight loads before griddepcontrol.wait, so under programmatic
// dependent launch the weight stream of kernel n+1 starts while kernel n drains.
#include "common.cuh"
#include "internal.h"

#include <math.h>

namespace qw {

constexpr int GEMV_WARPS = 8;
constexpr int GMAX = 8;  // most query heads per KV head handled by decode attention

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

// q/k/v rows in RoPE pairs (i, i + hd/2) of one head; items run over q heads, k heads,
// v heads, hd/2 pairs each. T: weight type, KV: cache element type.
template <typename T, typename KV>
struct OpQKV {
  int K, n_items, hd, nq, nkv, cap;
  const T *wq, *wk, *wv, *bq, *bk, *bv, *gain;
  const float* x;
  float eps;
  const int* d_pos;
  const float2* rope;  // [cap][hd/2] (cos, sin)
  float* q_out;
  KV *kc, *vc;  // [nkv][cap][hd] of this layer and sequence
  int pos;

  __device__ void prologue(float* xs, float* gs, float* scratch) {
    prologue_norm(xs, gs, scratch, x, gain, K, eps);
    pos = __ldcg(d_pos);
  }
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
  __device__ void epilogue(int item, float a, float b) {
    const int half = hd >> 1;
    int head = item / half;
    const int i = item - head * half;
    const T* bias;
    int h;
    if (head < nq) { bias = bq; h = head; }
    else if (head < nq + nkv) { bias = bk; h = head - nq; }
    else { bias = bv; h = head - nq - nkv; }
    if (bias) {
      a += to_f32(bias[h * hd + i]);
      b += to_f32(bias[h * hd + i + half]);
    }
    if (head < nq + nkv) {  // rotate (split-half RoPE): pair (i, i + hd/2)
      const float2 cs = rope[(size_t)pos * half + i];
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
      dst[i] = from_f32<KV>(a);
      dst[i + half] = from_f32<KV>(b);
    }
  }
  __device__ void finish(float*) {}
};

// gate row i and up row i -> act[i] = silu(gate) * up
template <typename T>
struct OpGateUp {
  int K, n_items;
  const T *wg, *wu, *gain;
  const float* x;
  float eps;
  float* act;
  __device__ void prologue(float* xs, float* gs, float* scratch) { prologue_norm(xs, gs, scratch, x, gain, K, eps); }
  __device__ const T* row(int item, int r) const {
    return (r == 0 ? wg : wu) + (size_t)item * K;
  }
  __device__ void epilogue(int item, float g, float u) {
    act[item] = (g / (1.f + expf(-g))) * u;
  }
  __device__ void finish(float*) {}
};

// y[r] += W[r, :] . in for rows (2 item, 2 item + 1)
template <typename T>
struct OpResid {
  int K, n_items, N;
  const T* W;
  const float* in;
  float* y;
  __device__ void prologue(float* xs, float*, float*) { prologue_copy(xs, in, K); }
  __device__ const T* row(int item, int r) const {
    const int rr = 2 * item + r;
    return rr < N ? W + (size_t)rr * K : nullptr;
  }
  __device__ void epilogue(int item, float a, float b) {
    const int r0 = 2 * item;
    y[r0] = __ldcg(y + r0) + a;
    if (r0 + 1 < N) y[r0 + 1] = __ldcg(y + r0 + 1) + b;
  }
  __device__ void finish(float*) {}
};

// logits[r] = W[r, :] . norm(x); greedy argmax over all rows
template <typename T>
struct OpLMHead {
  int K, n_items, N;
  const T *W, *gain;
  const float* x;
  float eps;
  float* logits;
  Finalize f;
  float best_v;
  int best_i;
  bool nonfinite;
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
  __device__ void take(int r, float v) {
    logits[r] = v;
    if (!isfinite(v)) nonfinite = true;
    if (v > best_v || best_i < 0) { best_v = v; best_i = r; }  // rows arrive in increasing order
  }
  __device__ void epilogue(int item, float a, float b) {
    take(2 * item, a);
    if (2 * item + 1 < N) take(2 * item + 1, b);
  }
  __device__ void finish(float* smem) {
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
// Warps form row groups of KS warps; a row group owns an item (two weight rows) and its
// KS warps split the inner dimension K into contiguous segments. Lane l of a warp reads
// 16-byte vectors l, l+32, ... of its segment, so each load instruction covers 512
// contiguous bytes of a row. The input-vector slice a lane needs never changes and lives
// in registers. Partial sums over segments meet in shared memory in a fixed order.
template <typename T, int MAXV, class Op>
__global__ void __launch_bounds__(GEMV_WARPS * 32)
gemv_kernel(const Op op_in, int KS) {
  Op op = op_in;
  extern __shared__ float smem[];
  __shared__ float scratch[32];
  __shared__ float red[GEMV_WARPS][2];
  constexpr int VN = Vec<T>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int RG = GEMV_WARPS / KS;
  const int rg = warp / KS, ks = warp - rg * KS;
  const int nvec = op.K / VN;
  const int seg = (nvec + KS - 1) / KS;
  const int v0 = ks * seg, v1 = min(nvec, v0 + seg);
  const int stride = gridDim.x * RG;

  uint4 w0[MAXV], w1[MAXV];
  auto load = [&](int item) {
    const T* r0 = op.row(item, 0);
    const T* r1 = op.row(item, 1);
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int v = v0 + lane + 32 * i;
      const bool ok = v < v1;
      w0[i] = ok ? ld_stream(r0 + (size_t)v * VN) : make_uint4(0, 0, 0, 0);
      w1[i] = (ok && r1) ? ld_stream(r1 + (size_t)v * VN) : make_uint4(0, 0, 0, 0);
    }
  };

  int base = blockIdx.x * RG;
  if (base + rg < op.n_items) load(base + rg);  // weights do not depend on upstream kernels
  pdl_wait();
  op.prologue(smem, smem + op.K, scratch);
  __syncthreads();
  pdl_trigger();

  float xr[MAXV][VN];
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int v = v0 + lane + 32 * i;
#pragma unroll
    for (int e = 0; e < VN; ++e) xr[i][e] = v < v1 ? smem[v * VN + e] : 0.f;
  }

  for (; base < op.n_items; base += stride) {
    const int item = base + rg;
    float a0 = 0.f, a1 = 0.f;
    if (item < op.n_items) {
#pragma unroll
      for (int i = 0; i < MAXV; ++i) {
        a0 = dotv(w0[i], xr[i], a0, T());
        a1 = dotv(w1[i], xr[i], a1, T());
      }
      if (item + stride < op.n_items) load(item + stride);
    }
    a0 = warp_sum(a0);
    a1 = warp_sum(a1);
    if (KS > 1) {
      if (lane == 0) {
        red[warp][0] = a0;
        red[warp][1] = a1;
      }
      __syncthreads();
      if (ks == 0 && lane == 0) {
        a0 = 0.f;
        a1 = 0.f;
        for (int k = 0; k < KS; ++k) {
          a0 += red[warp + k][0];
          a1 += red[warp + k][1];
        }
      }
    }
    if (ks == 0 && lane == 0 && item < op.n_items) op.epilogue(item, a0, a1);
    if (KS > 1) __syncthreads();
  }
  op.finish(smem);
}

// dynamic shared memory of a GEMV: the input vector and (norm prologues) the gains
static size_t gemv_smem_bytes(int K) { return (size_t)2 * K * sizeof(float); }

// ---- launch helpers ------------------------------------------------------------------

template <typename... KArgs, typename... Args>
static cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

// Choose the K split and the register tile (vectors per lane) of a GEMV, and a grid that
// is resident at once (each warp then loops over its items).
struct GemvPlan {
  int KS, MAXV, grid;
};
static int maxv_for(int nvec, int KS) {
  const int need = (((nvec + KS - 1) / KS) + 31) / 32;
  return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : need <= 6 ? 6 : need <= 8 ? 8 : 99;
}

template <typename T, class Op>
static void* gemv_fn(int maxv) {
  switch (maxv) {
    case 1: return (void*)gemv_kernel<T, 1, Op>;
    case 2: return (void*)gemv_kernel<T, 2, Op>;
    case 4: return (void*)gemv_kernel<T, 4, Op>;
    case 6: return (void*)gemv_kernel<T, 6, Op>;
    default: return (void*)gemv_kernel<T, 8, Op>;
  }
}

template <typename T, class Op>
static GemvPlan plan_gemv(int K, int n_items, int nsm) {
  const int nvec = K / Vec<T>::N;
  const size_t smem = gemv_smem_bytes(K);
  int KS = 1;
  while (KS < GEMV_WARPS && maxv_for(nvec, KS) > 8) KS *= 2;
  auto resident = [&](int ks) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_fn<T, Op>(maxv_for(nvec, ks)),
                                                  GEMV_WARPS * 32, smem);
    return (per_sm < 1 ? 1 : per_sm) * nsm;
  };
  // split K further while there are too few items to give every resident CTA one
  while (KS < GEMV_WARPS && (n_items + GEMV_WARPS / KS - 1) / (GEMV_WARPS / KS) < resident(KS)) KS *= 2;
  const int RG = GEMV_WARPS / KS;
  int grid = (n_items + RG - 1) / RG;
  const int cap = resident(KS);
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return {KS, maxv_for(nvec, KS), grid};
}

template <typename T, class Op>
static cudaError_t run_gemv(const Op& op, int nsm, cudaStream_t s, bool pdl) {
  const GemvPlan p = plan_gemv<T, Op>(op.K, op.n_items, nsm);
  if (p.MAXV > 8) return cudaErrorInvalidValue;
  const size_t smem = gemv_smem_bytes(op.K);
  const dim3 g(p.grid), b(GEMV_WARPS * 32);
  switch (p.MAXV) {
    case 1: return launch_k(gemv_kernel<T, 1, Op>, g, b, smem, s, pdl, op, p.KS);
    case 2: return launch_k(gemv_kernel<T, 2, Op>, g, b, smem, s, pdl, op, p.KS);
    case 4: return launch_k(gemv_kernel<T, 4, Op>, g, b, smem, s, pdl, op, p.KS);
    case 6: return launch_k(gemv_kernel<T, 6, Op>, g, b, smem, s, pdl, op, p.KS);
    default: return launch_k(gemv_kernel<T, 8, Op>, g, b, smem, s, pdl, op, p.KS);
  }
}

template <typename T, class Op>
static cudaError_t set_gemv_smem(int K) {
  const int bytes = (int)gemv_smem_bytes(K);
  if (bytes <= 48 * 1024) return cudaSuccess;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<T, 1, Op>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<T, 2, Op>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<T, 4, Op>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<T, 6, Op>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  return cudaFuncSetAttribute(gemv_kernel<T, 8, Op>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// ---- embedding ---------------------------------------------------------------------------

template <typename T>
__global__ void embed_kernel(const T* E, int V, int H, const int* tok, float* x, int* err) {
  constexpr int VN = Vec<T>::N;
  pdl_wait();
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
}

// ---- decode attention ------------------------------------------------------------------

template <typename T>
struct AttnArgs {
  const float* q;
  const T *k, *v;  // [nkv][stride][hd]
  int stride, hd, group, nsplit_max, chunk_min, ctx_host;
  const int* d_pos;
  float scale;
  float* out;
  float* part;            // [nq][nsplit_max][hd + 2]
  unsigned int* counter;  // [nkv]
};

// One CTA per (KV head, context chunk). The CTA copies q of its g query heads and the K and
// V rows of its chunk into shared memory with one batch of 16-byte loads, scores the chunk
// for all g heads (each K row read once for g heads), and keeps (max, sum of exp,
// unnormalised output) per head. The last CTA of the KV head to finish merges the chunks
// in chunk order (deterministic log-sum-exp combine).
constexpr int ATTN_THREADS = 256;
constexpr int COPY_BATCH = 8;

template <typename KV>
__global__ void __launch_bounds__(ATTN_THREADS) attn_decode_kernel(const AttnArgs<KV> a) {
  extern __shared__ __align__(16) float sm[];
  __shared__ bool s_last;
  const int g = blockIdx.x, split = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int G = a.group, hd = a.hd;
  pdl_wait();
  pdl_trigger();
  const int ctx = a.d_pos ? __ldcg(a.d_pos) + 1 : a.ctx_host;
  const int chunk = max(a.chunk_min, (ctx + a.nsplit_max - 1) / a.nsplit_max);
  const int nsplit = (ctx + chunk - 1) / chunk;
  if (split >= nsplit) return;
  const int j0 = split * chunk, j1 = min(ctx, j0 + chunk), n = j1 - j0;
  // shared layout: q [G][hd] f32 | scores [G][chunk] f32 | stats [G][2] | weights [G][nsplit_max]
  //                | K [chunk][hd] KV | V [chunk][hd] KV
  float* qs = sm;
  float* sc = qs + G * hd;
  float* st = sc + G * chunk;
  float* wts = st + 2 * G;
  const int kv_off = (G * hd + G * chunk + 2 * G + G * a.nsplit_max + 3) & ~3;  // 16-byte aligned
  KV* ks = reinterpret_cast<KV*>(sm + kv_off);
  KV* vs = ks + (size_t)chunk * hd;
  {
    const int qv = G * hd / 4;                               // 16-byte vectors of q
    const int kvv = n * hd * (int)sizeof(KV) / 16;           // of the K (and the V) rows
    const int total = qv + 2 * kvv;
    const uint4* qsrc = reinterpret_cast<const uint4*>(a.q + (size_t)g * G * hd);
    const uint4* ksrc = reinterpret_cast<const uint4*>(a.k + ((size_t)g * a.stride + j0) * hd);
    const uint4* vsrc = reinterpret_cast<const uint4*>(a.v + ((size_t)g * a.stride + j0) * hd);
    uint4* qdst = reinterpret_cast<uint4*>(qs);
    uint4* kdst = reinterpret_cast<uint4*>(ks);
    uint4* vdst = reinterpret_cast<uint4*>(vs);
    for (int base = tid; base < total; base += COPY_BATCH * blockDim.x) {
      uint4 r[COPY_BATCH];
#pragma unroll
      for (int i = 0; i < COPY_BATCH; ++i) {
        const int j = base + i * blockDim.x;
        if (j < qv) r[i] = __ldcg(qsrc + j);
        else if (j < qv + kvv) r[i] = __ldcg(ksrc + (j - qv));
        else if (j < total) r[i] = __ldcg(vsrc + (j - qv - kvv));
      }
#pragma unroll
      for (int i = 0; i < COPY_BATCH; ++i) {
        const int j = base + i * blockDim.x;
        if (j < qv) qdst[j] = r[i];
        else if (j < qv + kvv) kdst[j - qv] = r[i];
        else if (j < total) vdst[j - qv - kvv] = r[i];
      }
    }
  }
  __syncthreads();
  // scores: a warp per position, lanes over the head dimension
  for (int jj = warp; jj < n; jj += nwarps) {
    float part[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) part[h] = 0.f;
    for (int dd = lane; dd < hd; dd += 32) {
      const float kv = to_f32(ks[jj * hd + dd]);
#pragma unroll
      for (int h = 0; h < GMAX; ++h)
        if (h < G) part[h] = fmaf(qs[h * hd + dd], kv, part[h]);
    }
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      if (h < G) {
        const float sv = warp_sum(part[h]);
        if (lane == 0) sc[h * chunk + jj] = sv * a.scale;
      }
    }
  }
  __syncthreads();
  for (int h = warp; h < G; h += nwarps) {
    float m = -INFINITY;
    for (int jj = lane; jj < n; jj += 32) m = fmaxf(m, sc[h * chunk + jj]);
    m = warp_max(m);
    float l = 0.f;
    for (int jj = lane; jj < n; jj += 32) {
      const float p = expf(sc[h * chunk + jj] - m);
      sc[h * chunk + jj] = p;
      l += p;
    }
    l = warp_sum(l);
    if (lane == 0) {
      st[2 * h] = m;
      st[2 * h + 1] = l;
    }
  }
  __syncthreads();
  const int pstride = hd + 2;
  for (int idx = tid; idx < G * hd; idx += blockDim.x) {
    const int h = idx / hd, dd = idx - h * hd;
    float acc = 0.f;
    for (int jj = 0; jj < n; ++jj) acc = fmaf(sc[h * chunk + jj], to_f32(vs[jj * hd + dd]), acc);
    a.part[((size_t)(g * G + h) * a.nsplit_max + split) * pstride + dd] = acc;
  }
  if (tid < G) {
    float* p = a.part + ((size_t)(g * G + tid) * a.nsplit_max + split) * pstride;
    p[hd] = st[2 * tid];
    p[hd + 1] = st[2 * tid + 1];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.counter + g, 1u) == (unsigned)(nsplit - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // merge: weights w_s = exp(m_s - M) / sum_s l_s exp(m_s - M) per head, then out = sum_s w_s O_s
  for (int i = tid; i < G * nsplit; i += blockDim.x) {
    const int h = i / nsplit, sp = i - h * nsplit;
    const float* p = a.part + ((size_t)(g * G + h) * a.nsplit_max + sp) * pstride + hd;
    wts[h * a.nsplit_max + sp] = __ldcg(p);  // m_s
  }
  __syncthreads();
  for (int h = warp; h < G; h += nwarps) {
    float M = -INFINITY;
    for (int sp = lane; sp < nsplit; sp += 32) M = fmaxf(M, wts[h * a.nsplit_max + sp]);
    M = warp_max(M);
    float L = 0.f;
    for (int sp = lane; sp < nsplit; sp += 32) {
      const float* p = a.part + ((size_t)(g * G + h) * a.nsplit_max + sp) * pstride + hd;
      const float w = expf(wts[h * a.nsplit_max + sp] - M);
      wts[h * a.nsplit_max + sp] = w;
      L = fmaf(__ldcg(p + 1), w, L);
    }
    L = warp_sum(L);
    const float inv = 1.f / L;
    for (int sp = lane; sp < nsplit; sp += 32) wts[h * a.nsplit_max + sp] *= inv;
  }
  __syncthreads();
  constexpr int EPT = GMAX * 128 / ATTN_THREADS;  // output elements per thread (G*hd <= 1024)
  float acc[EPT];
#pragma unroll
  for (int k = 0; k < EPT; ++k) acc[k] = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += 4) {
    float v[EPT][4];
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const int idx = tid + k * blockDim.x;
      const int h = idx / hd, dd = idx - h * hd;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[k][u] = (idx < G * hd && s0 + u < nsplit)
                      ? __ldcg(a.part + ((size_t)(g * G + h) * a.nsplit_max + s0 + u) * pstride + dd)
                      : 0.f;
    }
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const int idx = tid + k * blockDim.x;
      const int h = idx / hd;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (idx < G * hd && s0 + u < nsplit) acc[k] = fmaf(v[k][u], wts[h * a.nsplit_max + s0 + u], acc[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < EPT; ++k) {
    const int idx = tid + k * blockDim.x;
    if (idx < G * hd) a.out[(size_t)g * G * hd + idx] = acc[k];
  }
  if (tid == 0) a.counter[g] = 0u;
}

// ---- host launchers ---------------------------------------------------------------------

size_t attn_workspace_bytes(int nq, int nkv, int hd, int nsplit) {
  size_t part = (size_t)nq * nsplit * (hd + 2) * sizeof(float);
  part = (part + 255) & ~(size_t)255;
  return part + (size_t)nkv * sizeof(unsigned int);
}

// Chunks of at least chunk_min positions and at most MAX_SPLITS chunks per KV head (short
// contexts spread over several CTAs, the merge stays short), unless the K and V rows of a
// chunk would exceed ~160 KB of shared memory; then the chunk count grows instead.
constexpr int MAX_SPLITS = 16;
int attn_nsplit_for(int cap, int chunk_min, int hd, int kv_bytes) {
  int chunk_max = (160 * 1024) / (2 * hd * kv_bytes);
  if (chunk_max > 256) chunk_max = 256;
  if (chunk_max < chunk_min) chunk_max = chunk_min;
  int n = (cap + chunk_min - 1) / chunk_min;
  if (n > MAX_SPLITS) n = MAX_SPLITS;
  const int need = (cap + chunk_max - 1) / chunk_max;
  if (n < need) n = need;
  return n < 1 ? 1 : n;
}

size_t attn_smem_bytes(int group, int hd, int cap, int nsplit, int chunk_min, int kv_bytes) {
  int chunk = (cap + nsplit - 1) / nsplit;
  if (chunk < chunk_min) chunk = chunk_min;
  const size_t f = ((size_t)group * hd + (size_t)group * chunk + 2 * group + (size_t)group * nsplit + 3) &
                   ~(size_t)3;
  return f * sizeof(float) + 2 * (size_t)chunk * hd * kv_bytes;
}

cudaError_t launch_attn(int kv_dtype, int nq, int nkv, int hd, int nsplit, int chunk_min,
                        size_t smem, const float* q, const void* kc, const void* vc,
                        int kv_stride, const int* d_pos, int ctx_host, float* out, void* ws,
                        cudaStream_t s, bool pdl) {
  const int G = nq / nkv;
  if (G > GMAX) return cudaErrorInvalidValue;
  size_t part_bytes = ((size_t)nq * nsplit * (hd + 2) * sizeof(float) + 255) & ~(size_t)255;
  const dim3 grid(nkv, nsplit), block(ATTN_THREADS);
  if (kv_dtype == 2) {
    AttnArgs<f16> a{q, (const f16*)kc, (const f16*)vc, kv_stride, hd, G, nsplit, chunk_min,
                     ctx_host, d_pos, 1.f / sqrtf((float)hd), out, (float*)ws,
                     (unsigned int*)((char*)ws + part_bytes)};
    return launch_k(attn_decode_kernel<f16>, grid, block, smem, s, pdl, a);
  }
  AttnArgs<float> a{q, (const float*)kc, (const float*)vc, kv_stride, hd, G, nsplit, chunk_min,
                    ctx_host, d_pos, 1.f / sqrtf((float)hd), out, (float*)ws,
                    (unsigned int*)((char*)ws + part_bytes)};
  return launch_k(attn_decode_kernel<float>, grid, block, smem, s, pdl, a);
}

cudaError_t attn_set_attributes(size_t smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<f16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e) return e;
  return cudaFuncSetAttribute(attn_decode_kernel<float>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <typename T>
static cudaError_t set_attrs_t(const Dims& d) {
  cudaError_t e;
  if ((e = set_gemv_smem<T, OpQKV<T, float>>(d.H))) return e;
  if ((e = set_gemv_smem<T, OpQKV<T, f16>>(d.H))) return e;
  if ((e = set_gemv_smem<T, OpGateUp<T>>(d.H))) return e;
  if ((e = set_gemv_smem<T, OpResid<T>>(d.I > d.nq * d.hd ? d.I : d.nq * d.hd))) return e;
  return set_gemv_smem<T, OpLMHead<T>>(d.H);
}

cudaError_t decode_set_attributes(const Dims& d) {
  return d.dtype == 1 ? set_attrs_t<bf16>(d) : set_attrs_t<float>(d);
}

cudaError_t launch_embed(const Dims& d, const void* E, const int* tok, float* x, int* err,
                         cudaStream_t s, bool pdl) {
  if (d.dtype == 1)
    return launch_k(embed_kernel<bf16>, dim3(1), dim3(256), 0, s, pdl, (const bf16*)E, d.V, d.H, tok, x, err);
  return launch_k(embed_kernel<float>, dim3(1), dim3(256), 0, s, pdl, (const float*)E, d.V, d.H, tok, x, err);
}

template <typename T, typename KV>
static cudaError_t qkv_t(const Dims& d, const LayerPtrs& w, const float* x, const int* d_pos,
                         const float2* rope, float* q, void* kc, void* vc, cudaStream_t s, bool pdl) {
  OpQKV<T, KV> op{};
  op.K = d.H;
  op.n_items = (d.nq + 2 * d.nkv) * (d.hd / 2);
  op.hd = d.hd; op.nq = d.nq; op.nkv = d.nkv; op.cap = d.cap;
  op.wq = (const T*)w.wq; op.wk = (const T*)w.wk; op.wv = (const T*)w.wv;
  op.bq = (const T*)w.bq; op.bk = (const T*)w.bk; op.bv = (const T*)w.bv;
  op.gain = (const T*)w.in_norm;
  op.x = x; op.eps = d.eps; op.d_pos = d_pos; op.rope = rope; op.q_out = q;
  op.kc = (KV*)kc; op.vc = (KV*)vc;
  return run_gemv<T>(op, d.nsm, s, pdl);
}
cudaError_t launch_qkv(const Dims& d, const LayerPtrs& w, const float* x, const int* d_pos,
                       const float2* rope, float* q, void* kc, void* vc, cudaStream_t s, bool pdl) {
  return d.dtype == 1 ? qkv_t<bf16, f16>(d, w, x, d_pos, rope, q, kc, vc, s, pdl)
                      : qkv_t<float, float>(d, w, x, d_pos, rope, q, kc, vc, s, pdl);
}

template <typename T>
static cudaError_t resid_t(const Dims& d, const void* W, int N, int K, const float* in, float* y,
                           cudaStream_t s, bool pdl) {
  OpResid<T> op{};
  op.K = K; op.N = N; op.n_items = (N + 1) / 2; op.W = (const T*)W; op.in = in; op.y = y;
  return run_gemv<T>(op, d.nsm, s, pdl);
}
cudaError_t launch_resid(const Dims& d, const void* W, int N, int K, const float* in, float* y,
                         cudaStream_t s, bool pdl) {
  return d.dtype == 1 ? resid_t<bf16>(d, W, N, K, in, y, s, pdl)
                      : resid_t<float>(d, W, N, K, in, y, s, pdl);
}

template <typename T>
static cudaError_t gateup_t(const Dims& d, const LayerPtrs& w, const float* x, float* act,
                            cudaStream_t s, bool pdl) {
  OpGateUp<T> op{};
  op.K = d.H; op.n_items = d.I; op.wg = (const T*)w.w_gate; op.wu = (const T*)w.w_up;
  op.gain = (const T*)w.post_norm; op.x = x; op.eps = d.eps; op.act = act;
  return run_gemv<T>(op, d.nsm, s, pdl);
}
cudaError_t launch_gateup(const Dims& d, const LayerPtrs& w, const float* x, float* act,
                          cudaStream_t s, bool pdl) {
  return d.dtype == 1 ? gateup_t<bf16>(d, w, x, act, s, pdl) : gateup_t<float>(d, w, x, act, s, pdl);
}

template <typename T>
static cudaError_t lmhead_t(const Dims& d, const void* W, const void* fn, const float* x,
                            float* logits, const Finalize& f, cudaStream_t s, bool pdl) {
  OpLMHead<T> op{};
  op.K = d.H; op.N = d.V; op.n_items = (d.V + 1) / 2; op.W = (const T*)W; op.gain = (const T*)fn;
  op.x = x; op.eps = d.eps; op.logits = logits; op.f = f;
  return run_gemv<T>(op, d.nsm, s, pdl);
}
cudaError_t launch_lmhead(const Dims& d, const void* W, const void* final_norm, const float* x,
                          float* logits, const Finalize& f, cudaStream_t s, bool pdl) {
  return d.dtype == 1 ? lmhead_t<bf16>(d, W, final_norm, x, logits, f, s, pdl)
                      : lmhead_t<float>(d, W, final_norm, x, logits, f, s, pdl);
}

}  // namespace qw
