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

// xs = x / sqrt(mean(x^2) + eps) * gain
template <typename T>
__device__ __forceinline__ void prologue_norm(float* xs, float* scratch, const float* x,
                                              const T* gain, int K, float eps) {
  float ss = 0.f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    float v = __ldcg(x + k);
    xs[k] = v;
    ss = fmaf(v, v, ss);
  }
  ss = block_sum(ss, scratch);
  const float inv = rsqrtf(ss / (float)K + eps);
  for (int k = threadIdx.x; k < K; k += blockDim.x) xs[k] = xs[k] * inv * to_f32(gain[k]);
}

__device__ __forceinline__ void prologue_copy(float* xs, const float* x, int K) {
  for (int k = threadIdx.x; k < K; k += blockDim.x) xs[k] = __ldcg(x + k);
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

  __device__ void prologue(float* xs, float* scratch) {
    prologue_norm(xs, scratch, x, gain, K, eps);
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
  __device__ void prologue(float* xs, float* scratch) { prologue_norm(xs, scratch, x, gain, K, eps); }
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
  __device__ void prologue(float* xs, float*) { prologue_copy(xs, in, K); }
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
  __device__ void prologue(float* xs, float* scratch) {
    prologue_norm(xs, scratch, x, gain, K, eps);
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
  op.prologue(smem, scratch);
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

// Choose the K split and the register tile (vectors per lane) of a GEMV.
struct GemvPlan {
  int KS, MAXV, grid;
};
static GemvPlan plan_gemv(int K, int vec, int n_items, int nsm) {
  const int nvec = K / vec;
  int KS = 1;
  while (KS < GEMV_WARPS && (((nvec + KS - 1) / KS) + 31) / 32 > 8) KS *= 2;
  // spread small matrices over all SMs
  while (KS < GEMV_WARPS && (n_items + GEMV_WARPS / KS - 1) / (GEMV_WARPS / KS) < 2 * nsm) KS *= 2;
  const int need = (((nvec + KS - 1) / KS) + 31) / 32;
  int MAXV = need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : need <= 6 ? 6 : 8;
  const int RG = GEMV_WARPS / KS;
  int grid = (n_items + RG - 1) / RG;
  const int cap = nsm * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return {KS, MAXV, grid};
}

template <typename T, class Op>
static cudaError_t run_gemv(const Op& op, int nsm, cudaStream_t s, bool pdl) {
  const GemvPlan p = plan_gemv(op.K, Vec<T>::N, op.n_items, nsm);
  if (p.MAXV > 8) return cudaErrorInvalidValue;
  const size_t smem = (size_t)op.K * sizeof(float);
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
  const int bytes = K * (int)sizeof(float);
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
  pdl_wait();
  int t = __ldcg(tok);
  if (t < 0 || t >= V) {
    if (threadIdx.x == 0) atomicOr(err, ERR_TOKEN);
    t = 0;
  }
  const T* row = E + (size_t)t * H;
  for (int k = threadIdx.x; k < H; k += blockDim.x) x[k] = to_f32(row[k]);
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

// One CTA per (KV head, context chunk). The CTA scores its chunk for all query heads of
// the KV head, keeps (max, sum of exp, unnormalised output) per head, and the last CTA of
// the KV head to finish merges the chunks in chunk order (deterministic).
template <typename T>
__global__ void __launch_bounds__(128) attn_decode_kernel(const AttnArgs<T> a) {
  extern __shared__ float sm[];
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
  float* qs = sm;                 // [G][hd]
  float* sc = sm + G * hd;        // [G][chunk]
  float* st = sc + G * chunk;     // [G][2]
  for (int i = tid; i < G * hd; i += blockDim.x) qs[i] = __ldcg(a.q + (size_t)g * G * hd + i) * a.scale;
  __syncthreads();
  const T* K = a.k + (size_t)g * a.stride * hd;
  const T* V = a.v + (size_t)g * a.stride * hd;
  for (int j = j0 + warp; j < j1; j += nwarps) {
    float part[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) part[h] = 0.f;
    for (int dd = lane; dd < hd; dd += 32) {
      const float kv = to_f32(K[(size_t)j * hd + dd]);
#pragma unroll
      for (int h = 0; h < GMAX; ++h)
        if (h < G) part[h] = fmaf(qs[h * hd + dd], kv, part[h]);
    }
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      if (h < G) {
        const float s = warp_sum(part[h]);
        if (lane == 0) sc[h * chunk + (j - j0)] = s;
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
  for (int dd = tid; dd < hd; dd += blockDim.x) {
    float acc[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) acc[h] = 0.f;
    for (int jj = 0; jj < n; ++jj) {
      const float vv = to_f32(V[(size_t)(j0 + jj) * hd + dd]);
#pragma unroll
      for (int h = 0; h < GMAX; ++h)
        if (h < G) acc[h] = fmaf(sc[h * chunk + jj], vv, acc[h]);
    }
#pragma unroll
    for (int h = 0; h < GMAX; ++h)
      if (h < G) a.part[((size_t)(g * G + h) * a.nsplit_max + split) * pstride + dd] = acc[h];
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
  for (int idx = tid; idx < G * hd; idx += blockDim.x) {
    const int h = idx / hd, dd = idx - h * hd;
    const float* p = a.part + (size_t)(g * G + h) * a.nsplit_max * pstride;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldcg(p + s * pstride + hd));
    float L = 0.f, o = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float w = expf(__ldcg(p + s * pstride + hd) - M);
      L = fmaf(__ldcg(p + s * pstride + hd + 1), w, L);
      o = fmaf(__ldcg(p + s * pstride + dd), w, o);
    }
    a.out[(size_t)(g * G + h) * hd + dd] = o / L;
  }
  if (tid == 0) a.counter[g] = 0u;
}

// ---- host launchers ---------------------------------------------------------------------

size_t attn_workspace_bytes(int nq, int nkv, int hd, int nsplit) {
  size_t part = (size_t)nq * nsplit * (hd + 2) * sizeof(float);
  part = (part + 255) & ~(size_t)255;
  return part + (size_t)nkv * sizeof(unsigned int);
}

int attn_nsplit_for(int nsm, int nkv, int cap, int chunk_min) {
  int by_ctx = (cap + chunk_min - 1) / chunk_min;
  int by_sm = (2 * nsm + nkv - 1) / nkv;
  int n = by_ctx < by_sm ? by_ctx : by_sm;
  return n < 1 ? 1 : n;
}

size_t attn_smem_bytes(int group, int hd, int cap, int nsplit, int chunk_min) {
  int chunk = (cap + nsplit - 1) / nsplit;
  if (chunk < chunk_min) chunk = chunk_min;
  return ((size_t)group * hd + (size_t)group * chunk + 2 * group) * sizeof(float);
}

cudaError_t launch_attn(int kv_dtype, int nq, int nkv, int hd, int nsplit, int chunk_min,
                        size_t smem, const float* q, const void* kc, const void* vc,
                        int kv_stride, const int* d_pos, int ctx_host, float* out, void* ws,
                        cudaStream_t s, bool pdl) {
  const int G = nq / nkv;
  if (G > GMAX) return cudaErrorInvalidValue;
  size_t part_bytes = ((size_t)nq * nsplit * (hd + 2) * sizeof(float) + 255) & ~(size_t)255;
  const dim3 grid(nkv, nsplit), block(128);
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
