// Prefill of T prompt tokens of one sequence ("augur", Features: prefill/decode split;
// "LLM Speedrun: Architecture", Transformer architecture / Implementing Qwen).
//
// Row-major activations [T][features] in fp32. Per layer:
//   norm rows -> Q/K/V GEMMs (+bias) -> RoPE + KV-cache write -> causal GQA attention ->
//   o_proj GEMM (+= residual) -> norm rows -> gate/up GEMMs -> SwiGLU -> down GEMM (+=).
// This translation unit holds the CUDA-core (SIMT) versions (exact fp32 arithmetic on any
// shape: the fp32 models and the general path), the row kernels, the mma.sync attention,
// and prefill_tc, the bf16 models' chain on the tensor cores: RMSNorm -> one q|k|v GEMM with
// bias, RoPE and the KV append in its epilogue -> tcgen05 attention -> o_proj GEMM
// (+= residual) -> RMSNorm -> gate/up GEMM with SwiGLU in its epilogue -> down GEMM (+=),
// every kernel after the embedding launched with programmatic dependent launch.
#include "common.cuh"
#include "internal.h"

#include <math.h>
#include <stdlib.h>
#include <cstring>

namespace qw {

// ---- row kernels -------------------------------------------------------------------------

template <typename T>
__global__ void embed_rows_kernel(const T* E, int V, int H, const int* ids, float* X, int* err) {
  const int t = blockIdx.x;
  int id = ids[t];
  if (id < 0 || id >= V) {
    if (threadIdx.x == 0) atomicOr(err, ERR_TOKEN);
    id = 0;
  }
  const T* row = E + (size_t)id * H;
  for (int k = threadIdx.x; k < H; k += blockDim.x) X[(size_t)t * H + k] = to_f32(row[k]);
}

__device__ __forceinline__ void store_norm(float* y, float v, int*) { *y = v; }
__device__ __forceinline__ void store_norm(f16* y, float v, int* err) { *y = to_half_checked(v, err); }

template <typename T, typename OutT>
__global__ void norm_rows_kernel(const float* X, const T* gain, int H, float eps, OutT* Y, int* err) {
  __shared__ float scratch[32];
  const float* x = X + (size_t)blockIdx.x * H;
  float ss = 0.f;
  for (int k = threadIdx.x; k < H; k += blockDim.x) ss = fmaf(x[k], x[k], ss);
  ss = block_sum(ss, scratch);
  const float inv = rsqrtf(ss / (float)H + eps);
  OutT* y = Y + (size_t)blockIdx.x * H;
  for (int k = threadIdx.x; k < H; k += blockDim.x) store_norm(y + k, x[k] * inv * to_f32(gain[k]), err);
}

// The same for fp16 output rows with H a multiple of 128: one warp per row, float4 loads
// and 8-byte stores. The row is read twice (sum of squares, then the scaled values); the
// second read comes from L2. Sums in a fixed order: deterministic.
// Warp per row, the row held in registers (MAXV float4 per lane: H <= 128 MAXV), one read
// of X; fp16 range errors gathered per lane and raised once.
template <int MAXV>
__global__ void norm_rows_h_kernel(const float* X, const bf16* gain, int T, int H, float eps, f16* Y, int* err) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= T) return;
  const int nv = H >> 7;  // float4 per lane
  const float4* x = reinterpret_cast<const float4*>(X + (size_t)row * H);
  float4 v[MAXV];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    v[j] = j < nv ? __ldcg(x + lane + 32 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
    ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)H + eps);
  const uint2* gp = reinterpret_cast<const uint2*>(gain);
  uint2* y = reinterpret_cast<uint2*>(Y + (size_t)row * H);
  bool bad = false;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    if (j < nv) {
      const int k = lane + 32 * j;
      const uint2 gb = __ldg(gp + k);
      const float a = v[j].x * inv * __uint_as_float(gb.x << 16), b = v[j].y * inv * __uint_as_float(gb.x & 0xffff0000u);
      const float c = v[j].z * inv * __uint_as_float(gb.y << 16), d = v[j].w * inv * __uint_as_float(gb.y & 0xffff0000u);
      bad |= !(fabsf(a) < 65520.f) || !(fabsf(b) < 65520.f) || !(fabsf(c) < 65520.f) || !(fabsf(d) < 65520.f);  // NaN too
      const __half2 lo = __floats2half2_rn(a, b), hi = __floats2half2_rn(c, d);
      y[k] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
  }
  if (bad) atomicOr(err, ERR_RANGE);
}

// Short prompts: one 128-thread block per row (float4 loads, 8-byte stores), so that every
// SM has rows.
__global__ void __launch_bounds__(128) norm_row_block_h_kernel(const float* X, const bf16* gain, int H, float eps,
                                                               f16* Y, int* err) {
  pdl_trigger();
  pdl_wait();
  __shared__ float scratch[32];
  const int row = blockIdx.x;
  const float4* x = reinterpret_cast<const float4*>(X + (size_t)row * H);
  const uint2* gp = reinterpret_cast<const uint2*>(gain);
  uint2* y = reinterpret_cast<uint2*>(Y + (size_t)row * H);
  constexpr int MAXV = 8;  // float4 per thread: H <= 4096
  float4 v[MAXV];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int k = threadIdx.x + 128 * j;
    v[j] = k < H / 4 ? x[k] : make_float4(0.f, 0.f, 0.f, 0.f);
    ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
  }
  ss = block_sum(ss, scratch);
  const float inv = rsqrtf(ss / (float)H + eps);
  bool bad = false;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int k = threadIdx.x + 128 * j;
    if (k < H / 4) {
      const uint2 gb = __ldg(gp + k);
      const float a = v[j].x * inv * __uint_as_float(gb.x << 16), b = v[j].y * inv * __uint_as_float(gb.x & 0xffff0000u);
      const float c = v[j].z * inv * __uint_as_float(gb.y << 16), d = v[j].w * inv * __uint_as_float(gb.y & 0xffff0000u);
      bad |= !(fabsf(a) < 65520.f) || !(fabsf(b) < 65520.f) || !(fabsf(c) < 65520.f) || !(fabsf(d) < 65520.f);  // NaN too
      const __half2 lo = __floats2half2_rn(a, b), hi = __floats2half2_rn(c, d);
      y[k] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
  }
  if (bad) atomicOr(err, ERR_RANGE);
}

static void norm_rows_h(const float* X, const bf16* gain, int T_, int H, float eps, f16* Y, int* err, cudaStream_t s,
                        int nsm) {
  const bool vec = H % 128 == 0 && ((uintptr_t)gain & 7) == 0;
  // programmatic dependent launch (the kernels wait for the previous grid before reading X)
  const bool pdl = tc_pdl();
  if (vec && T_ < 4 * nsm && H <= 4096) {
    launch_k(norm_row_block_h_kernel, dim3(T_), dim3(128), 0, s, pdl, X, gain, H, eps, Y, err);
  } else if (vec && H <= 128 * 12) {
    launch_k(norm_rows_h_kernel<12>, dim3((T_ + 7) / 8), dim3(256), 0, s, pdl, X, gain, T_, H, eps, Y, err);
  } else if (vec && H <= 128 * 32) {
    launch_k(norm_rows_h_kernel<32>, dim3((T_ + 7) / 8), dim3(256), 0, s, pdl, X, gain, T_, H, eps, Y, err);
  } else {
    norm_rows_kernel<bf16, f16><<<T_, 256, 0, s>>>(X, gain, H, eps, Y, err);
  }
}

// fp32 -> fp16 rows (tensor-core A operand)
__global__ void to_half_kernel(const float* X, f16* Y, size_t n, int* err) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    Y[i] = to_half_checked(X[i], err);
}

__global__ void swiglu_kernel(const float* G, const float* U, float* A, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float g = G[i];
    A[i] = (g / (1.f + expf(-g))) * U[i];
  }
}

// Y [T][nq*hd + 2*nkv*hd] (q | k | v, bias included; with pairs, each head's columns in
// RoPE-pair order) -> Q [T][nq*hd] rotated (fp32); K, V rotated/copied into the cache at
// positions pos0 + t.
template <typename KV>
__global__ void rope_kv_kernel(const float* Y, int T_, int nq, int nkv, int hd, int pos0, int cap,
                               const float2* rope, float* Q, KV* kc, KV* vc, int* err, bool pairs = false) {
  const int t = blockIdx.x;
  const int half = hd / 2;
  const int width = (nq + 2 * nkv) * hd;
  const int pos = pos0 + t;
  const float* y = Y + (size_t)t * width;
  for (int idx = threadIdx.x; idx < (nq + 2 * nkv) * half; idx += blockDim.x) {
    const int head = idx / half, i = idx - head * half;
    // pairs: Y's head columns in pair order (2i, 2i + 1), else split-half (i, i + hd/2)
    const float a = pairs ? y[head * hd + 2 * i] : y[head * hd + i];
    const float b = pairs ? y[head * hd + 2 * i + 1] : y[head * hd + i + half];
    if (head < nq + nkv) {
      const float2 cs = rope[(size_t)pos * half + i];
      const float ra = a * cs.x - b * cs.y, rb = b * cs.x + a * cs.y;
      if (head < nq) {
        const size_t o = (size_t)t * nq * hd + head * hd + i;
        Q[o] = ra;
        Q[o + half] = rb;
      } else {
        KV* dst = kc + ((size_t)(head - nq) * cap + pos) * hd;
        store_kv(dst + i, ra, err);
        store_kv(dst + i + half, rb, err);
      }
    } else {
      KV* dst = vc + ((size_t)(head - nq - nkv) * cap + pos) * hd;
      store_kv(dst + i, a, err);
      store_kv(dst + i + half, b, err);
    }
  }
}

// ---- SIMT GEMM: C[M,N] (=|+=) A[M,K] . B[N,K]^T (+ bias) ---------------------------------

constexpr int GB_M = 64, GB_N = 64, GB_K = 16;

template <typename T, bool ACCUM>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const float* A, int lda, const T* B, int ldb, const T* bias, float* C, int ldc,
                 int M, int N, int K) {
  __shared__ float As[GB_K][GB_M + 4];
  __shared__ float Bs[GB_K][GB_N + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * GB_M, n0 = blockIdx.x * GB_N;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += GB_K) {
    for (int i = threadIdx.x; i < GB_M * GB_K; i += 256) {
      const int r = i / GB_K, c = i - r * GB_K;
      const int gm = m0 + r, gk = k0 + c;
      As[c][r] = (gm < M && gk < K) ? A[(size_t)gm * lda + gk] : 0.f;
      const int gn = n0 + r;
      Bs[c][r] = (gn < N && gk < K) ? to_f32(B[(size_t)gn * ldb + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < GB_K; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty + 16 * i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx + 16 * j;
      if (gn >= N) continue;
      float v = acc[i][j];
      if (bias) v += to_f32(bias[gn]);
      float* c = C + (size_t)gm * ldc + gn;
      *c = ACCUM ? *c + v : v;
    }
  }
}

template <typename T>
static void gemm_simt(const float* A, int lda, const void* B, int ldb, const void* bias, float* C,
                      int ldc, int M, int N, int K, bool accum, cudaStream_t s) {
  dim3 grid((N + GB_N - 1) / GB_N, (M + GB_M - 1) / GB_M), block(256);
  if (accum)
    gemm_simt_kernel<T, true><<<grid, block, 0, s>>>(A, lda, (const T*)B, ldb, (const T*)bias, C, ldc, M, N, K);
  else
    gemm_simt_kernel<T, false><<<grid, block, 0, s>>>(A, lda, (const T*)B, ldb, (const T*)bias, C, ldc, M, N, K);
}

// ---- causal GQA flash attention (SIMT) -----------------------------------------------------
//
// One CTA per (block of 64 queries, query head). Keys and values of the head's KV group
// stream through shared memory in blocks of 64 positions; scores, the running max and
// the running sum follow the online-softmax recurrence, so each query row ends with
// exactly softmax(q K^T / sqrt(d)) V over keys at positions <= its own.
constexpr int FA_BQ = 64, FA_BK = 64;

template <typename T, int HD>
__global__ void __launch_bounds__(256)
attn_prefill_simt_kernel(const float* Q, int T_, int nq, int nkv, int pos0, const T* kc,
                         const T* vc, int cap, float scale, float* O) {  // T: KV element type
  extern __shared__ float fsm[];
  float* qs = fsm;                       // [BQ][HD+1]
  float* ks = qs + FA_BQ * (HD + 1);     // [BK][HD+1]
  float* vs = ks + FA_BK * (HD + 1);     // [BK][HD]
  float* ps = vs + FA_BK * HD;           // [BQ][BK+1]
  const int qb = blockIdx.x, h = blockIdx.y, g = h / (nq / nkv);
  const int tid = threadIdx.x;
  const int r = tid >> 2, c = tid & 3;   // row r of the query block; quarter c
  const int q0 = qb * FA_BQ;
  const int nrows = min(FA_BQ, T_ - q0);
  for (int i = tid; i < FA_BQ * HD; i += 256) {
    const int rr = i / HD, dd = i - rr * HD;
    qs[rr * (HD + 1) + dd] = rr < nrows ? Q[(size_t)(q0 + rr) * nq * HD + h * HD + dd] * scale : 0.f;
  }
  const int my_pos = pos0 + q0 + r;
  const int last_pos = pos0 + q0 + nrows - 1;
  constexpr int DPT = HD / 4;  // output dims per thread
  float o[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) o[i] = 0.f;
  float m = -INFINITY, l = 0.f;
  const T* K = kc + (size_t)g * cap * HD;
  const T* V = vc + (size_t)g * cap * HD;
  for (int k0 = 0; k0 <= last_pos; k0 += FA_BK) {
    const int nk = min(FA_BK, last_pos + 1 - k0);
    __syncthreads();
    for (int i = tid; i < FA_BK * HD; i += 256) {
      const int jj = i / HD, dd = i - jj * HD;
      const bool ok = jj < nk;
      ks[jj * (HD + 1) + dd] = ok ? to_f32(K[(size_t)(k0 + jj) * HD + dd]) : 0.f;
      vs[jj * HD + dd] = ok ? to_f32(V[(size_t)(k0 + jj) * HD + dd]) : 0.f;
    }
    __syncthreads();
    // scores of row r against keys c, c+4, ..., (16 per thread)
    float s[FA_BK / 4];
    float mloc = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < FA_BK / 4; ++jj) {
      const int j = c + 4 * jj;
      float acc = 0.f;
#pragma unroll 8
      for (int dd = 0; dd < HD; ++dd) acc = fmaf(qs[r * (HD + 1) + dd], ks[j * (HD + 1) + dd], acc);
      const bool open = (j < nk) && (k0 + j <= my_pos) && (r < nrows);
      s[jj] = open ? acc : -INFINITY;
      mloc = fmaxf(mloc, s[jj]);
    }
    mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
    mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
    const float mnew = fmaxf(m, mloc);
    const float corr = (mnew == -INFINITY) ? 1.f : expf(m - mnew);
    float lsum = 0.f;
#pragma unroll
    for (int jj = 0; jj < FA_BK / 4; ++jj) {
      const float p = (s[jj] == -INFINITY) ? 0.f : expf(s[jj] - mnew);
      ps[r * (FA_BK + 1) + c + 4 * jj] = p;
      lsum += p;
    }
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    l = l * corr + lsum;
    m = mnew;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < DPT; ++i) o[i] *= corr;
    for (int j = 0; j < nk; ++j) {
      const float p = ps[r * (FA_BK + 1) + j];
#pragma unroll
      for (int i = 0; i < DPT; ++i) o[i] = fmaf(p, vs[j * HD + c * DPT + i], o[i]);
    }
  }
  if (r < nrows) {
    const float inv = 1.f / l;
    float* out = O + (size_t)(q0 + r) * nq * HD + h * HD + c * DPT;
#pragma unroll
    for (int i = 0; i < DPT; ++i) out[i] = o[i] * inv;
  }
}

template <typename T, int HD>
static size_t fa_smem() {
  return (size_t)(FA_BQ * (HD + 1) + FA_BK * (HD + 1) + FA_BK * HD + FA_BQ * (FA_BK + 1)) * sizeof(float);
}

template <typename T, int HD>
static cudaError_t fa_set_attr() {
  return cudaFuncSetAttribute(attn_prefill_simt_kernel<T, HD>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fa_smem<T, HD>());
}

template <typename T>
static cudaError_t attn_prefill(const Dims& d, const float* Q, int T_, int pos0, const void* kc,
                                const void* vc, float* O, cudaStream_t s) {
  const dim3 grid((T_ + FA_BQ - 1) / FA_BQ, d.nq), block(256);
  const float scale = 1.f / sqrtf((float)d.hd);
  switch (d.hd) {
    case 16: attn_prefill_simt_kernel<T, 16><<<grid, block, fa_smem<T, 16>(), s>>>(Q, T_, d.nq, d.nkv, pos0, (const T*)kc, (const T*)vc, d.cap, scale, O); break;
    case 32: attn_prefill_simt_kernel<T, 32><<<grid, block, fa_smem<T, 32>(), s>>>(Q, T_, d.nq, d.nkv, pos0, (const T*)kc, (const T*)vc, d.cap, scale, O); break;
    case 64: attn_prefill_simt_kernel<T, 64><<<grid, block, fa_smem<T, 64>(), s>>>(Q, T_, d.nq, d.nkv, pos0, (const T*)kc, (const T*)vc, d.cap, scale, O); break;
    case 128: attn_prefill_simt_kernel<T, 128><<<grid, block, fa_smem<T, 128>(), s>>>(Q, T_, d.nq, d.nkv, pos0, (const T*)kc, (const T*)vc, d.cap, scale, O); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename T>
static cudaError_t set_attr_t() {
  cudaError_t e;
  if ((e = fa_set_attr<T, 16>())) return e;
  if ((e = fa_set_attr<T, 32>())) return e;
  if ((e = fa_set_attr<T, 64>())) return e;
  return fa_set_attr<T, 128>();
}

static cudaError_t pm_set_attributes();

cudaError_t prefill_set_attributes(const Dims& d) {
  cudaError_t e = d.dtype == 1 ? set_attr_t<f16>() : set_attr_t<float>();
  if (e || d.dtype != 1) return e;
  if ((e = pm_set_attributes())) return e;
  if (!gemm_tc_available()) return cudaSuccess;
  if ((e = attn_prefill_tc_set_attributes())) return e;
  return gemm_tc_set_attributes();
}

template <typename W, typename KV>
static cudaError_t prefill_simt(const Dims& d, const LayerPtrs* layers, const void* embed,
                                const int* ids, int T_, int pos0, const float2* rope, void* kcache,
                                const PrefillBufs& b, int* err, cudaStream_t s) {
  const int H = d.H, qd = d.nq * d.hd, kvd = d.nkv * d.hd, Wd = qd + 2 * kvd;
  embed_rows_kernel<W><<<T_, 256, 0, s>>>((const W*)embed, d.V, H, ids, b.X, err);
  const size_t layer_stride = (size_t)d.nkv * d.cap * d.hd;  // elements per layer per K or V
  for (int l = 0; l < d.L; ++l) {
    const LayerPtrs& w = layers[l];
    KV* kc = (KV*)kcache + (size_t)l * 2 * layer_stride;
    KV* vc = kc + layer_stride;
    norm_rows_kernel<W, float><<<T_, 256, 0, s>>>(b.X, (const W*)w.in_norm, H, d.eps, b.Xn, err);
    gemm_simt<W>(b.Xn, H, w.wq, H, w.bq, b.Y, Wd, T_, qd, H, false, s);
    gemm_simt<W>(b.Xn, H, w.wk, H, w.bk, b.Y + qd, Wd, T_, kvd, H, false, s);
    gemm_simt<W>(b.Xn, H, w.wv, H, w.bv, b.Y + qd + kvd, Wd, T_, kvd, H, false, s);
    rope_kv_kernel<KV><<<T_, 256, 0, s>>>(b.Y, T_, d.nq, d.nkv, d.hd, pos0, d.cap, rope, b.Q, kc, vc, err);
    cudaError_t e = attn_prefill<KV>(d, b.Q, T_, pos0, kc, vc, b.O, s);
    if (e) return e;
    gemm_simt<W>(b.O, qd, w.wo, qd, nullptr, b.X, H, T_, H, qd, true, s);
    norm_rows_kernel<W, float><<<T_, 256, 0, s>>>(b.X, (const W*)w.post_norm, H, d.eps, b.Xn, err);
    gemm_simt<W>(b.Xn, H, w.w_gate, H, nullptr, b.G, d.I, T_, d.I, H, false, s);
    gemm_simt<W>(b.Xn, H, w.w_up, H, nullptr, b.U, d.I, T_, d.I, H, false, s);
    const size_t n = (size_t)T_ * d.I;
    swiglu_kernel<<<(unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0, s>>>(b.G, b.U, b.G, n);
    gemm_simt<W>(b.G, d.I, w.w_down, d.I, nullptr, b.X, H, T_, H, d.I, true, s);
  }
  return cudaGetLastError();
}

// ---- prefill attention on the tensor cores (bf16 models: fp16 cache) --------------------
//
// Causal attention of T query rows over keys 0..pos0+T-1 ("LLM Speedrun: Architecture":
// Attention, Causal mask, Grouped Query Attention), in the streaming form with a running
// maximum and sum per row. One CTA per (128 query rows, head), eight warps of 16 rows each.
// S = Q K^T and O += P V run as mma.sync m16n8k16 with fp16 operands and fp32
// accumulators: q (scaled by 1/sqrt(hd)) and the probabilities are rounded to fp16 like the
// cache. Q stays in registers as A fragments; key and value tiles of 64 rows arrive by
// cp.async (two buffers, rows padded by 16 bytes so fragment loads are bank-conflict free):
// key B fragments are 32-bit shared loads, value B fragments come from ldmatrix.trans. The
// output goes straight to the fp16 operand of the o_proj GEMM.
constexpr int PM_WARPS = 8, PM_Q = 16 * PM_WARPS, PM_K = 64;

template <int HD>
__global__ void __launch_bounds__(PM_WARPS * 32) attn_prefill_mma_kernel(const float* Q, int T_, int nq, int nkv,
                                                                        int pos0, const f16* kc, const f16* vc,
                                                                        int cap, float scale, f16* Oh) {
  constexpr int KS = HD + 8;      // halves per key / value row in shared memory (16-byte pad)
  constexpr int NKK = HD / 16;    // k-steps of S = Q K^T
  constexpr int NNT = HD / 8;     // n-tiles of O
  extern __shared__ __align__(16) unsigned char pm_smem[];
  f16* Ks = reinterpret_cast<f16*>(pm_smem);  // [2][PM_K][KS]
  f16* Vs = Ks + 2 * PM_K * KS;               // [2][PM_K][KS]
  const int qb = gridDim.x - 1 - blockIdx.x;  // the longest (last) query blocks first
  const int h = blockIdx.y, g = h / (nq / nkv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  const int q0 = qb * PM_Q;
  const int r_lo = q0 + warp * 16 + gid, r_hi = r_lo + 8;  // this thread's two query rows
  const int last_q = min(T_, q0 + PM_Q) - 1;
  const int last_key = pos0 + last_q;
  const int ntiles = last_key / PM_K + 1;
  const f16* K = kc + (size_t)g * cap * HD;
  const f16* V = vc + (size_t)g * cap * HD;

  uint32_t qa[NKK][4];  // Q as A fragments, scaled
#pragma unroll
  for (int kk = 0; kk < NKK; ++kk) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = (r & 1) ? r_hi : r_lo;
      const int col = 16 * kk + ((r & 2) ? 8 : 0) + 2 * tig;
      float2 v = make_float2(0.f, 0.f);
      if (row < T_) v = *reinterpret_cast<const float2*>(Q + (size_t)row * nq * HD + (size_t)h * HD + col);
      qa[kk][r] = pack_half2(v.x * scale, v.y * scale);
    }
  }
  auto load_tile = [&](int t, int buf) {  // key and value rows by cp.async, zeros past the last key
    constexpr int NV = PM_K * HD / 8;
    const int k0 = t * PM_K;
    for (int i = tid; i < 2 * NV; i += PM_WARPS * 32) {
      const int which = i >= NV, idx = i - which * NV;
      const int j = idx / (HD / 8), c8 = idx - j * (HD / 8);
      f16* dst = (which ? Vs : Ks) + (size_t)buf * PM_K * KS + j * KS + c8 * 8;
      if (k0 + j <= last_key) cp_async16(dst, (which ? V : K) + (size_t)(k0 + j) * HD + c8 * 8);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  float o[NNT][4];
#pragma unroll
  for (int nt = 0; nt < NNT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  const int pos_lo = pos0 + r_lo, pos_hi = pos0 + r_hi;
  const int warp_first = pos0 + q0 + warp * 16;  // smallest position among this warp's rows
  // value rows of ldmatrix.trans: row (lane % 8) + 8 ((lane / 8) % 2) of a 16-key step,
  // columns of n-tile pair (lane / 16)
  const int v_row = (lane & 7) + ((lane >> 3) & 1) * 8, v_col = (lane >> 4) * 8;

  load_tile(0, 0);
  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1, k0 = t * PM_K;
    if (t + 1 < ntiles) {
      load_tile(t + 1, buf ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();  // tile t visible to every warp
    const f16* kt = Ks + (size_t)buf * PM_K * KS;
    const f16* vt = Vs + (size_t)buf * PM_K * KS;
    if (k0 <= pos0 + min(q0 + warp * 16 + 15, last_q)) {  // some key of the tile is visible to this warp
      float sc[PM_K / 8][4];
#pragma unroll
      for (int nt = 0; nt < PM_K / 8; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        const f16* krow = kt + (size_t)(8 * nt + gid) * KS + 2 * tig;
#pragma unroll
        for (int kk = 0; kk < NKK; ++kk) {
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow + 16 * kk);
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(krow + 16 * kk + 8);
          mma16816(sc[nt], qa[kk], b0, b1);
        }
      }
      if (k0 + PM_K - 1 > warp_first) {  // the tile reaches past some row's position: mask
#pragma unroll
        for (int nt = 0; nt < PM_K / 8; ++nt) {
          const int j = k0 + 8 * nt + 2 * tig;
          if (j > pos_lo) sc[nt][0] = -INFINITY;
          if (j + 1 > pos_lo) sc[nt][1] = -INFINITY;
          if (j > pos_hi) sc[nt][2] = -INFINITY;
          if (j + 1 > pos_hi) sc[nt][3] = -INFINITY;
        }
      }
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < PM_K / 8; ++nt) {
        mx_lo = fmaxf(mx_lo, fmaxf(sc[nt][0], sc[nt][1]));
        mx_hi = fmaxf(mx_hi, fmaxf(sc[nt][2], sc[nt][3]));
      }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      // rows with no visible key yet (only padding rows past T) keep a zero state
      const float c_lo = m_lo == -INFINITY ? 0.f : expf(m_lo - mn_lo);
      const float c_hi = m_hi == -INFINITY ? 0.f : expf(m_hi - mn_hi);
      float s_lo = 0.f, s_hi = 0.f;
      uint32_t pa[PM_K / 16][4];
#pragma unroll
      for (int nt = 0; nt < PM_K / 8; ++nt) {
        const float p0 = mn_lo == -INFINITY ? 0.f : expf(sc[nt][0] - mn_lo);
        const float p1 = mn_lo == -INFINITY ? 0.f : expf(sc[nt][1] - mn_lo);
        const float p2 = mn_hi == -INFINITY ? 0.f : expf(sc[nt][2] - mn_hi);
        const float p3 = mn_hi == -INFINITY ? 0.f : expf(sc[nt][3] - mn_hi);
        s_lo += p0 + p1;
        s_hi += p2 + p3;
        pa[nt >> 1][(nt & 1) * 2 + 0] = pack_half2(p0, p1);
        pa[nt >> 1][(nt & 1) * 2 + 1] = pack_half2(p2, p3);
      }
      s_lo += __shfl_xor_sync(0xffffffffu, s_lo, 1);
      s_lo += __shfl_xor_sync(0xffffffffu, s_lo, 2);
      s_hi += __shfl_xor_sync(0xffffffffu, s_hi, 1);
      s_hi += __shfl_xor_sync(0xffffffffu, s_hi, 2);
      l_lo = l_lo * c_lo + s_lo;
      l_hi = l_hi * c_hi + s_hi;
      m_lo = mn_lo;
      m_hi = mn_hi;
#pragma unroll
      for (int nt = 0; nt < NNT; ++nt) {
        o[nt][0] *= c_lo;
        o[nt][1] *= c_lo;
        o[nt][2] *= c_hi;
        o[nt][3] *= c_hi;
      }
#pragma unroll
      for (int kk = 0; kk < PM_K / 16; ++kk) {
        const f16* vrow = vt + (size_t)(16 * kk + v_row) * KS + v_col;
#pragma unroll
        for (int nt = 0; nt < NNT; nt += 2) {
          uint32_t b[4];
          ldmatrix_x4_trans(b, vrow + nt * 8);
          mma16816(o[nt], pa[kk], b[0], b[1]);
          mma16816(o[nt + 1], pa[kk], b[2], b[3]);
        }
      }
    }
    __syncthreads();  // every warp is done with buffer buf
  }
  const float i_lo = l_lo > 0.f ? 1.f / l_lo : 0.f, i_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
#pragma unroll
  for (int nt = 0; nt < NNT; ++nt) {
    const int col = h * HD + 8 * nt + 2 * tig;
    if (r_lo < T_)
      *reinterpret_cast<__half2*>(Oh + (size_t)r_lo * nq * HD + col) = __floats2half2_rn(o[nt][0] * i_lo, o[nt][1] * i_lo);
    if (r_hi < T_)
      *reinterpret_cast<__half2*>(Oh + (size_t)r_hi * nq * HD + col) = __floats2half2_rn(o[nt][2] * i_hi, o[nt][3] * i_hi);
  }
}

template <int HD>
static constexpr size_t pm_smem() {
  return (size_t)2 * 2 * PM_K * (HD + 8) * sizeof(f16);
}

static cudaError_t pm_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(attn_prefill_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pm_smem<128>());
  if (e) return e;
  return cudaFuncSetAttribute(attn_prefill_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)pm_smem<64>());
}

// tensor-core prefill attention into the fp16 o_proj operand; false if the head size has no
// instance (the caller then uses the CUDA-core kernel)
static bool attn_prefill_mma(const Dims& d, const float* Q, int T_, int pos0, const f16* kc, const f16* vc, f16* Oh,
                             cudaStream_t s, cudaError_t* e) {
  const dim3 grid((T_ + PM_Q - 1) / PM_Q, d.nq), block(PM_WARPS * 32);
  const float scale = 1.f / sqrtf((float)d.hd);
  if (d.hd == 128) {
    attn_prefill_mma_kernel<128><<<grid, block, pm_smem<128>(), s>>>(Q, T_, d.nq, d.nkv, pos0, kc, vc, d.cap, scale, Oh);
  } else if (d.hd == 64) {
    attn_prefill_mma_kernel<64><<<grid, block, pm_smem<64>(), s>>>(Q, T_, d.nq, d.nkv, pos0, kc, vc, d.cap, scale, Oh);
  } else {
    return false;
  }
  *e = cudaGetLastError();
  return true;
}

// Prefill attention of the bf16 models: QW_PREFILL_ATTN=tc (tcgen05, the default), mma
// (mma.sync) or simt (CUDA cores), for comparison; read at every prefill.
enum { PA_TC, PA_MMA, PA_SIMT };
static int prefill_attention_kind() {
  const char* e = std::getenv("QW_PREFILL_ATTN");
  if (e && !std::strcmp(e, "mma")) return PA_MMA;
  if (e && !std::strcmp(e, "simt")) return PA_SIMT;
  return PA_TC;
}

// bf16 models: every projection on the tensor cores with fp16 operands (fp16 copies of the
// bf16 weights are exact from 2^-14 to 65504 in magnitude, smaller ones round among the fp16
// subnormals; fp16 activations round 8x finer than bf16), fp32 accumulation, fp32 residual
// stream, fp16 KV cache.
static cudaError_t prefill_tc(const Dims& d, const LayerPtrs* layers, const void* embed,
                              const int* ids, int T_, int pos0, const float2* rope, void* kcache,
                              const PrefillBufs& b, int* err, cudaStream_t s) {
  const int H = d.H, qd = d.nq * d.hd, kvd = d.nkv * d.hd, Wd = qd + 2 * kvd;
  // Every kernel after the embedding is launched with programmatic dependent launch: it starts
  // while the previous one drains, requests its weights, and waits for that grid before it
  // touches activations.
  const bool pdl = tc_pdl();
  const int kind = prefill_attention_kind();
  embed_rows_kernel<bf16><<<T_, 256, 0, s>>>((const bf16*)embed, d.V, H, ids, b.X, err);
  const size_t layer_stride = (size_t)d.nkv * d.cap * d.hd;
  cudaError_t e;
  for (int l = 0; l < d.L; ++l) {
    const LayerPtrs& w = layers[l];
    f16* kc = (f16*)kcache + (size_t)l * 2 * layer_stride;
    f16* vc = kc + layer_stride;
    norm_rows_h(b.X, (const bf16*)w.in_norm, T_, H, d.eps, b.Xh, err, s, d.nsm);
    // q | k | v as one projection: the three fp16 matrices lie back to back (each head's rows
    // in RoPE-pair order), and so do the columns of the output
    if (w.wk16 != (const f16*)w.wq16 + (size_t)qd * H || w.wv16 != (const f16*)w.wk16 + (size_t)kvd * H ||
        (w.bq && !w.bqkv))
      return cudaErrorInvalidValue;
    const f16* wqkv = (const f16*)w.wq16;
    const bf16* bqkv = (const bf16*)w.bqkv;
    if (kind == PA_TC && attn_prefill_tc_supported(d.hd) && d.I >= qd) {
      // bias, RoPE and the K/V append in the projection's epilogue; q in fp16, scaled into
      // base-2 scores, in the (still free) SwiGLU operand buffer
      const QkvOut o{b.Ah, kc, vc, rope, 1.4426950408889634f / sqrtf((float)d.hd), d.nq, d.nkv, d.hd, pos0, d.cap};
      if ((e = gemm_tc_qkv(b.Xh, H, wqkv, H, bqkv, T_, Wd, H, o, err, s, b.ws, b.ws_floats, d.nsm, pdl))) return e;
      if ((e = attn_prefill_tc(d, T_, pos0, b.Ah, kc, vc, b.Oh, err, s))) return e;
    } else {
      if ((e = gemm_tc(b.Xh, H, wqkv, H, bqkv, b.Y, Wd, T_, Wd, H, false, err, s, b.ws, b.ws_floats, d.nsm, pdl))) return e;
      rope_kv_kernel<f16><<<T_, 256, 0, s>>>(b.Y, T_, d.nq, d.nkv, d.hd, pos0, d.cap, rope, b.Q, kc, vc, err, true);
      const bool mma = kind != PA_SIMT && attn_prefill_mma(d, b.Q, T_, pos0, kc, vc, b.Oh, s, &e);
      if (mma && e) return e;
      if (!mma) {
        if ((e = attn_prefill<f16>(d, b.Q, T_, pos0, kc, vc, b.O, s))) return e;
        const size_t no = (size_t)T_ * qd;
        to_half_kernel<<<(unsigned)((no + 255) / 256 < 4096 ? (no + 255) / 256 : 4096), 256, 0, s>>>(b.O, b.Oh, no,
                                                                                                     err);
      }
    }
    if ((e = gemm_tc(b.Oh, qd, (const f16*)w.wo16, qd, nullptr, b.X, H, T_, H, qd, true, err, s, b.ws, b.ws_floats, d.nsm, pdl))) return e;
    norm_rows_h(b.X, (const bf16*)w.post_norm, T_, H, d.eps, b.Xh, err, s, d.nsm);
    if ((e = gemm_tc_swiglu(b.Xh, H, (const f16*)w.wg16, (const f16*)w.wu16, H, b.Ah, d.I, T_, d.I, H, err, s, b.ws,
                              b.ws_floats, d.nsm, pdl)))
      return e;
    if ((e = gemm_tc(b.Ah, d.I, (const f16*)w.wd16, d.I, nullptr, b.X, H, T_, H, d.I, true, err, s, b.ws, b.ws_floats, d.nsm, pdl))) return e;
  }
  return cudaGetLastError();
}

cudaError_t prefill_layers(const Dims& d, const LayerPtrs* layers, const void* embed,
                           const int* ids_dev, int T, int pos0, const float2* rope,
                           void* kcache_seq, const PrefillBufs& b, int* err, cudaStream_t s) {
  if (d.dtype == 1) {
    if (b.use_tc) return prefill_tc(d, layers, embed, ids_dev, T, pos0, rope, kcache_seq, b, err, s);
    return prefill_simt<bf16, f16>(d, layers, embed, ids_dev, T, pos0, rope, kcache_seq, b, err, s);
  }
  return prefill_simt<float, float>(d, layers, embed, ids_dev, T, pos0, rope, kcache_seq, b, err, s);
}

// bf16 -> fp16 weight copy. A bf16 value has 8 significant bits, so the copy is exact for
// 2^-17 <= |x| <= 65504; smaller magnitudes land among the fp16 subnormals and round to a
// multiple of 2^-24 (an absolute error below 2^-25), larger ones set ERR_RANGE.
__global__ void bf16_to_half_kernel(const bf16* src, f16* dst, size_t n, int* err) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = to_half_checked(__bfloat162float(src[i]), err);
}

cudaError_t convert_bf16_to_half(const void* src, void* dst, size_t n, int* err, cudaStream_t s) {
  const size_t blocks = (n + 255) / 256;
  bf16_to_half_kernel<<<(unsigned)(blocks < 8192 ? blocks : 8192), 256, 0, s>>>((const bf16*)src, (f16*)dst, n, err);
  return cudaGetLastError();
}

// The same copy of a matrix of whole heads (rows = heads x hd, K columns each) with every
// head's rows in RoPE-pair order: row 2i + e of a head is source row i + e hd/2, so the two
// members of each rotation pair come out of a projection as adjacent columns.
__global__ void bf16_to_half_pairs_kernel(const bf16* src, f16* dst, size_t rows, int K, int hd, int* err) {
  const int half = hd >> 1;
  for (size_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const size_t head = r / hd;
    const int j = (int)(r - head * hd);
    const bf16* s_row = src + (head * hd + (j >> 1) + (j & 1) * half) * (size_t)K;
    f16* d_row = dst + r * (size_t)K;
    for (int k = threadIdx.x; k < K; k += blockDim.x) d_row[k] = to_half_checked(__bfloat162float(s_row[k]), err);
  }
}

cudaError_t convert_bf16_to_half_pairs(const void* src, void* dst, size_t rows, int K, int hd, int* err,
                                       cudaStream_t s) {
  if (hd <= 0 || hd % 2 || rows % hd) return cudaErrorInvalidValue;
  bf16_to_half_pairs_kernel<<<(unsigned)(rows < 8192 ? rows : 8192), 256, 0, s>>>((const bf16*)src, (f16*)dst, rows,
                                                                                 K, hd, err);
  return cudaGetLastError();
}

// a bias vector of whole heads into the same pair order (bf16 kept)
__global__ void bias_pairs_kernel(const bf16* src, bf16* dst, int n, int hd) {
  const int half = hd >> 1;
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < n; c += gridDim.x * blockDim.x) {
    const int head = c / hd, j = c - head * hd;
    dst[c] = src[head * hd + (j >> 1) + (j & 1) * half];
  }
}

cudaError_t copy_bias_pairs(const void* src, void* dst, int n, int hd, cudaStream_t s) {
  if (hd <= 0 || hd % 2 || n % hd) return cudaErrorInvalidValue;
  bias_pairs_kernel<<<(n + 255) / 256, 256, 0, s>>>((const bf16*)src, (bf16*)dst, n, hd);
  return cudaGetLastError();
}

}  // namespace qw
