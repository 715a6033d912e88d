// Decode attention of one token over the KV cache ("LLM Speedrun: Architecture":
// Attention, Causal mask, Grouped Query Attention): for every query head h, softmax over
// positions j <= pos of q_h . K_j / sqrt(d), then the weighted sum of V_j, where query head h
// reads KV head h / (n_heads / n_kv_heads). The context is split into chunks whose softmax
// statistics are merged exactly (log-sum-exp).
#include "common.cuh"
#include "internal.h"

#include <math.h>

namespace qw {

constexpr int GMAX = 8;  // most query heads per KV head

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
  unsigned long long* tl;  // timeline slots or null
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
  tl_stamp(a.tl, 0);
  pdl_wait();
  pdl_trigger();
  tl_stamp(a.tl, 1);
  const int ctx = a.d_pos ? __ldcg(a.d_pos) + 1 : a.ctx_host;
  const int chunk = max(a.chunk_min, (ctx + a.nsplit_max - 1) / a.nsplit_max);
  const int nsplit = (ctx + chunk - 1) / chunk;
  if (split >= nsplit) {
    tl_stamp(a.tl, 2);
    return;
  }
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
  if (!s_last) {
    tl_stamp(a.tl, 2);
    return;
  }
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
  tl_stamp(a.tl, 2);
}

// ---- host side ------------------------------------------------------------

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
                        unsigned long long* tl, cudaStream_t s, bool pdl) {
  const int G = nq / nkv;
  if (G > GMAX) return cudaErrorInvalidValue;
  size_t part_bytes = ((size_t)nq * nsplit * (hd + 2) * sizeof(float) + 255) & ~(size_t)255;
  const dim3 grid(nkv, nsplit), block(ATTN_THREADS);
  if (kv_dtype == 2) {
    AttnArgs<f16> a{q, (const f16*)kc, (const f16*)vc, kv_stride, hd, G, nsplit, chunk_min,
                     ctx_host, d_pos, 1.f / sqrtf((float)hd), out, (float*)ws,
                     (unsigned int*)((char*)ws + part_bytes), tl};
    return launch_k(attn_decode_kernel<f16>, grid, block, smem, s, pdl, a);
  }
  AttnArgs<float> a{q, (const float*)kc, (const float*)vc, kv_stride, hd, G, nsplit, chunk_min,
                    ctx_host, d_pos, 1.f / sqrtf((float)hd), out, (float*)ws,
                    (unsigned int*)((char*)ws + part_bytes), tl};
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

}  // namespace qw
