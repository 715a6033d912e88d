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
  float* part;            // [nq][nsplit_max][attn_part_stride(hd)]: output, max, sum
  unsigned int* counter;  // [nkv]
  unsigned long long* tl;  // timeline slots or null
  // several sequences (grid z): per-sequence strides of q, the KV cache, the output, the
  // partials (elements) and the counters; an fp16 output instead of out; active flags
  size_t q_zs, kv_zs, out_zs, part_zs;
  int counter_zs;
  f16* out16;
  const int* active;
  int merge;  // 0: stop after the partials (the consumer merges them)
};

// One CTA per (KV head, context chunk). The CTA copies q of its g query heads and the K and
// V rows of its chunk into shared memory with one batch of 16-byte loads, then:
//   scores  8 lanes per position, each summing over every 8th 16-byte vector of the row for
//           all g heads at once (each K row read once), the 8 partial dot products added
//           with 3 shuffles;
//   softmax a warp per head: running max and sum of exp over the chunk;
//   values  a thread per (position group, head, 16-byte vector of the row), accumulating
//           with independent lanes of the vector, the position groups added in shared memory.
// The unnormalised output, max and sum of every chunk go to the workspace; the last CTA of
// the KV head to finish merges the chunks (deterministic log-sum-exp combine) with every
// value it reads requested before the first is used.
constexpr int ATTN_THREADS = 256;
constexpr int COPY_BATCH = 8;
constexpr int RED_FLOATS = ATTN_THREADS * 8;  // position-group partial sums of the values
constexpr int MERGE_BATCH = 8;                // chunks merged per batch of loads

template <typename KV> struct KVec;
template <> struct KVec<f16> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4& r, float* f) {
    const __half2* h = reinterpret_cast<const __half2*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __half22float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
};
template <> struct KVec<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4& r, float* f) {
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
  }
};

template <typename KV>
__global__ void __launch_bounds__(ATTN_THREADS) attn_decode_kernel(const AttnArgs<KV> a_in) {
  extern __shared__ __align__(16) float sm[];
  __shared__ bool s_last;
  const int z = blockIdx.z;  // sequence
  if (a_in.active && !a_in.active[z]) return;
  AttnArgs<KV> a = a_in;
  a.q += z * a.q_zs;
  a.k += z * a.kv_zs;
  a.v += z * a.kv_zs;
  if (a.d_pos) a.d_pos += z;
  a.part += z * a.part_zs;
  a.counter += z * a.counter_zs;
  if (a.out16) a.out16 += z * a.out_zs;
  else a.out += z * a.out_zs;
  constexpr int EV = KVec<KV>::N;  // KV elements per 16-byte vector
  const int g = blockIdx.x, split = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = ATTN_THREADS >> 5;
  const int G = a.group, hd = a.hd, NV = hd / EV;
  tl_stamp(a.tl, 0);
  // The context length and every K/V row but the newest were written before this decode
  // step began (the position by the previous step's LM head, the rows by earlier steps):
  // they are read before the dependency wait, which only the query and the newest row
  // (written by the projections just before) have to follow.
  const int ctx = a.d_pos ? __ldcg(a.d_pos) + 1 : a.ctx_host;
  const int chunk = max(a.chunk_min, (ctx + a.nsplit_max - 1) / a.nsplit_max);
  const int nsplit = (ctx + chunk - 1) / chunk;
  if (split >= nsplit) return;  // an exited CTA counts as triggered
  const int j0 = split * chunk, j1 = min(ctx, j0 + chunk), n = j1 - j0;
  const int n_old = j1 == ctx ? n - 1 : n;  // rows of the chunk written by earlier steps
  // shared layout: q [G][hd] | scores [G][chunk] | stats [G][2] | merge (m, l) [2][G][nsplit_max]
  //                | value partials [RED_FLOATS] | K [chunk][hd] KV | V [chunk][hd] KV
  float* qs = sm;
  float* sc = qs + G * hd;
  float* st = sc + G * chunk;
  float* mw = st + 2 * G;
  float* red = mw + 2 * G * a.nsplit_max;
  const int kv_off = (G * hd + G * chunk + 2 * G + 2 * G * a.nsplit_max + RED_FLOATS + 3) & ~3;
  KV* ks = reinterpret_cast<KV*>(sm + kv_off);
  KV* vs = ks + (size_t)chunk * hd;
  const uint4* ksrc = reinterpret_cast<const uint4*>(a.k + ((size_t)g * a.stride + j0) * hd);
  const uint4* vsrc = reinterpret_cast<const uint4*>(a.v + ((size_t)g * a.stride + j0) * hd);
  uint4* kdst = reinterpret_cast<uint4*>(ks);
  uint4* vdst = reinterpret_cast<uint4*>(vs);
  {
    const int kvv = n_old * NV;  // 16-byte vectors of the K (and the V) rows
    for (int base = tid; base < 2 * kvv; base += COPY_BATCH * ATTN_THREADS) {
      uint4 r[COPY_BATCH];
#pragma unroll
      for (int i = 0; i < COPY_BATCH; ++i) {
        const int j = base + i * ATTN_THREADS;
        if (j < kvv) r[i] = __ldcg(ksrc + j);
        else if (j < 2 * kvv) r[i] = __ldcg(vsrc + (j - kvv));
      }
#pragma unroll
      for (int i = 0; i < COPY_BATCH; ++i) {
        const int j = base + i * ATTN_THREADS;
        if (j < kvv) kdst[j] = r[i];
        else if (j < 2 * kvv) vdst[j - kvv] = r[i];
      }
    }
  }
  pdl_wait();
  pdl_trigger();
  tl_stamp(a.tl, 1);
  {  // q of the G heads and, in the last chunk, the newest K/V row
    const int qv = G * hd / 4;
    const int nv_new = n_old < n ? NV : 0;
    const uint4* qsrc = reinterpret_cast<const uint4*>(a.q + (size_t)g * G * hd);
    uint4* qdst = reinterpret_cast<uint4*>(qs);
    for (int j = tid; j < qv + 2 * nv_new; j += ATTN_THREADS) {
      if (j < qv) qdst[j] = __ldcg(qsrc + j);
      else if (j < qv + nv_new) kdst[n_old * NV + (j - qv)] = __ldcg(ksrc + n_old * NV + (j - qv));
      else vdst[n_old * NV + (j - qv - nv_new)] = __ldcg(vsrc + n_old * NV + (j - qv - nv_new));
    }
  }
  __syncthreads();

  // ---- scores: position jb + tid / 8, vectors (tid % 8) + 8 i of its K row
  const int p8 = lane & 7;
  for (int jb = 0; jb < n; jb += ATTN_THREADS / 8) {
    const int jj = jb + (tid >> 3);
    float dot[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) dot[h] = 0.f;
    if (jj < n) {
      const uint4* krow = reinterpret_cast<const uint4*>(ks + (size_t)jj * hd);
      for (int v = p8; v < NV; v += 8) {
        float kf[EV];
        KVec<KV>::unpack(krow[v], kf);
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          if (h < G) {
            const float4* q4 = reinterpret_cast<const float4*>(qs + h * hd + v * EV);
#pragma unroll
            for (int e4 = 0; e4 < EV / 4; ++e4) {
              const float4 t = q4[e4];
              dot[h] = fmaf(t.x, kf[4 * e4], fmaf(t.y, kf[4 * e4 + 1],
                       fmaf(t.z, kf[4 * e4 + 2], fmaf(t.w, kf[4 * e4 + 3], dot[h]))));
            }
          }
        }
      }
    }
    float mine = 0.f;  // lane p8 keeps the score of head p8
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      if (h < G) {
        float d = dot[h];
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        if (p8 == h) mine = d;
      }
    }
    if (jj < n && p8 < G) sc[p8 * chunk + jj] = mine * a.scale;
  }
  __syncthreads();

  // ---- softmax statistics of the chunk, a warp per head
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

  // ---- values: thread (pg, h, v) sums positions pg, pg + PG, ... of head h, vector v
  const int units = G * NV;  // <= ATTN_THREADS since G * hd <= 1024
  const int PG = ATTN_THREADS / units;
  const int t_pg = tid / units, t_u = tid - t_pg * units;
  const int th = t_u / NV, tv = t_u - th * NV;
  float acc[EV];
#pragma unroll
  for (int e = 0; e < EV; ++e) acc[e] = 0.f;
  if (t_pg < PG) {
    const uint4* vcol = reinterpret_cast<const uint4*>(vs) + tv;
    const float* ph = sc + th * chunk;
    for (int jj = t_pg; jj < n; jj += PG) {
      float vf[EV];
      KVec<KV>::unpack(vcol[(size_t)jj * NV], vf);
      const float pj = ph[jj];
#pragma unroll
      for (int e = 0; e < EV; ++e) acc[e] = fmaf(pj, vf[e], acc[e]);
    }
    if (PG > 1) {
#pragma unroll
      for (int e = 0; e < EV; ++e) red[tid * EV + e] = acc[e];
    }
  }
  if (PG > 1) {
    __syncthreads();
    if (tid < units) {
      for (int pg = 1; pg < PG; ++pg) {
#pragma unroll
        for (int e = 0; e < EV; ++e) acc[e] += red[(pg * units + tid) * EV + e];
      }
    }
  }
  const int pstride = attn_part_stride(hd);
  if (tid < units) {
    float* dst = a.part + ((size_t)(g * G + th) * a.nsplit_max + split) * pstride + tv * EV;
#pragma unroll
    for (int e = 0; e < EV; ++e) dst[e] = acc[e];
  }
  if (tid < G) {
    float* p = a.part + ((size_t)(g * G + tid) * a.nsplit_max + split) * pstride;
    p[hd] = st[2 * tid];
    p[hd + 1] = st[2 * tid + 1];
  }
  if (!a.merge) {
    tl_stamp(a.tl, 2);
    return;
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

  // ---- merge: w_s = exp(m_s - M) / sum_s l_s exp(m_s - M) per head, out = sum_s w_s O_s.
  // The first batch of partial outputs is requested before the (m, l) pairs are read.
  constexpr int EPT = GMAX * 128 / ATTN_THREADS;  // output elements per thread (G*hd <= 1024)
  const float* pbase = a.part + (size_t)g * G * a.nsplit_max * pstride;
  float vals[EPT][MERGE_BATCH];
  auto load_batch = [&](int s0) {
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const int idx = tid + k * ATTN_THREADS;
      const int h = idx / hd, dd = idx - h * hd;
#pragma unroll
      for (int u = 0; u < MERGE_BATCH; ++u)
        vals[k][u] = (idx < G * hd && s0 + u < nsplit)
                         ? __ldcg(pbase + ((size_t)h * a.nsplit_max + s0 + u) * pstride + dd)
                         : 0.f;
    }
  };
  load_batch(0);
  for (int i = tid; i < G * nsplit; i += ATTN_THREADS) {  // (m, l) of every (head, chunk)
    const int h = i / nsplit, sp = i - h * nsplit;
    const float* p = pbase + ((size_t)h * a.nsplit_max + sp) * pstride + hd;
    const float m = __ldcg(p), l = __ldcg(p + 1);
    mw[h * a.nsplit_max + sp] = m;
    mw[(G + h) * a.nsplit_max + sp] = l;
  }
  __syncthreads();
  for (int h = warp; h < G; h += nwarps) {
    float M = -INFINITY;
    for (int sp = lane; sp < nsplit; sp += 32) M = fmaxf(M, mw[h * a.nsplit_max + sp]);
    M = warp_max(M);
    float L = 0.f;
    for (int sp = lane; sp < nsplit; sp += 32) {
      const float w = expf(mw[h * a.nsplit_max + sp] - M);
      mw[h * a.nsplit_max + sp] = w;
      L = fmaf(mw[(G + h) * a.nsplit_max + sp], w, L);
    }
    L = warp_sum(L);
    const float inv = 1.f / L;
    for (int sp = lane; sp < nsplit; sp += 32) mw[h * a.nsplit_max + sp] *= inv;
  }
  __syncthreads();
  float out[EPT];
#pragma unroll
  for (int k = 0; k < EPT; ++k) out[k] = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += MERGE_BATCH) {
    if (s0) load_batch(s0);
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const int idx = tid + k * ATTN_THREADS;
      const int h = idx / hd;
#pragma unroll
      for (int u = 0; u < MERGE_BATCH; ++u)
        if (idx < G * hd && s0 + u < nsplit) out[k] = fmaf(vals[k][u], mw[h * a.nsplit_max + s0 + u], out[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < EPT; ++k) {
    const int idx = tid + k * ATTN_THREADS;
    if (idx < G * hd) {
      if (a.out16) a.out16[(size_t)g * G * hd + idx] = __float2half_rn(out[k]);
      else a.out[(size_t)g * G * hd + idx] = out[k];
    }
  }
  if (tid == 0) a.counter[g] = 0u;
  tl_stamp(a.tl, 2);
}

// ---- decode attention of several sequences on the tensor cores (batched decode) ---------
//
// One CTA per (KV head, context chunk, sequence). The g query heads of the KV head are the
// rows of one m16n8k16 A operand (fp16 q scaled by 1/sqrt(hd), rows >= g zero). Key/value
// tiles of 64 positions arrive by cp.async into two buffers (rows padded by 16 bytes; the
// first two tiles are requested before the dependency wait, but for the newest row); each
// of the four warps takes 16 positions of a tile: S = Q K^T as two n-tiles, a running
// maximum and sum per row, O += P V with the value B fragments loaded by ldmatrix.trans.
// The warps' states are combined (log-sum-exp) in shared memory into the chunk's partial
// (unnormalised output, maximum, sum) for the merge kernel.
constexpr int DM_K = 64, DM_WARPS = 4;

struct DecMmaArgs {
  const float* q;    // [nseq][nq * hd]
  const f16 *k, *v;  // layer caches of sequence 0: [nkv][stride][hd]
  size_t kv_zs;      // elements from one sequence's caches to the next's
  int stride, hd, group, nq, nsplit_max, chunk_min;
  const int* d_pos;  // [nseq]
  const int* active; // [nseq], or null: all
  float scale;
  float* part;       // [nseq][part_zs]: [nq][nsplit_max][attn_part_stride(hd)]
  size_t part_zs;
  unsigned long long* tl;
};

template <int HD>
static constexpr size_t dm_smem() {
  return (size_t)2 * 2 * DM_K * (HD + 8) * sizeof(f16);  // K and V, two buffers (the combine reuses them)
}

template <int HD>
__global__ void __launch_bounds__(DM_WARPS * 32) attn_decode_mma_kernel(const DecMmaArgs a) {
  constexpr int KS = HD + 8, NKK = HD / 16, NNT = HD / 8;
  extern __shared__ __align__(16) unsigned char dm_smem_raw[];
  f16* Ks = reinterpret_cast<f16*>(dm_smem_raw);  // [2][DM_K][KS]
  f16* Vs = Ks + 2 * DM_K * KS;                    // [2][DM_K][KS]
  const int g = blockIdx.x, split = blockIdx.y, z = blockIdx.z;
  if (a.active && !a.active[z]) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  const int G = a.group;
  tl_stamp(a.tl, 0);
  const int ctx = __ldcg(a.d_pos + z) + 1;
  const int chunk = max(a.chunk_min, (ctx + a.nsplit_max - 1) / a.nsplit_max);
  const int nsplit = (ctx + chunk - 1) / chunk;
  if (split >= nsplit) return;
  const int j0 = split * chunk, j1 = min(ctx, j0 + chunk), n = j1 - j0;
  const int ntiles = (n + DM_K - 1) / DM_K;
  const f16* K = a.k + z * a.kv_zs + ((size_t)g * a.stride + j0) * HD;
  const f16* V = a.v + z * a.kv_zs + ((size_t)g * a.stride + j0) * HD;
  // the first tile's rows written by earlier steps are fetched before the dependency wait;
  // q and the newest row (written by the projections just before) only after it
  const int newest = j1 == ctx ? n - 1 : -1;  // chunk-relative, or none in this chunk
  auto load_tile = [&](int t, int buf, int skip) {  // rows t*DM_K.. of K and V (row skip left out)
    constexpr int NV = DM_K * HD / 8;  // 16-byte vectors of a K (or V) tile
    for (int i = tid; i < 2 * NV; i += DM_WARPS * 32) {
      const int which = i >= NV, idx = i - which * NV;
      const int j = idx / (HD / 8), c8 = idx - j * (HD / 8);
      f16* dst = (which ? Vs : Ks) + (size_t)buf * DM_K * KS + j * KS + c8 * 8;
      const int key = t * DM_K + j;
      if (key == skip) continue;
      if (key < n) cp_async16(dst, (which ? V : K) + (size_t)key * HD + c8 * 8);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // the first two tiles (both buffers) are requested before the wait, all but the newest row
  const int pre = ntiles < 2 ? ntiles : 2;
  const bool newest_in_pre = newest >= 0 && newest < pre * DM_K;
  load_tile(0, 0, newest_in_pre ? newest : -1);
  if (pre == 2) load_tile(1, 1, newest_in_pre ? newest : -1);
  pdl_wait();
  pdl_trigger();
  tl_stamp(a.tl, 1);
  if (newest_in_pre) {  // its own copy group, after the rest of the preloaded tiles
    for (int i = tid; i < 2 * (HD / 8); i += DM_WARPS * 32) {
      const int which = i >= HD / 8, c8 = i - which * (HD / 8);
      f16* dst = (which ? Vs : Ks) + (size_t)newest * KS + c8 * 8;  // (buffer newest / DM_K)
      cp_async16(dst, (which ? V : K) + (size_t)newest * HD + c8 * 8);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  uint32_t qa[NKK][4];
  {
    const float* qz = a.q + (size_t)z * a.nq * HD + (size_t)g * G * HD;
#pragma unroll
    for (int kk = 0; kk < NKK; ++kk)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = (r & 1) ? gid + 8 : gid;
        const int col = 16 * kk + ((r & 2) ? 8 : 0) + 2 * tig;
        float2 v = make_float2(0.f, 0.f);
        if (row < G) v = __ldcg(reinterpret_cast<const float2*>(qz + (size_t)row * HD + col));
        qa[kk][r] = pack_half2(v.x * a.scale, v.y * a.scale);
      }
  }
  float o[NNT][4];
#pragma unroll
  for (int nt = 0; nt < NNT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  const int kw = 16 * warp;  // this warp's positions within a tile
  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1;
    if (t + 1 < ntiles && t + 1 >= pre) {
      load_tile(t + 1, buf ^ 1, -1);  // (the newest row lies in a preloaded tile or is loaded here after the wait)
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const f16* kt = Ks + (size_t)buf * DM_K * KS;
    const f16* vt = Vs + (size_t)buf * DM_K * KS;
    if (t * DM_K + kw < n) {  // some of this warp's positions exist
      float sc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        const f16* krow = kt + (size_t)(kw + 8 * nt + gid) * KS + 2 * tig;
#pragma unroll
        for (int kk = 0; kk < NKK; ++kk)
          mma16816(sc[nt], qa[kk], *reinterpret_cast<const uint32_t*>(krow + 16 * kk),
                   *reinterpret_cast<const uint32_t*>(krow + 16 * kk + 8));
        const int key = t * DM_K + kw + 8 * nt + 2 * tig;  // positions past the chunk: masked
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
      float p[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        p[nt][0] = mn_lo == -INFINITY ? 0.f : expf(sc[nt][0] - mn_lo);
        p[nt][1] = mn_lo == -INFINITY ? 0.f : expf(sc[nt][1] - mn_lo);
        p[nt][2] = mn_hi == -INFINITY ? 0.f : expf(sc[nt][2] - mn_hi);
        p[nt][3] = mn_hi == -INFINITY ? 0.f : expf(sc[nt][3] - mn_hi);
      }
      float s_lo = p[0][0] + p[0][1] + p[1][0] + p[1][1], s_hi = p[0][2] + p[0][3] + p[1][2] + p[1][3];
      s_lo += __shfl_xor_sync(0xffffffffu, s_lo, 1);
      s_lo += __shfl_xor_sync(0xffffffffu, s_lo, 2);
      s_hi += __shfl_xor_sync(0xffffffffu, s_hi, 1);
      s_hi += __shfl_xor_sync(0xffffffffu, s_hi, 2);
      l_lo = l_lo * c_lo + s_lo;
      l_hi = l_hi * c_hi + s_hi;
      m_lo = mn_lo;
      m_hi = mn_hi;
      const uint32_t pa[4] = {pack_half2(p[0][0], p[0][1]), pack_half2(p[0][2], p[0][3]),
                              pack_half2(p[1][0], p[1][1]), pack_half2(p[1][2], p[1][3])};
      // value rows kw + (lane % 8) + 8 ((lane / 8) % 2), columns of n-tile pair nt, nt + 1
      const f16* vrow = vt + (size_t)(kw + (lane & 7) + ((lane >> 3) & 1) * 8) * KS + (lane >> 4) * 8;
#pragma unroll
      for (int nt = 0; nt < NNT; nt += 2) {
        o[nt][0] *= c_lo;
        o[nt][1] *= c_lo;
        o[nt][2] *= c_hi;
        o[nt][3] *= c_hi;
        o[nt + 1][0] *= c_lo;
        o[nt + 1][1] *= c_lo;
        o[nt + 1][2] *= c_hi;
        o[nt + 1][3] *= c_hi;
        uint32_t b[4];
        ldmatrix_x4_trans(b, vrow + nt * 8);
        mma16816(o[nt], pa, b[0], b[1]);
        mma16816(o[nt + 1], pa, b[2], b[3]);
      }
    }
    __syncthreads();  // buffer buf is free again
  }
  // combine the four warps (rows < G) in shared memory (the tile buffers are free now)
  float* cO = reinterpret_cast<float*>(dm_smem_raw);  // [DM_WARPS][16][HD]
  float* cM = cO + DM_WARPS * 16 * HD;                 // [DM_WARPS][16]
  float* cL = cM + DM_WARPS * 16;
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
  __syncthreads();
  const int ps = attn_part_stride(HD);
  float* part = a.part + (size_t)z * a.part_zs;
  for (int idx = tid; idx < G * HD; idx += DM_WARPS * 32) {
    const int r = idx / HD, d = idx - r * HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < DM_WARPS; ++w) M = fmaxf(M, cM[w * 16 + r]);
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < DM_WARPS; ++w) {
      const float mw = cM[w * 16 + r];
      if (mw != -INFINITY) acc = fmaf(expf(mw - M), cO[(size_t)(w * 16 + r) * HD + d], acc);
    }
    part[((size_t)(g * G + r) * a.nsplit_max + split) * ps + d] = acc;
  }
  if (tid < G) {
    float M = -INFINITY, L = 0.f;
#pragma unroll
    for (int w = 0; w < DM_WARPS; ++w) M = fmaxf(M, cM[w * 16 + tid]);
#pragma unroll
    for (int w = 0; w < DM_WARPS; ++w) {
      const float mw = cM[w * 16 + tid];
      if (mw != -INFINITY) L = fmaf(expf(mw - M), cL[w * 16 + tid], L);
    }
    float* pp = part + ((size_t)(g * G + tid) * a.nsplit_max + split) * ps;
    pp[HD] = M;
    pp[HD + 1] = L;
  }
  tl_stamp(a.tl, 2);
}

// Tensor-core decode attention of nseq sequences (fp16 caches, head_dim 64 or 128, at most
// 16 query heads per KV head): chunk partials in ws as for launch_attn_batched (merge 0).
cudaError_t launch_attn_decode_mma(int nq, int nkv, int hd, int nsplit, int chunk_min, const float* q, const f16* kc,
                                   const f16* vc, size_t kv_zs, int kv_stride, const int* d_pos, const int* active,
                                   int nseq, void* ws, unsigned long long* tl, cudaStream_t s, bool pdl) {
  const int G = nq / nkv;
  if (G > 16 || (hd != 64 && hd != 128)) return cudaErrorInvalidValue;
  DecMmaArgs a{q, kc, vc, kv_zs, kv_stride, hd, G, nq, nsplit, chunk_min, d_pos, active, 1.f / sqrtf((float)hd),
               (float*)ws, attn_batched_part_floats(nq, hd, nsplit), tl};
  const dim3 grid(nkv, nsplit, nseq), block(DM_WARPS * 32);
  if (hd == 128) return launch_k(attn_decode_mma_kernel<128>, grid, block, dm_smem<128>(), s, pdl, a);
  return launch_k(attn_decode_mma_kernel<64>, grid, block, dm_smem<64>(), s, pdl, a);
}

cudaError_t attn_decode_mma_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(attn_decode_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)dm_smem<128>());
  if (e) return e;
  return cudaFuncSetAttribute(attn_decode_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)dm_smem<64>());
}

// ---- host side ------------------------------------------------------------

size_t attn_workspace_bytes(int nq, int nkv, int hd, int nsplit) {
  size_t part = (size_t)nq * nsplit * attn_part_stride(hd) * sizeof(float);
  part = (part + 255) & ~(size_t)255;
  return part + (size_t)nkv * sizeof(unsigned int);
}

// Chunks of at least chunk_min positions and at most MAX_SPLITS chunks per KV head (short
// contexts spread over several CTAs, the merge stays short), unless the K and V rows of a
// chunk would exceed ~160 KB of shared memory; then the chunk count grows instead.
int attn_nsplit_for(int cap, int chunk_min, int hd, int kv_bytes, int max_splits) {
  int chunk_max = (160 * 1024) / (2 * hd * kv_bytes);
  if (chunk_max > 256) chunk_max = 256;
  if (chunk_max < chunk_min) chunk_max = chunk_min;
  int n = (cap + chunk_min - 1) / chunk_min;
  if (n > max_splits) n = max_splits;
  const int need = (cap + chunk_max - 1) / chunk_max;
  if (n < need) n = need;
  return n < 1 ? 1 : n;
}

size_t attn_smem_bytes(int group, int hd, int cap, int nsplit, int chunk_min, int kv_bytes) {
  int chunk = (cap + nsplit - 1) / nsplit;
  if (chunk < chunk_min) chunk = chunk_min;
  const size_t f = ((size_t)group * hd + (size_t)group * chunk + 2 * group + 2 * (size_t)group * nsplit +
                    RED_FLOATS + 3) & ~(size_t)3;
  return f * sizeof(float) + 2 * (size_t)chunk * hd * kv_bytes;
}

cudaError_t launch_attn(int kv_dtype, int nq, int nkv, int hd, int nsplit, int chunk_min,
                        size_t smem, const float* q, const void* kc, const void* vc,
                        int kv_stride, const int* d_pos, int ctx_host, float* out, void* ws,
                        unsigned long long* tl, cudaStream_t s, bool pdl, int merge) {  // merge: see AttnArgs
  const int G = nq / nkv;
  if (G > GMAX) return cudaErrorInvalidValue;
  size_t part_bytes = ((size_t)nq * nsplit * attn_part_stride(hd) * sizeof(float) + 255) & ~(size_t)255;
  const dim3 grid(nkv, nsplit), block(ATTN_THREADS);
  if (kv_dtype == 2) {
    AttnArgs<f16> a{q, (const f16*)kc, (const f16*)vc, kv_stride, hd, G, nsplit, chunk_min,
                     ctx_host, d_pos, 1.f / sqrtf((float)hd), out, (float*)ws,
                     (unsigned int*)((char*)ws + part_bytes), tl, 0, 0, 0, 0, 0, nullptr, nullptr, merge};
    return launch_k(attn_decode_kernel<f16>, grid, block, smem, s, pdl, a);
  }
  AttnArgs<float> a{q, (const float*)kc, (const float*)vc, kv_stride, hd, G, nsplit, chunk_min,
                    ctx_host, d_pos, 1.f / sqrtf((float)hd), out, (float*)ws,
                    (unsigned int*)((char*)ws + part_bytes), tl, 0, 0, 0, 0, 0, nullptr, nullptr, merge};
  return launch_k(attn_decode_kernel<float>, grid, block, smem, s, pdl, a);
}

// Decode attention of nseq sequences in one launch (grid z = sequence, inactive ones exit):
// q [nseq][nq*hd] fp32; the fp16 caches of sequence z start kv_zs elements after those of
// sequence z - 1; output fp16 [nseq][nq*hd]; workspace: partials [nseq][...] then counters
// [nseq][nkv] (attn_batched_workspace_bytes).
size_t attn_batched_part_floats(int nq, int hd, int nsplit) {
  return (((size_t)nq * nsplit * attn_part_stride(hd) * sizeof(float) + 255) & ~(size_t)255) / sizeof(float);
}
size_t attn_batched_workspace_bytes(int nq, int nkv, int hd, int nsplit, int nseq) {
  const size_t part = ((size_t)nq * nsplit * attn_part_stride(hd) * sizeof(float) + 255) & ~(size_t)255;
  return part * nseq + (size_t)nkv * nseq * sizeof(unsigned int);
}
cudaError_t launch_attn_batched(int nq, int nkv, int hd, int nsplit, int chunk_min, size_t smem,
                                const float* q, const f16* kc, const f16* vc, size_t kv_zs, int kv_stride,
                                const int* d_pos, const int* active, int nseq, f16* out16, void* ws,
                                unsigned long long* tl, cudaStream_t s, int merge) {
  const int G = nq / nkv;
  if (G > GMAX) return cudaErrorInvalidValue;
  const size_t part_bytes = ((size_t)nq * nsplit * attn_part_stride(hd) * sizeof(float) + 255) & ~(size_t)255;
  AttnArgs<f16> a{q, kc, vc, kv_stride, hd, G, nsplit, chunk_min, 0, d_pos, 1.f / sqrtf((float)hd), nullptr,
                  (float*)ws, (unsigned int*)((char*)ws + part_bytes * nseq), tl,
                  (size_t)nq * hd, kv_zs, (size_t)nq * hd, part_bytes / sizeof(float), nkv, out16, active, merge};
  return launch_k(attn_decode_kernel<f16>, dim3(nkv, nsplit, nseq), dim3(ATTN_THREADS), smem, s, batched_pdl(), a);
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
