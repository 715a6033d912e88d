// Batched greedy decode: one decode step of up to 16 independent sequences, each at its own
// position, with every weight matrix read once per step for all of them ("augur",
// Features: batched generation; the per-sequence computation is the decoder forward pass of
// "LLM Speedrun: Architecture", Transformer architecture and Implementing Qwen).
//
// Per layer:
//   norm     x[b] -> RMSNorm -> fp16 row b of X            (rows of absent sequences: 0)
//   qkv      skinny tensor-core GEMM of Wq|Wk|Wv against X (split-K fp32 partials)
//   qkv_epi  partial sums + bias, split-half RoPE at pos[b], q out, K/V append for seq b
//   attn     decode attention, grid z = sequence, fp16 output rows
//   o        skinny GEMM of Wo, then x[b] += partial sums
//   norm     post-attention RMSNorm -> X
//   gate/up  skinny GEMM of Wg|Wu, then SwiGLU -> fp16 rows A
//   down     skinny GEMM of Wd against A, then x[b] += partial sums
// then the final norm (bf16 rows), the LM head as a skinny GEMM over the bf16 embedding
// with a fused per-sequence argmax, and the per-sequence token / position bookkeeping.
//
// Layer matrices use the fp16 copies made for the prefill (fp16 activations keep the
// error of the bf16 path inside its tolerance); the LM head uses the bf16 embedding with
// bf16 activations (a one-layer error, far inside the tolerance).
#include "common.cuh"
#include <cooperative_groups.h>
#include "internal.h"

#include <math.h>
#include <stdlib.h>

namespace qw {

constexpr int BT = 256;  // threads of the element-wise kernels

constexpr int MAX_SPLITS = SKINNY_MAX_SPLITS;

// Sum of the split partials of column c of sequence b (fixed split order); every load is
// issued before the first add.
__device__ __forceinline__ float psum(const float* part, int splits, int n_total, int b, int c) {
  float v[MAX_SPLITS];
#pragma unroll
  for (int s = 0; s < MAX_SPLITS; ++s) v[s] = s < splits ? __ldcg(part + ((size_t)s * 16 + b) * n_total + c) : 0.f;
  float acc = 0.f;
#pragma unroll
  for (int s = 0; s < MAX_SPLITS; ++s) acc += v[s];
  return acc;
}

// one element of a normalised row: fp16 rows feed the tensor cores (range checked), bf16
// rows the LM head (the fp32 range)
__device__ __forceinline__ void store_row(f16* o, float v, int* err) { *o = to_half_checked(v, err); }
__device__ __forceinline__ void store_row(bf16* o, float v, int*) { *o = __float2bfloat16_rn(v); }

constexpr int RN_CL = 8;         // CTAs per sequence (one thread-block cluster)
constexpr int RN_THREADS = 256;
constexpr int RN_COLS = 4;       // columns per thread: H <= RN_CL * RN_THREADS * RN_COLS

// Row b of out = RMSNorm(x[b]) * gain after x[b] += the split partials (part may be null:
// no residual add; embed non-null: x[b] = embedding row of tok[b] first). A cluster of RN_CL
// CTAs per sequence, each owning a contiguous share of the columns: every load of a share is
// issued before the first use, and the CTAs' sums of squares meet through distributed shared
// memory, added in rank order (deterministic). Rows of absent or inactive sequences are zero.
template <typename OutT>
__global__ void __cluster_dims__(RN_CL, 1, 1) __launch_bounds__(RN_THREADS)
bresid_norm_kernel(const float* part, int splits, int n_total, const bf16* embed, int V, const int* tok, float* x,
                   const bf16* gain, int H, float eps, const int* active, int nseq, OutT* out, int* err,
                   unsigned long long* tl) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  __shared__ float scratch[32];
  __shared__ float s_ss;
  tl_stamp(tl, 0);
  pdl_wait();
  pdl_trigger();
  tl_stamp(tl, 1);
  const int rank = (int)cl.block_rank(), b = blockIdx.y;
  const int per = (H + RN_CL - 1) / RN_CL;
  const int c0 = rank * per, c1 = min(H, c0 + per);
  OutT* o = out + (size_t)b * H;
  if (b >= nseq || !active[b]) {  // the whole cluster takes this branch
    for (int k = c0 + threadIdx.x; k < c1; k += RN_THREADS) o[k] = from_f32<OutT>(0.f);
    tl_stamp(tl, 2);
    return;
  }
  float* xb = x + (size_t)b * H;
  const bf16* erow = nullptr;
  if (embed) {
    int t = __ldcg(tok + b);
    if (t < 0 || t >= V) {
      if (threadIdx.x == 0 && rank == 0) atomicOr(err, ERR_TOKEN);
      t = 0;
    }
    erow = embed + (size_t)t * H;
  }
  float v[RN_COLS], g[RN_COLS];
#pragma unroll
  for (int j = 0; j < RN_COLS; ++j) {
    const int k = c0 + threadIdx.x + j * RN_THREADS;
    v[j] = 0.f;
    g[j] = 0.f;
    if (k < c1) {
      v[j] = erow ? __bfloat162float(erow[k]) : __ldcg(xb + k);
      g[j] = __bfloat162float(gain[k]);
      if (part) v[j] += psum(part, splits, n_total, b, k);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < RN_COLS; ++j) {
    const int k = c0 + threadIdx.x + j * RN_THREADS;
    if (k < c1) {
      if (part || erow) xb[k] = v[j];
      ss = fmaf(v[j], v[j], ss);
    }
  }
  ss = block_sum(ss, scratch);
  if (threadIdx.x == 0) s_ss = ss;
  cl.sync();  // every CTA's share of the sum is in its shared memory
  float tot = 0.f;
#pragma unroll
  for (int r = 0; r < RN_CL; ++r) tot += *cl.map_shared_rank(&s_ss, r);
  cl.sync();  // the peers have read this CTA's share: it may exit
  const float inv = rsqrtf(tot / (float)H + eps);
#pragma unroll
  for (int j = 0; j < RN_COLS; ++j) {
    const int k = c0 + threadIdx.x + j * RN_THREADS;
    if (k < c1) store_row(o + k, v[j] * inv * g[j], err);
  }
  tl_stamp(tl, 2);
}


// q/k/v of sequence b from the partials (each head's columns in RoPE-pair order, as the fp16
// weight copies' rows are): + bias, split-half RoPE of q and k at pos[b], q to
// q_out[b], k and v appended to the sequence's cache at pos[b]. One thread per RoPE pair.
__global__ void bqkv_epi_kernel(const float* part, int splits, int n_total, int nq, int nkv, int hd,
                                const bf16* bq, const bf16* bk, const bf16* bv, const float2* rope,
                                const int* pos, const int* active, float* q_out, f16* kc0, size_t kv_zs,
                                int cap, int* err, unsigned long long* tl) {
  tl_stamp(tl, 0);
  pdl_wait();
  pdl_trigger();
  tl_stamp(tl, 1);
  const int b = blockIdx.y;
  if (!active[b]) return;
  const int half = hd >> 1;
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= (nq + 2 * nkv) * half) return;
  const int p = __ldcg(pos + b);
  if (p < 0 || p >= cap) return;  // the host checks capacity before every step
  int head = item / half;
  const int i = item - head * half;
  const int ca = head * hd + 2 * i, cb = ca + 1;  // columns of the pair in q|k|v (pair-ordered weights)
  float a = psum(part, splits, n_total, b, ca), c = psum(part, splits, n_total, b, cb);
  const bf16* bias;
  int h;
  if (head < nq) { bias = bq; h = head; }
  else if (head < nq + nkv) { bias = bk; h = head - nq; }
  else { bias = bv; h = head - nq - nkv; }
  if (bias) {
    a += __bfloat162float(bias[h * hd + i]);
    c += __bfloat162float(bias[h * hd + i + half]);
  }
  if (head < nq + nkv) {
    const float2 cs = rope[(size_t)p * half + i];
    const float ra = a * cs.x - c * cs.y, rc = c * cs.x + a * cs.y;
    a = ra;
    c = rc;
  }
  if (head < nq) {
    float* qb = q_out + (size_t)b * nq * hd;
    qb[h * hd + i] = a;
    qb[h * hd + i + half] = c;
  } else {
    // the layer's cache of sequence b: [2][nkv][cap][hd], K then V
    f16* base = kc0 + (size_t)b * kv_zs + (head < nq + nkv ? 0 : (size_t)nkv * cap * hd);
    f16* dst = base + ((size_t)h * cap + p) * hd;
    dst[i] = to_half_checked(a, err);
    dst[i + half] = to_half_checked(c, err);
  }
  tl_stamp(tl, 2);
}

// A[b][i] = silu(gate) * up as fp16 (gate columns [0, I), up columns [I, 2I)); rows of
// absent or inactive sequences are zero
__global__ void bswiglu_kernel(const float* part, int splits, int n_total, int I, const int* active, int nseq,
                               f16* A, int* err, unsigned long long* tl) {
  tl_stamp(tl, 0);
  pdl_wait();
  pdl_trigger();
  tl_stamp(tl, 1);
  const int b = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= I) return;
  float v = 0.f;
  if (b < nseq && active[b]) {
    const float g = psum(part, splits, n_total, b, i), u = psum(part, splits, n_total, b, I + i);
    v = (g / (1.f + expf(-g))) * u;
  }
  A[(size_t)b * I + i] = to_half_checked(v, err);
  tl_stamp(tl, 2);
}

// Attention output of sequence b, head h from the chunk partials of the attention kernel
// (per chunk: unnormalised output, maximum m_s, sum of exponentials l_s): o = sum_s w_s O_s
// with w_s = exp(m_s - M) / sum_s' l_s' exp(m_s' - M) (exact log-sum-exp combine, chunk
// order), written as the fp16 row of the o_proj GEMM. One CTA per (head, sequence), one
// thread per output element; every partial it reads is requested before the first use.
constexpr int BM_SPLITS = 32;  // chunks merged per (sequence, head), at most
__global__ void __launch_bounds__(128) bmerge_kernel(const float* part, size_t part_zs, int nq, int hd,
                                                     int nsplit_max, int chunk_min, const int* pos,
                                                     const int* active, f16* O16, unsigned long long* tl) {
  __shared__ float w[BM_SPLITS];
  tl_stamp(tl, 0);
  pdl_wait();
  pdl_trigger();
  tl_stamp(tl, 1);
  const int h = blockIdx.x, b = blockIdx.y;
  if (!active[b]) return;
  const int ctx = __ldcg(pos + b) + 1;
  const int chunk = max(chunk_min, (ctx + nsplit_max - 1) / nsplit_max);
  const int ns = min((ctx + chunk - 1) / chunk, BM_SPLITS);
  const int ps = attn_part_stride(hd);
  const float* base = part + (size_t)b * part_zs + (size_t)h * nsplit_max * ps;
  float v[BM_SPLITS];
#pragma unroll
  for (int s = 0; s < BM_SPLITS; ++s)
    v[s] = (int)threadIdx.x < hd && s < ns ? __ldcg(base + (size_t)s * ps + threadIdx.x) : 0.f;
  if (threadIdx.x < 32) {  // warp 0: the merge weights
    const int s = threadIdx.x;
    const float m = s < ns ? __ldcg(base + (size_t)s * ps + hd) : -INFINITY;
    const float l = s < ns ? __ldcg(base + (size_t)s * ps + hd + 1) : 0.f;
    const float M = warp_max(m);
    const float e = s < ns ? expf(m - M) : 0.f;
    const float L = warp_sum(l * e);
    w[s] = e / L;
  }
  __syncthreads();
  if ((int)threadIdx.x < hd) {
    float acc = 0.f;
#pragma unroll
    for (int s = 0; s < BM_SPLITS; ++s)
      if (s < ns) acc = fmaf(v[s], w[s], acc);
    O16[((size_t)b * nq + h) * hd + threadIdx.x] = __float2half_rn(acc);
  }
  tl_stamp(tl, 2);
}

// per active sequence: token = argmax (lowest index among equal maxima), history, length
__global__ void bfinalize_kernel(unsigned long long* keys, int* tok, int* pos, int* hist, int* hist_n, int cap,
                                 const int* active, int nseq, unsigned long long* tl) {
  tl_stamp(tl, 0);
  pdl_wait();
  pdl_trigger();
  tl_stamp(tl, 1);
  tl_stamp(tl, 2);
  const int b = threadIdx.x;
  if (b >= nseq || !active[b]) return;
  const unsigned long long k = keys[b];
  const int idx = argmax_key_index(k);
  tok[b] = idx;
  const int n = hist_n[b];
  if (n < cap) hist[(size_t)b * cap + n] = idx;
  hist_n[b] = n + 1;
  pos[b] += 1;
  keys[b] = 0ull;
}

cudaError_t batched_set_attributes() { return skinny_set_attributes(); }

// Programmatic dependent launch between the kernels of a batched step (QW_BATCHED_NOPDL=1:
// plain stream order, for comparison).
bool batched_pdl() {
  static const bool on = [] {
    const char* v = std::getenv("QW_BATCHED_NOPDL");
    return !(v && v[0] == '1');
  }();
  return on;
}

cudaError_t batched_step(const BatchedCtx& c, cudaStream_t s) {
  const bool pdl = batched_pdl();
  const Dims& d = c.d;
  const int S = d.max_seqs, H = d.H, I = d.I;
  if (H > RN_CL * RN_THREADS * RN_COLS) return cudaErrorInvalidValue;
  cudaError_t e;
  const dim3 rn_grid(RN_CL, 16), rn_block(RN_THREADS);
  const float* no_part = nullptr;
  const bf16* no_embed = nullptr;
  const int* no_tok = nullptr;
  int li = 0;  // launch index: timeline slots [3 li, 3 li + 3)
  auto tl = [&]() -> unsigned long long* { return c.tl ? c.tl + 3 * (li++) : nullptr; };
  // layer 0 input: embedding rows, then the first RMSNorm
  if ((e = launch_k(bresid_norm_kernel<f16>, rn_grid, rn_block, 0, s, pdl, no_part, 0, 0, (const bf16*)c.embed,
                    d.V, (const int*)c.tok, c.x, (const bf16*)c.layers[0].in_norm, H, d.eps, c.active, S, c.X16,
                    c.err, tl())))
    return e;
  for (int l = 0; l < d.L; ++l) {
    const LayerPtrs& w = c.layers[l];
    const BatchedLayerPlans& pl = c.plans[l];
    f16* kc0 = (f16*)c.kv + (size_t)l * 2 * d.nkv * d.cap * d.hd;  // layer l of sequence 0
    if ((e = skinny_run(pl.qkv, c.part, nullptr, 0, S, c.active, nullptr, c.err, tl(), s))) return e;
    const int pairs = (d.nq + 2 * d.nkv) * (d.hd / 2);
    if ((e = launch_k(bqkv_epi_kernel, dim3((pairs + BT - 1) / BT, S), dim3(BT), 0, s, pdl, (const float*)c.part,
                      pl.qkv.splits, pl.qkv.n_total, d.nq, d.nkv, d.hd, (const bf16*)w.bq, (const bf16*)w.bk,
                      (const bf16*)w.bv, c.rope, (const int*)c.pos, c.active, c.q, kc0, c.kv_seq_elems, d.cap,
                      c.err, tl())))
      return e;
    // attention leaves its chunk partials; the merge kernel writes the fp16 rows of the o GEMM
    if (c.attn_mma)
      e = launch_attn_decode_mma(d.nq, d.nkv, d.hd, c.attn_nsplit, c.attn_chunk, c.q, kc0,
                                 kc0 + (size_t)d.nkv * d.cap * d.hd, c.kv_seq_elems, d.cap, c.pos, c.active, S,
                                 c.attn_ws, tl(), s, pdl);
    else
      e = launch_attn_batched(d.nq, d.nkv, d.hd, c.attn_nsplit, c.attn_chunk, c.attn_smem, c.q, kc0,
                              kc0 + (size_t)d.nkv * d.cap * d.hd, c.kv_seq_elems, d.cap, c.pos, c.active, S, c.O16,
                              c.attn_ws, tl(), s, /*merge=*/0);
    if (e) return e;
    if ((e = launch_k(bmerge_kernel, dim3(d.nq, S), dim3(128), 0, s, pdl, (const float*)c.attn_ws,
                      attn_batched_part_floats(d.nq, d.hd, c.attn_nsplit), d.nq, d.hd, c.attn_nsplit,
                      c.attn_chunk, (const int*)c.pos, c.active, c.O16, tl())))
      return e;
    if ((e = skinny_run(pl.o, c.part, nullptr, 0, S, c.active, nullptr, c.err, tl(), s))) return e;
    if ((e = launch_k(bresid_norm_kernel<f16>, rn_grid, rn_block, 0, s, pdl, (const float*)c.part, pl.o.splits,
                      pl.o.n_total, no_embed, 0, no_tok, c.x, (const bf16*)w.post_norm, H, d.eps, c.active, S, c.X16,
                      c.err, tl())))
      return e;
    if (pl.gu.glu) {  // SwiGLU in the GEMM's epilogue
      if ((e = skinny_run(pl.gu, nullptr, nullptr, 0, S, c.active, nullptr, c.err, tl(), s, c.A16))) return e;
    } else {
      if ((e = skinny_run(pl.gu, c.part, nullptr, 0, S, c.active, nullptr, c.err, tl(), s))) return e;
      if ((e = launch_k(bswiglu_kernel, dim3((I + BT - 1) / BT, 16), dim3(BT), 0, s, pdl, (const float*)c.part,
                        pl.gu.splits, pl.gu.n_total, I, c.active, S, c.A16, c.err, tl())))
        return e;
    }
    if ((e = skinny_run(pl.down, c.part, nullptr, 0, S, c.active, nullptr, c.err, tl(), s))) return e;
    // x += down partials, then the next layer's input norm (fp16) or the final norm (bf16)
    if (l + 1 < d.L)
      e = launch_k(bresid_norm_kernel<f16>, rn_grid, rn_block, 0, s, pdl, (const float*)c.part, pl.down.splits,
                   pl.down.n_total, no_embed, 0, no_tok, c.x, (const bf16*)c.layers[l + 1].in_norm, H, d.eps,
                   c.active, S, c.X16, c.err, tl());
    else
      e = launch_k(bresid_norm_kernel<bf16>, rn_grid, rn_block, 0, s, pdl, (const float*)c.part, pl.down.splits,
                   pl.down.n_total, no_embed, 0, no_tok, c.x, (const bf16*)c.final_norm, H, d.eps, c.active, S,
                   c.Xb16, c.err, tl());
    if (e) return e;
  }
  if ((e = skinny_run(c.lm, nullptr, c.logits, d.V, S, c.active, c.keys, c.err, tl(), s))) return e;
  return launch_k(bfinalize_kernel, dim3(1), dim3(32), 0, s, pdl, c.keys, c.tok, c.pos, c.hist, c.hist_n, d.cap,
                  c.active, S, tl());
}

}  // namespace qw
