// Host-side declarations shared by the libqw translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qw {

// Device-side error bits (ERR_*) are defined in common.cuh.

struct Dims {
  int L, H, nq, nkv, hd, I, V;
  float eps, theta;
  int dtype;      // 0 f32, 1 bf16 (weights and KV cache)
  int cap;        // KV positions per sequence
  int max_seqs;
  int nsm;        // SM count of the device
  int attn_nsplit;  // maximum context splits of decode attention
  int attn_chunk_min;
};

struct LayerPtrs {
  const void *in_norm, *wq, *bq, *wk, *bk, *wv, *bv, *wo, *post_norm, *w_gate, *w_up, *w_down;
  // fp16 copies of the matrices (bf16 models; prefill tensor-core operands). wq16, wk16 and
  // wv16 lie back to back (one [nq*hd + 2*nkv*hd][H] matrix) with every head's rows in
  // RoPE-pair order (row 2i + e = source row i + e hd/2), bqkv holds bq | bk | bv (bf16) in
  // the same order, or is null without q/k/v biases.
  const void *wq16, *wk16, *wv16, *wo16, *wg16, *wu16, *wd16;
  const void* bqkv;
};

// Argmax / position bookkeeping written by the last CTA of the LM-head kernel.
struct Finalize {
  unsigned long long* key;  // packed argmax key, reset to 0 after use
  unsigned int* counter;    // CTA arrival counter, reset to 0 after use
  int* tok;                 // greedy token out
  int* pos;                 // sequence length
  int pos_set;              // >= 0: set length to this value; < 0: length += 1
  int* hist;                // token history (may be null)
  int* hist_n;              // its count
  int hist_cap;
  int* err;
};

// ---- api.cu ----
void set_error_message(const char* msg);  // message returned by qw_last_error on this thread
// bytes of workspace qw_op_decode_attention uses for this shape and KV type (kv_dtype a
// qw_dtype); the per-KV-head counters occupy its last n_kv_heads * 4 bytes
size_t op_attn_workspace_exact(int kv_dtype, int n_heads, int n_kv_heads, int head_dim, int kv_stride);

// Floats per (head, chunk) row of the decode-attention partials: hd outputs, the maximum,
// the sum of exponentials, padding to 16 bytes (rows stay aligned for vector loads).
__host__ __device__ constexpr int attn_part_stride(int hd) { return hd + 4; }

// ---- decode.cu ----
size_t attn_workspace_bytes(int nq, int nkv, int hd, int nsplit);
// Context chunks of decode attention for a cache of cap positions: at least chunk_min
// positions each, at most max_splits chunks unless a chunk's K and V rows would exceed
// ~160 KB of shared memory.
int attn_nsplit_for(int cap, int chunk_min, int hd, int kv_bytes, int max_splits = 16);
size_t attn_smem_bytes(int group, int hd, int cap, int nsplit, int chunk_min, int kv_bytes);
cudaError_t decode_set_attributes(const Dims& d);
cudaError_t attn_set_attributes(size_t smem);  // not during stream capture
size_t attn_batched_workspace_bytes(int nq, int nkv, int hd, int nsplit, int nseq);
cudaError_t launch_attn_batched(int nq, int nkv, int hd, int nsplit, int chunk_min, size_t smem,
                                const float* q, const __half* kc, const __half* vc, size_t kv_zs, int kv_stride,
                                const int* d_pos, const int* active, int nseq, __half* out16, void* ws,
                                unsigned long long* tl, cudaStream_t s, int merge = 1);
size_t attn_batched_part_floats(int nq, int hd, int nsplit);  // partial floats per sequence
cudaError_t launch_attn_decode_mma(int nq, int nkv, int hd, int nsplit, int chunk_min, const float* q,
                                   const __half* kc, const __half* vc, size_t kv_zs, int kv_stride, const int* d_pos,
                                   const int* active, int nseq, void* ws, unsigned long long* tl, cudaStream_t s,
                                   bool pdl);
cudaError_t attn_decode_mma_set_attributes();

// tl: three timeline slots (start, past the dependency wait, end) or null
cudaError_t launch_embed(const Dims& d, const void* E, const int* tok, float* x, int* err,
                         unsigned long long* tl, cudaStream_t s, bool pdl);
cudaError_t launch_qkv(const Dims& d, const LayerPtrs& w, const float* x, const int* d_pos,
                       const float2* rope, float* q, void* kc, void* vc, int* err,
                       unsigned long long* tl, cudaStream_t s, bool pdl);
// ctx = d_pos ? d_pos[0] + 1 : ctx_host
// kv_dtype: 0 fp32, 2 fp16
cudaError_t launch_attn(int kv_dtype, int nq, int nkv, int hd, int nsplit, int chunk_min,
                        size_t smem, const float* q, const void* kc, const void* vc,
                        int kv_stride, const int* d_pos, int ctx_host, float* out, void* ws,
                        unsigned long long* tl, cudaStream_t s, bool pdl, int merge = 1);
// x += Wo . o with o merged from the attention partials in ws (attention run with merge 0);
// mlp (may be null): the layer whose MLP weights may be requested into L2 ahead of use
cudaError_t launch_oproj(const Dims& d, const void* W, const float* part, const int* d_pos, float* y, int* err,
                         unsigned long long* tl, cudaStream_t s, bool pdl, const LayerPtrs* mlp = nullptr);
// y[r] += W[r,:] . in  (r < N), W [N, K]
cudaError_t launch_resid(const Dims& d, const void* W, int N, int K, const float* in, float* y,
                         int* err, unsigned long long* tl, cudaStream_t s, bool pdl);
cudaError_t launch_gateup(const Dims& d, const LayerPtrs& w, const float* x, float* act, int* err,
                          unsigned long long* tl, cudaStream_t s, bool pdl);
cudaError_t launch_lmhead(const Dims& d, const void* W, const void* final_norm, const float* x,
                          float* logits, const Finalize& f, unsigned long long* tl, cudaStream_t s,
                          bool pdl);

// ---- attn_tc.cu (causal prefill attention on tcgen05 / TMEM) ----
bool attn_prefill_tc_supported(int hd);
cudaError_t attn_prefill_tc_set_attributes();
// Qh [T][nq*hd] fp16 holding q * log2(e) / sqrt(hd) for positions pos0 .. pos0+T-1; kc, vc: the
// layer's fp16 cache [nkv][cap][hd], filled through position pos0+T-1; Oh [T][nq*hd] fp16.
cudaError_t attn_prefill_tc(const Dims& d, int T, int pos0, const __half* Qh, const __half* kc, const __half* vc,
                            __half* Oh, int* err, cudaStream_t s);

// ---- gemm_tc.cu (tcgen05 tensor-core GEMMs, bf16 in, fp32 accumulate) ----
bool gemm_tc_available();
// Tensor map (128-byte CUtensorMap) of a 2-D fp16 (bf16 when bf) row-major [rows][cols] array with
// a row pitch of ld elements, box of 64 columns x box_rows rows, 128-byte swizzle; false if the
// encoder is unavailable or the arguments break its rules.
bool make_map(void* map, const void* base, int rows, int cols, int ld, int box_rows, bool bf = false);
// Tensor map of one layer's fp16 K or V cache [nkv][cap][hd] over its first `keys` positions:
// boxes of 64 head columns x box_keys positions of one KV head, 128-byte swizzle.
bool make_map_kv(void* map, const void* base, int hd, int keys, int nkv, int cap, int box_keys);
cudaError_t gemm_tc_set_attributes();
// whether the prefill's tensor-core path launches its kernels with programmatic dependent
// launch (QW_PREFILL_PDL=0 turns it off)
bool tc_pdl();
// fp16 operands (A activations, B weights), fp32 accumulate; bias bf16
// ws (optional): fp32 workspace of ws_floats for split-K partial tiles, used when the
// output has too few 128x256 tiles for nsm SMs
// pdl: programmatic dependent launch after the previous kernel of the stream; the kernels then
// request B (which no kernel of the stream may be writing: weights) before that kernel ends
cudaError_t gemm_tc(const __half* A, int lda, const __half* B, int ldb, const __nv_bfloat16* bias,
                    float* C, int ldc, int M, int N, int K, bool accumulate, int* err,
                    cudaStream_t s, float* ws = nullptr, size_t ws_floats = 0, int nsm = 0, bool pdl = false);
// Outputs of the fused q/k/v projection (columns q | k | v, each head's columns in RoPE-pair
// order as the weights' rows are): + bias, rotation of q and k rows m at position pos0 + m,
// q times qscale to Qh [M][nq*hd] (fp16), k and v to the layer's fp16 caches [nkv][cap][hd]
// at positions pos0 .. pos0 + M - 1 (fp16 range errors set ERR_RANGE).
struct QkvOut {
  __half* Qh;
  __half *kc, *vc;
  const float2* rope;  // (cos, sin) [position][hd/2]
  float qscale;
  int nq, nkv, hd, pos0, cap;
};
cudaError_t gemm_tc_qkv(const __half* A, int lda, const __half* B, int ldb, const __nv_bfloat16* bias, int M, int N,
                        int K, const QkvOut& o, int* err, cudaStream_t s, float* ws = nullptr, size_t ws_floats = 0,
                        int nsm = 0, bool pdl = false);
cudaError_t gemm_tc_swiglu(const __half* A, int lda, const __half* Wg, const __half* Wu, int ldb,
                           __half* Act, int ldc, int M, int N, int K, int* err, cudaStream_t s, float* ws = nullptr,
                           size_t ws_floats = 0, int nsm = 0, bool pdl = false);

// ---- megastep.cu (one persistent kernel per decode step of one sequence, bf16 models) ----
struct MegaLaunch {
  Dims d;
  const void* layers_dev;          // device array of n_layers megastep layer records
  const void *embed, *final_norm, *head;
  const float2* rope;
  void* kv_seq;                    // fp16 cache of the sequence [L][2][nkv][cap][hd]
  float *q, *logits;
  float* work;                     // megastep_work_floats: copies of x, the activation, partials
  int *tok, *pos;
  unsigned long long* key;
  int *hist, *hist_n;
  int hist_cap;
  unsigned long long *bar, *bar_base;  // grid-barrier counter and its value at the step start
  int *abort, *err;
  unsigned long long* tl;          // per phase [start, units done, end], then per phase [input
                                   // staged, barrier passed, last arrival], or null
  int grid;
  int pf_mode;                     // when the MLP rows are requested into L2 (0 never, 1 at the
                                   // attention phase, 2 at the o_proj phase, 3 by the producers)
};
bool megastep_supported(const Dims& d, int nsm);
size_t megastep_smem(const Dims& d);
size_t megastep_work_floats(const Dims& d);
cudaError_t megastep_set_attributes(const Dims& d);
int megastep_threads();
cudaError_t megastep_occupancy(const Dims& d, int* per_sm);  // resident CTAs per SM
size_t megastep_layer_bytes();
void megastep_fill_layer(void* dst, const LayerPtrs& w);
cudaError_t launch_megastep(const MegaLaunch& a, cudaStream_t s);

// ---- gemm_tc.cu: skinny GEMM of batched decode ----
// Precomputed tensor maps (opaque 128-byte CUtensorMap storage) and the launch shape of one
// skinny GEMM: nz weight matrices against the 16 activation rows of the sequences.
struct SkinnyPlan {
  alignas(64) unsigned char wmap[3][128];
  alignas(64) unsigned char xmap[128];
  int nz, K, tiles, splits, n_total;
  int tile_start[3], rows[3], col_off[3];
  bool lm;   // bf16 operands, one split, logits + argmax epilogue
  bool glu;  // gate/up with SwiGLU into fp16 activation rows (one split)
};
cudaError_t skinny_set_attributes();
bool skinny_plan(SkinnyPlan* p, int nz, const void* const* W, const int* rows, const void* X, int K, bool bf,
                 int nsm);
cudaError_t skinny_run(const SkinnyPlan& p, float* part, float* logits, int V, int nseq, const int* active,
                       unsigned long long* keys, int* err, unsigned long long* tl, cudaStream_t s,
                       __half* act = nullptr);
bool skinny_plan_glu(SkinnyPlan* p, const void* Wg, const void* Wu, int I, const void* X, int K, int nsm);

// ---- batched.cu ----
struct BatchedLayerPlans {
  SkinnyPlan qkv, o, gu, down;
};
// Everything one batched decode step touches (device pointers; plans built at setup).
struct BatchedCtx {
  Dims d;
  const LayerPtrs* layers;          // host array [L]
  const BatchedLayerPlans* plans;   // host array [L]
  SkinnyPlan lm;
  const void *embed, *final_norm;
  const float2* rope;
  void* kv;                         // fp16 caches of all sequences
  size_t kv_seq_elems;              // elements per sequence
  float *x, *q, *part, *logits;     // x [S][H], q [16][nq*hd], partials, logits [S][V]
  __half *X16, *O16, *A16;          // fp16 activation rows [16][H], [16][nq*hd], [16][I]
  __nv_bfloat16* Xb16;              // bf16 rows of the LM head [16][H]
  int *tok, *pos, *hist, *hist_n, *err;
  const int* active;                // [S]
  unsigned long long* keys;         // [S]
  void* attn_ws;                    // attn_batched_workspace_bytes(.., S)
  size_t attn_smem;
  int attn_nsplit;                  // context chunks per sequence and KV head
  int attn_chunk;                   // fewest positions per chunk
  bool attn_mma;                    // tensor-core attention (else CUDA cores)
  unsigned long long* tl;           // timeline: 3 slots per launch, or null
};
cudaError_t batched_set_attributes();
bool batched_pdl();
constexpr int SKINNY_MAX_SPLITS = 16;  // split-K partials one consumer thread sums
cudaError_t batched_step(const BatchedCtx& c, cudaStream_t s);

// ---- prefill.cu ----
struct PrefillBufs {
  float *X, *Xn, *Y, *Q, *O, *G, *U;  // [T][..] fp32 activations
  __half *Xh, *Oh, *Ah;               // fp16 tensor-core operands [T][H], [T][nq*hd], [T][I]
  float* ws;                          // split-K partial tiles of the tensor-core GEMMs
  size_t ws_floats;
  int cap_tokens;
  bool use_tc;
};
cudaError_t prefill_set_attributes(const Dims& d);
// Runs all layers over T tokens at positions pos0..pos0+T-1 of one sequence.
cudaError_t prefill_layers(const Dims& d, const LayerPtrs* layers, const void* embed,
                           const int* ids_dev, int T, int pos0, const float2* rope,
                           void* kcache_seq, const PrefillBufs& b, int* err, cudaStream_t s);
cudaError_t convert_bf16_to_half(const void* src, void* dst, size_t n, int* err, cudaStream_t s);
// fp16 copy of a matrix of whole heads with each head's rows in RoPE-pair order (row 2i + e
// of a head = source row i + e hd/2), and a bf16 bias vector into the same order
cudaError_t convert_bf16_to_half_pairs(const void* src, void* dst, size_t rows, int K, int hd, int* err,
                                       cudaStream_t s);
cudaError_t copy_bias_pairs(const void* src, void* dst, int n, int hd, cudaStream_t s);

}  // namespace qw
