/*
 * qw.h - C ABI of libqw, a GB300 (sm_103a) implementation of the forward pass of a
 * Qwen2-style decoder-only transformer: prompt prefill into a preallocated KV cache and
 * KV-cached greedy decode.
 *
 * The operations follow these pages (cited by title and section):
 *   [LSA] "LLM Speedrun: Architecture": Transformer architecture (attention, causal mask,
 *         SwiGLU FFN, pre-norm residual stacking, GQA, RoPE, Decoding / LM head / KV
 *         cache) and Implementing Qwen (q/k/v bias, split-half RoPE, the model code's
 *         Decoder.step and generate_tokens).
 *   [AUG] "augur": Features (prefill/decode split, preallocated KV cache, greedy
 *         generation, EOS stopping).
 *   [QIE] "Building a Qwen2.5-1.5B Inference Engine From Scratch": §1 (prefill is
 *         compute-bound, decode is memory-bandwidth-bound).
 *
 * Conventions for every call:
 *   - Every call returns a qw_status; nothing aborts and nothing throws across the ABI.
 *     qw_last_error() gives a message for the last failing call on the calling thread.
 *   - "device" pointers are CUDA global-memory addresses on the device that was current
 *     when qw_create ran; "host" pointers are ordinary CPU memory.
 *   - Weights are BORROWED: the caller owns them, keeps them alive and unchanged until
 *     qw_destroy, and the library never writes them.
 *   - The library OWNS the KV cache, activations, logits, the RoPE table and the CUDA
 *     graph of a decode step; all are released by qw_destroy.
 *   - Work runs on the stream given to qw_create (or a stream the library creates when
 *     that argument is NULL). Calls that return host values synchronise that stream
 *     before returning.
 *   - After QW_ERR_CUDA or QW_ERR_TIMEOUT the model must be destroyed.
 */
#ifndef QW_H
#define QW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QW_OK = 0,
  QW_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent config */
  QW_ERR_UNSUPPORTED = 2,   /* a shape the library has no kernel for */
  QW_ERR_CAPACITY = 3,      /* a sequence would exceed kv_capacity */
  QW_ERR_TOKEN_RANGE = 4,   /* a token id outside [0, vocab) */
  QW_ERR_CUDA = 5,          /* a CUDA runtime call failed; destroy the model */
  QW_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up; destroy the model */
  QW_ERR_FAULT_INJECTED = 7,/* QW_FAULT environment variable forced a failure */
  QW_ERR_NUMERIC = 8        /* non-finite logits, or a value outside the fp16 range of the
                               KV cache (QW_BF16 models) or of a tensor-core operand */
} qw_status;

typedef enum { QW_F32 = 0, QW_BF16 = 1, QW_F16 = 2 } qw_dtype;

/* Model shape [LSA Implementing Qwen, the model configuration; AUG Qwen model config].
 * head_dim must be even and equal hidden / n_heads (the score scale 1/sqrt(d_k) uses
 * d_k = hidden / n_heads); n_heads must be a multiple of n_kv_heads. dtype is the storage
 * type of the weights, QW_F32 or QW_BF16. The KV cache is fp32 for QW_F32 models and fp16
 * for QW_BF16 models (same two bytes as bf16, eight times finer rounding); decode
 * activations, accumulators and logits are fp32; the prefill projections of QW_BF16 models
 * run on the tensor cores with fp16 operands (fp16 copies of the weights made by qw_create:
 * exact for 2^-17 <= |w| <= 65504, smaller weights round to a multiple of 2^-24, larger ones
 * are rejected) and fp32 accumulation. A key, value or operand that would overflow fp16 is
 * reported as QW_ERR_NUMERIC by the next call that checks device errors. */
typedef struct {
  int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, intermediate, vocab;
  float rms_eps;          /* RMSNorm epsilon, inside the square root (1e-6) */
  float rope_theta;       /* RoPE base (1e6) */
  int32_t tied_embeddings;/* 1: LM head is the embedding matrix */
  int32_t qkv_bias;       /* 1: q/k/v projections carry a bias [LSA Introducing bias] */
  int32_t dtype;          /* qw_dtype */
  int32_t max_seqs;       /* independent sequences held at once (1..16) */
  int32_t kv_capacity;    /* positions per sequence in the preallocated KV cache */
} qw_config;

/* Device pointers of one decoder layer, row-major [out, in], in qw_config.dtype.
 * Sizes: in_norm, post_norm [hidden]; wq [n_heads*head_dim, hidden]; wk, wv
 * [n_kv_heads*head_dim, hidden]; bq/bk/bv the matching vectors (NULL when qkv_bias is 0);
 * wo [hidden, n_heads*head_dim]; w_gate, w_up [intermediate, hidden];
 * w_down [hidden, intermediate]. Every pointer must be 16-byte aligned. */
typedef struct {
  const void *in_norm, *wq, *bq, *wk, *bk, *wv, *bv, *wo, *post_norm, *w_gate, *w_up,
      *w_down;
} qw_layer_weights;

/* embed [vocab, hidden]; final_norm [hidden]; lm_head [vocab, hidden] or NULL when tied;
 * layers is a HOST array of n_layers entries (copied by qw_create). */
typedef struct {
  const void *embed, *final_norm, *lm_head;
  const qw_layer_weights *layers;
} qw_weights;

typedef struct qw_model qw_model;

/* Build a model from its configuration and borrowed weights [LSA Implementing Qwen: the
 * model configuration and the Decoder that holds the embedding, the layers, the final
 * norm and the LM head; AUG Features: preallocated KV cache]. Validates the shape,
 * allocates the KV cache [max_seqs][n_layers][2][n_kv_heads][kv_capacity][head_dim] and
 * the working buffers, and builds the RoPE cos/sin table [LSA RoPE: angle = position *
 * theta^(-2i/head_dim)] with float64 angles on the host. cuda_stream is a cudaStream_t or
 * NULL. On success *out holds the model (release it with qw_destroy); on failure *out is
 * NULL and nothing stays allocated. Errors: QW_ERR_INVALID_ARG for a null, misaligned or
 * inconsistent argument, QW_ERR_UNSUPPORTED for a shape without kernels, QW_ERR_CUDA when
 * no GPU is usable or an allocation fails, QW_ERR_FAULT_INJECTED under QW_FAULT=alloc. */
qw_status qw_create(const qw_config *cfg, const qw_weights *w, void *cuda_stream,
                    qw_model **out);
void qw_destroy(qw_model *m);

/* Prefill [AUG Prefill/decode split; LSA Decoder.step on the whole prompt]: reset
 * sequence `seq`, run the n prompt tokens (host array) at positions 0..n-1, fill their
 * keys and values into the cache and compute the logits of the last position and its
 * greedy token. Afterwards the sequence holds n positions and its next decode step feeds
 * that token. next_token (host, may be NULL) receives it. Errors: QW_ERR_CAPACITY when
 * n > kv_capacity, QW_ERR_TOKEN_RANGE for an id outside [0, vocab). */
qw_status qw_prefill(qw_model *m, int32_t seq, const int32_t *ids, int32_t n,
                     int32_t *next_token);

/* The same with the prompt already in device memory; nothing is copied back and the
 * stream is not synchronised (token ids are range-checked on the device, reported by
 * qw_sync). */
qw_status qw_prefill_device(qw_model *m, int32_t seq, const int32_t *ids_dev, int32_t n);

/* One greedy decode step [LSA Decoding / KV cache; AUG greedy generation] for every
 * sequence that has been prefilled: run one token at position pos (the sequence's current
 * length), append its key and value at pos, compute the logits and the argmax, and
 * advance the length by one. feed (host [max_seqs], may be NULL) overrides the token run
 * for each sequence (teacher forcing); NULL runs each sequence's previous greedy token.
 * next_tokens (host [max_seqs], may be NULL) receives the new tokens; when it is NULL the
 * call does not synchronise. Errors: QW_ERR_CAPACITY when a sequence is full. */
qw_status qw_decode_step(qw_model *m, const int32_t *feed, int32_t *next_tokens);

/* n_steps decode steps of every active sequence, each feeding its own greedy token, with
 * no host synchronisation. Tokens are kept on the device (qw_tokens_device). */
qw_status qw_decode_steps(qw_model *m, int32_t n_steps);

/* Greedy generation of one sequence (seq 0) [AUG EOS stopping; LSA generate_tokens]:
 * prefill the n prompt ids (host), then decode until max_new tokens exist in total (the
 * prefill's token counts) or a token equal to eos (eos < 0: never) has been produced; that
 * token is kept. out (host [max_new]) receives the tokens, n_out their number. */
qw_status qw_generate(qw_model *m, const int32_t *ids, int32_t n, int32_t max_new,
                      int32_t eos, int32_t *out, int32_t *n_out);

/* The same with a set of stop ids [LSA Implementing Qwen: generate_tokens stops on any id of
 * its eos_ids set, the chat template's end tokens among them]: generation stops after the
 * first produced token that equals any of stop_ids[0 .. n_stop-1] (host array, may hold
 * duplicates; n_stop = 0: no stop id). That token is kept, and the sequence continues
 * from it as after qw_generate. Errors: QW_ERR_INVALID_ARG for n_stop < 0 or a null
 * stop_ids with n_stop > 0, and those of qw_generate. */
qw_status qw_generate_stops(qw_model *m, const int32_t *ids, int32_t n, int32_t max_new,
                            const int32_t *stop_ids, int32_t n_stop, int32_t *out,
                            int32_t *n_out);

/* Wait for queued work and report a device-side error (token range, non-finite logits). */
qw_status qw_sync(qw_model *m);

/* Device pointer to the fp32 logits [max_seqs][vocab] of the last step [LSA Decoding and
 * Decoder.step: the logits of the last position, LM head applied to the final norm];
 * row seq holds sequence seq's. Owned by the model; valid until the next call that runs
 * it. NULL for a null model. */
const float *qw_logits(const qw_model *m);

/* Copy the fp32 logits [vocab] of sequence seq's last step to host memory (synchronises). */
qw_status qw_read_logits(qw_model *m, int32_t seq, float *host_out);

/* Device pointer to int32 [max_seqs]: the greedy token of each sequence's last step. */
const int32_t *qw_tokens_device(const qw_model *m);

/* Current length of sequence seq: the positions its KV cache holds, which is also the
 * position the next decode step runs at [LSA Decoder.step: positions of the new token;
 * KV cache]. 0 for a sequence that is not active. Errors: QW_ERR_INVALID_ARG. */
qw_status qw_position(const qw_model *m, int32_t seq, int32_t *pos);

/* Kernel launches one single-sequence decode step makes: 1 when the step runs as one
 * persistent kernel (bf16 models whose shape it supports, the default), else
 * n_layers * 5 + 2 (embedding, q/k/v, attention, o_proj, gate/up, down per layer, LM head).
 * 0 for a null model. */
int32_t qw_decode_kernels_per_step(const qw_model *m);

/* Forget sequence seq [LSA KVCache: a fresh cache per sequence; AUG Features:
 * preallocated KV cache]: its length becomes 0 and it leaves the set of active sequences;
 * its cache rows are overwritten by its next prefill. Does not synchronise. Errors:
 * QW_ERR_INVALID_ARG for a null model or a sequence index outside [0, max_seqs). */
qw_status qw_reset(qw_model *m, int32_t seq);

/* Profiling hook. With begin and end non-NULL (host arrays of n_layers cudaEvent_t created
 * with timing enabled), every later decode step records begin[l] just before and end[l]
 * just after kernel `kind` of layer l: 0 qkv, 1 attention, 2 o_proj, 3 gate/up, 4 down;
 * kind 5 is the LM head (begin[0], end[0] only). The traced kernel and the one after it
 * then launch without programmatic dependent launch. NULL arrays remove the hook. The
 * decode graphs are rebuilt on the next step. */
qw_status qw_set_trace(qw_model *m, int32_t kind, void *const *begin, void *const *end);

/* Device timeline (profiling). With enable 1, every later decode step records, for each of
 * its kernel launches (embedding, then per layer qkv, attention, o_proj, gate/up, down, then
 * the LM head), three %globaltimer stamps in ns: the first CTA's start, the first CTA past
 * its wait for the previous kernel, and the last CTA's end. qw_read_timeline copies the
 * stamps of the last step, 3 per launch in launch order, into out (host, 3 * max_launches
 * uint64) and the launch count into n_launches. Timing differs slightly from an
 * uninstrumented run (one atomic per CTA per stamp). enable 0 frees the buffer.
 * When a single-sequence step runs as one persistent kernel (qw_decode_kernels_per_step
 * is 1), entry k < 5 * n_layers + 1 is phase k of the step instead (q/k/v, attention,
 * o_proj, gate/up, down per layer, then the LM head): [start after the previous grid
 * barrier, its weight units consumed, end before the next grid barrier], stamped by the
 * first CTA. */
qw_status qw_set_timeline(qw_model *m, int32_t enable);
qw_status qw_read_timeline(qw_model *m, uint64_t *out, int32_t max_launches, int32_t *n_launches);

/* Message for the last failing call on this thread ("" if none). */
const char *qw_last_error(void);

/* ---- single operations, for testing a step of the path in isolation ---- */

/* GQA decode attention of one token [LSA Attention, Causal mask, GQA]: for every query
 * head h, scores s_j = q_h . K_j / sqrt(head_dim) over positions j = 0..ctx-1 of KV head
 * h / (n_heads / n_kv_heads), softmax, and out_h = sum_j p_j V_j. The context is split
 * into chunks whose partial softmax statistics are merged exactly (log-sum-exp).
 *   q    device fp32 [n_heads*head_dim]
 *   k, v device, kv_dtype (QW_F32 or QW_F16) elements, [n_kv_heads][kv_stride][head_dim]
 *        (position-major per head), ctx <= kv_stride
 *   out  device fp32 [n_heads*head_dim]
 *   workspace device, at least qw_op_decode_attention_workspace() bytes, 16-byte
 *        aligned; its counters must be zero before the first call (cudaMemset) and the
 *        call leaves them zero again.
 * Shapes: head_dim a multiple of 8, at most 8 query heads per KV head and
 * (n_heads / n_kv_heads) * head_dim <= 1024; others return QW_ERR_UNSUPPORTED.
 * Runs on cuda_stream (NULL = default stream) and does not synchronise. */
size_t qw_op_decode_attention_workspace(int32_t n_heads, int32_t n_kv_heads,
                                        int32_t head_dim, int32_t max_ctx);
qw_status qw_op_decode_attention(int32_t kv_dtype, int32_t n_heads, int32_t n_kv_heads,
                                 int32_t head_dim, int32_t ctx, int32_t kv_stride,
                                 const float *q, const void *k, const void *v, float *out,
                                 void *workspace, size_t workspace_bytes,
                                 void *cuda_stream);

/* Decode attention for callers that cannot allocate device memory. The pages have no
 * counterpart: this is a deployment variant of qw_op_decode_attention, computing the same
 * result (same kernel) with its scratch (the split-context partials and the per-KV-head
 * counters) in one fixed 1 MiB array inside the library instead of a caller workspace.
 * It is meant for callers that cannot call cudaMalloc where they call attention: code
 * embedded in another runtime that owns all device memory, or loops that must not pay
 * cudaMalloc's implicit device synchronisation or risk an allocation failure mid-run.
 *   - Arguments, layouts and errors are those of qw_op_decode_attention, without the
 *     workspace. Shapes whose scratch exceeds qw_op_decode_attention_noalloc_limit()
 *     bytes are rejected with QW_ERR_UNSUPPORTED (1 MiB fits, for example, 12 query /
 *     2 KV heads of dimension 128 with kv_stride up to 8192).
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library routine. Every
 *     GPU that loads the library holds the array until the process exits.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current); make that first call before any stream capture. A first
 *     call on a stream that is capturing returns QW_ERR_INVALID_ARG and does nothing.
 *   - Each call clears the counters it needs (cudaMemsetAsync on cuda_stream). All calls
 *     share the one array: calls that overlap on the GPU (other streams, other threads)
 *     race on it and must be serialised by the caller. */
qw_status qw_op_decode_attention_noalloc(int32_t kv_dtype, int32_t n_heads, int32_t n_kv_heads,
                                         int32_t head_dim, int32_t ctx, int32_t kv_stride,
                                         const float *q, const void *k, const void *v,
                                         float *out, void *cuda_stream);
size_t qw_op_decode_attention_noalloc_limit(void);

/* Dense GEMM on the tensor cores (tcgen05), the contraction of every prefill projection
 * [LSA Implementing Qwen: W @ x for all prompt columns at once; QIE §1: prefill is
 * compute-bound]: C[M][N] = A[M][K] . B[N][K]^T (+ bias[N]), or C += A . B^T when
 * accumulate is 1 (the residual add). A, B fp16 row-major, bias bf16 (may be NULL), C fp32
 * row-major, all device, contiguous (row pitch = K for A and B, N for C), 16-byte aligned;
 * K and N multiples of 8. err_dev is a device int32 that receives QW device error bits (a
 * bounded wait that expired). Runs on cuda_stream without synchronising. */
qw_status qw_op_gemm_f16(int32_t M, int32_t N, int32_t K, const void *A, const void *B,
                          const void *bias, float *C, int32_t accumulate, int32_t *err_dev,
                          void *cuda_stream);

/* Fused gate/up projection and SwiGLU [LSA SwiGLU FFN]: act[M][N] =
 * silu(A . Wg^T) * (A . Wu^T), A [M][K], Wg/Wu [N][K] fp16, act fp16 [M][N]; the same
 * layout rules as qw_op_gemm_f16. */
qw_status qw_op_gemm_swiglu_f16(int32_t M, int32_t N, int32_t K, const void *A,
                                 const void *Wg, const void *Wu, void *act, int32_t *err_dev,
                                 void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* QW_H */
