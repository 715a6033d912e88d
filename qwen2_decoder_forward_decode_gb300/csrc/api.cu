// libqw C ABI: model creation, prefill, KV-cached greedy decode, generation.
//
// The model keeps all state on the device: the KV cache of every sequence, each
// sequence's length and next token, the argmax key and a token history. A decode step of
// one sequence is one CUDA graph (embedding, n_layers x {qkv, attn, o_proj, gate/up,
// down}, LM head) captured on first use with programmatic-dependent-launch edges; because
// positions and tokens live in device memory the same graph serves every step.
#include "../../include/qw.h"
#include "common.cuh"
#include "internal.h"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

using namespace qw;

namespace {

thread_local std::string g_err;

qw_status fail(qw_status s, const std::string& msg) {
  g_err = msg;
  return s;
}

qw_status cuda_fail(cudaError_t e, const char* where) {
  return fail(QW_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

#define QW_CUDA(call)                                  \
  do {                                                 \
    cudaError_t e_ = (call);                           \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

bool fault_injected(const char* what) {
  const char* f = std::getenv("QW_FAULT");
  return f && std::strcmp(f, what) == 0;
}

constexpr int ATTN_CHUNK_MIN = 32;

}  // namespace

void qw::set_error_message(const char* msg) { g_err = msg; }

struct qw_model {
  Dims d;
  qw_config cfg;
  std::vector<LayerPtrs> layers;
  const void *embed = nullptr, *final_norm = nullptr, *lm_head = nullptr;
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  int device = 0;
  size_t esize = 4;
  // device state
  void* kv = nullptr;
  float *x = nullptr, *q = nullptr, *attn = nullptr, *act = nullptr, *logits = nullptr;
  float2* rope = nullptr;
  void* attn_ws = nullptr;
  size_t attn_smem = 0;
  unsigned long long* keys = nullptr;
  unsigned int* lm_counter = nullptr;
  int *pos = nullptr, *tok = nullptr, *hist = nullptr, *hist_n = nullptr, *err = nullptr;
  int* ids = nullptr;
  int* pinned = nullptr;  // host staging, max(cap, max_seqs) ints
  PrefillBufs pf{};
  void* pf_block = nullptr;
  void* pf_ws = nullptr;  // split-K workspace of the prefill GEMMs
  void* w16 = nullptr;  // fp16 copies of the layer matrices (bf16 models)
  // host mirror
  std::vector<int> h_pos;
  std::vector<char> active;
  std::vector<cudaGraphExec_t> graphs;
  bool use_graphs = true;
  bool merge_in_oproj = false;  // decode attention leaves its partials to the o_proj GEMV
  bool attn_mma = false;        // decode attention on the tensor cores (fp16 cache)
  int trace_kind = -1;
  std::vector<cudaEvent_t> trace_begin, trace_end;
  // one persistent kernel per decode step of one sequence (bf16 models)
  bool use_mega = false;
  void* mega_layers = nullptr;       // device layer records
  float* mega_part = nullptr;        // copies of the residual, the activation and the attention partials
  unsigned long long* mega_bar = nullptr;  // [0] barrier counter, [1] its value at a step start
  int* mega_abort = nullptr;
  // batched decode (bf16 models with the fp16 matrix copies, several sequences)
  bool use_batched = false;
  std::vector<BatchedLayerPlans> bplans;
  SkinnyPlan blm{};
  void* bblock = nullptr;          // one allocation for the buffers below
  float *bq = nullptr, *bpart = nullptr;
  __half *bX16 = nullptr, *bO16 = nullptr, *bA16 = nullptr;
  __nv_bfloat16* bXb16 = nullptr;
  void* battn_ws = nullptr;
  int battn_nsplit = 0;            // context chunks of the batched attention
  int battn_chunk = 0;             // fewest positions per chunk
  bool battn_mma = false;          // tensor-core batched attention
  size_t battn_smem = 0;
  int* bactive = nullptr;          // device copy of the active flags
  bool bactive_dirty = true;
  cudaGraphExec_t bgraph = nullptr;
  unsigned long long* tl_buf = nullptr;  // device timeline of one decode step (or null)
  int tl_n = 0;                          // launches per decode step
  std::vector<unsigned long long> tl_init;

  size_t seq_kv_elems() const { return (size_t)d.L * 2 * d.nkv * d.cap * d.hd; }
  char* kv_seq(int s) const { return (char*)kv + (size_t)s * seq_kv_elems() * esize; }
  char* kc_layer(int s, int l) const {
    return kv_seq(s) + (size_t)l * 2 * d.nkv * d.cap * d.hd * esize;
  }
  char* vc_layer(int s, int l) const {
    return kc_layer(s, l) + (size_t)d.nkv * d.cap * d.hd * esize;
  }
  const void* head_w() const { return lm_head ? lm_head : embed; }

  Finalize fin(int s, int pos_set) const {
    Finalize f;
    f.key = keys + s;
    f.counter = lm_counter + s;
    f.tok = tok + s;
    f.pos = pos + s;
    f.pos_set = pos_set;
    f.hist = hist + (size_t)s * d.cap;
    f.hist_n = hist_n + s;
    f.hist_cap = d.cap;
    f.err = err;
    return f;
  }

  // Enqueue one decode step of sequence s (no host work besides launches).
  cudaError_t enqueue_decode(int s) {
    cudaError_t e;
    float* xs = x + (size_t)s * d.H;
    bool pdl = true;
    int launch_idx = 0;
    // timeline slots of launch i: [i] start, [n + i] past the wait, [2n + i] end
    auto tl = [&]() -> unsigned long long* { return tl_buf ? tl_buf + 3 * (launch_idx++) : nullptr; };
    // launch k-th kernel of layer l, with the optional trace events around it
    auto run = [&](int kind, int l, auto&& launch) -> cudaError_t {
      const bool traced = kind == trace_kind;
      cudaError_t r;
      if (traced && (r = cudaEventRecordWithFlags(trace_begin[l], stream, cudaEventRecordExternal)))
        return r;
      if ((r = launch(pdl && !traced))) return r;
      pdl = true;
      if (traced) {
        if ((r = cudaEventRecordWithFlags(trace_end[l], stream, cudaEventRecordExternal))) return r;
        pdl = false;
      }
      return cudaSuccess;
    };
    if ((e = launch_embed(d, embed, tok + s, xs, err, tl(), stream, false))) return e;
    for (int l = 0; l < d.L; ++l) {
      const LayerPtrs& w = layers[l];
      void* kc = kc_layer(s, l);
      void* vc = vc_layer(s, l);
      if ((e = run(0, l, [&](bool p) { return launch_qkv(d, w, xs, pos + s, rope, q, kc, vc, err, tl(), stream, p); })))
        return e;
      if ((e = run(1, l, [&](bool p) {
             if (attn_mma)  // tensor cores; the o_proj GEMV merges the chunks
               return launch_attn_decode_mma(d.nq, d.nkv, d.hd, d.attn_nsplit, d.attn_chunk_min, q,
                                             (const __half*)kc, (const __half*)vc, 0, d.cap, pos + s, nullptr, 1,
                                             attn_ws, tl(), stream, p);
             return launch_attn(d.dtype == QW_BF16 ? 2 : 0, d.nq, d.nkv, d.hd, d.attn_nsplit, d.attn_chunk_min,
                                attn_smem, q, kc, vc, d.cap, pos + s, 0, attn, attn_ws, tl(), stream, p,
                                merge_in_oproj ? 0 : 1);
           })))
        return e;
      // the o_proj GEMV merges the attention partials into its input vector (up to 2048
      // attention outputs), else reads the output the attention kernel merged
      if ((e = run(2, l, [&](bool p) {
             return merge_in_oproj ? launch_oproj(d, w.wo, (const float*)attn_ws, pos + s, xs, err, tl(), stream, p, &w)
                                   : launch_resid(d, w.wo, d.H, d.nq * d.hd, attn, xs, err, tl(), stream, p);
           })))
        return e;
      if ((e = run(3, l, [&](bool p) { return launch_gateup(d, w, xs, act, err, tl(), stream, p); }))) return e;
      if ((e = run(4, l, [&](bool p) { return launch_resid(d, w.w_down, d.H, d.I, act, xs, err, tl(), stream, p); })))
        return e;
    }
    return run(5, 0, [&](bool p) {
      return launch_lmhead(d, head_w(), final_norm, xs, logits + (size_t)s * d.V, fin(s, -1), tl(), stream, p);
    });
  }

  void drop_graphs() {
    for (auto& g : graphs)
      if (g) { cudaGraphExecDestroy(g); g = nullptr; }
    if (bgraph) { cudaGraphExecDestroy(bgraph); bgraph = nullptr; }
  }

  cudaError_t run_mega(int s) {
    MegaLaunch a{};
    a.d = d;
    a.layers_dev = mega_layers;
    a.embed = embed;
    a.final_norm = final_norm;
    a.head = head_w();
    a.rope = rope;
    a.kv_seq = kv_seq(s);
    a.q = q;
    a.logits = logits + (size_t)s * d.V;
    a.work = mega_part;
    a.tok = tok + s;
    a.pos = pos + s;
    a.key = keys + s;
    a.hist = hist + (size_t)s * d.cap;
    a.hist_n = hist_n + s;
    a.hist_cap = d.cap;
    a.bar = mega_bar;
    a.bar_base = mega_bar + 1;
    a.abort = mega_abort;
    a.err = err;
    a.tl = tl_buf;
    a.grid = d.nsm;
    static const int pf = [] {
      const char* v = std::getenv("QW_MK_PF");
      return v ? std::atoi(v) : 0;
    }();
    a.pf_mode = pf;
    if (tl_buf) {  // atomicMax stamps start from zero
      cudaError_t e = cudaMemsetAsync(tl_buf, 0, sizeof(unsigned long long) * 3 * tl_n, stream);
      if (e) return e;
    }
    return launch_megastep(a, stream);
  }

  cudaError_t run_decode(int s) {
    if (use_mega && trace_kind < 0) return run_mega(s);
    if (tl_buf) {  // per launch: start and wait-release reduce with min, end with max
      cudaError_t e = cudaMemcpyAsync(tl_buf, tl_init.data(), sizeof(unsigned long long) * 3 * tl_n,
                                      cudaMemcpyHostToDevice, stream);
      if (e) return e;
    }
    if (!use_graphs) return enqueue_decode(s);
    if (!graphs[s]) {
      cudaGraph_t g = nullptr;
      cudaError_t e = cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal);
      if (e) return e;
      e = enqueue_decode(s);
      cudaError_t e2 = cudaStreamEndCapture(stream, &g);
      if (e) { if (g) cudaGraphDestroy(g); return e; }
      if (e2) return e2;
      e = cudaGraphInstantiate(&graphs[s], g, 0);
      cudaGraphDestroy(g);
      if (e) { graphs[s] = nullptr; return e; }
    }
    return cudaGraphLaunch(graphs[s], stream);
  }

  int n_active() const {
    int n = 0;
    for (char a : active) n += a != 0;
    return n;
  }

  // One decode step of every active sequence with the weights read once (batched path).
  cudaError_t run_decode_batched() {
    cudaError_t e;
    if (bactive_dirty) {
      std::vector<int> h(d.max_seqs);
      for (int s = 0; s < d.max_seqs; ++s) h[s] = active[s] ? 1 : 0;
      if ((e = cudaMemcpyAsync(bactive, h.data(), sizeof(int) * d.max_seqs, cudaMemcpyHostToDevice, stream)))
        return e;
      if ((e = cudaStreamSynchronize(stream))) return e;  // h is a stack buffer
      bactive_dirty = false;
    }
    BatchedCtx c{};
    c.d = d;
    c.layers = layers.data();
    c.plans = bplans.data();
    c.lm = blm;
    c.embed = embed;
    c.final_norm = final_norm;
    c.rope = rope;
    c.kv = kv;
    c.kv_seq_elems = seq_kv_elems();
    c.x = x;
    c.q = bq;
    c.part = bpart;
    c.logits = logits;
    c.X16 = bX16;
    c.O16 = bO16;
    c.A16 = bA16;
    c.Xb16 = bXb16;
    c.tok = tok;
    c.pos = pos;
    c.hist = hist;
    c.hist_n = hist_n;
    c.err = err;
    c.active = bactive;
    c.keys = keys;
    c.attn_ws = battn_ws;
    c.attn_smem = battn_smem;
    c.attn_nsplit = battn_nsplit;
    c.attn_chunk = battn_chunk;
    c.attn_mma = battn_mma;
    c.tl = tl_buf;
    if (tl_buf && (e = cudaMemcpyAsync(tl_buf, tl_init.data(), sizeof(unsigned long long) * 3 * tl_n,
                                       cudaMemcpyHostToDevice, stream)))
      return e;
    if (!use_graphs) return batched_step(c, stream);
    if (!bgraph) {
      cudaGraph_t g = nullptr;
      if ((e = cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal))) return e;
      e = batched_step(c, stream);
      cudaError_t e2 = cudaStreamEndCapture(stream, &g);
      if (e) { if (g) cudaGraphDestroy(g); return e; }
      if (e2) return e2;
      e = cudaGraphInstantiate(&bgraph, g, 0);
      cudaGraphDestroy(g);
      if (e) { bgraph = nullptr; return e; }
    }
    return cudaGraphLaunch(bgraph, stream);
  }

  // decode step of all active sequences: batched when two or more are active
  cudaError_t decode_all() {
    if (use_batched && n_active() >= 2) {
      cudaError_t e = run_decode_batched();
      if (e) return e;
      for (int s = 0; s < d.max_seqs; ++s)
        if (active[s]) h_pos[s] += 1;
      return cudaSuccess;
    }
    for (int s = 0; s < d.max_seqs; ++s) {
      if (!active[s]) continue;
      cudaError_t e = run_decode(s);
      if (e) return e;
      h_pos[s] += 1;
    }
    return cudaSuccess;
  }

  cudaError_t ensure_prefill(int T) {
    if (pf.cap_tokens >= T) return cudaSuccess;
    if (pf_block) { cudaFree(pf_block); pf_block = nullptr; }
    if (pf_ws) { cudaFree(pf_ws); pf_ws = nullptr; }
    {  // split-K partial tiles: 16 splits of a 512-token output at most (short prompts)
      const size_t n = std::max(16 * (size_t)std::min(T, 512) * std::max((size_t)d.nq * d.hd, (size_t)d.H),
                                4 * (size_t)std::min(T, 512) * 2 * d.I);  // gate|up partials
      cudaError_t e = cudaMalloc(&pf_ws, n * sizeof(float));
      if (e) { pf_ws = nullptr; pf.cap_tokens = 0; return e; }
      pf.ws = (float*)pf_ws;
      pf.ws_floats = n;
    }
    const size_t H = d.H, qd = (size_t)d.nq * d.hd, W = qd + 2 * (size_t)d.nkv * d.hd, I = d.I;
    const size_t per_tok = H * 2 + W + qd * 2 + I * 2;  // X Xn Y Q O G U (fp32)
    const size_t per_tok_h = H + qd + I;               // Xh Oh Ah (fp16)
    const size_t f32_bytes = (per_tok * T * sizeof(float) + 255) & ~(size_t)255;
    cudaError_t e = cudaMalloc(&pf_block, f32_bytes + per_tok_h * T * sizeof(__half) + 256);
    if (e) { pf_block = nullptr; pf.cap_tokens = 0; return e; }
    float* p = (float*)pf_block;
    pf.X = p; p += H * T;
    pf.Xn = p; p += H * T;
    pf.Y = p; p += W * T;
    pf.Q = p; p += qd * T;
    pf.O = p; p += qd * T;
    pf.G = p; p += I * T;
    pf.U = p;
    __half* h = (__half*)((char*)pf_block + f32_bytes);
    pf.Xh = h; h += H * T;
    pf.Oh = h; h += qd * T;
    pf.Ah = h;
    pf.cap_tokens = T;
    return cudaSuccess;
  }

  // prompt already in device memory at ids_dev
  cudaError_t enqueue_prefill(int s, const int* ids_dev, int n) {
    cudaError_t e;
    if ((e = ensure_prefill(n))) return e;
    if ((e = cudaMemsetAsync(hist_n + s, 0, sizeof(int), stream))) return e;
    if ((e = prefill_layers(d, layers.data(), embed, ids_dev, n, 0, rope, kv_seq(s), pf, err, stream)))
      return e;
    return launch_lmhead(d, head_w(), final_norm, pf.X + (size_t)(n - 1) * d.H,
                         logits + (size_t)s * d.V, fin(s, n), nullptr, stream, false);
  }

  qw_status check_device_errors() {
    int h = 0;
    QW_CUDA(cudaMemcpyAsync(&h, err, sizeof(int), cudaMemcpyDeviceToHost, stream));
    QW_CUDA(cudaStreamSynchronize(stream));
    if (h) {
      QW_CUDA(cudaMemsetAsync(err, 0, sizeof(int), stream));
      QW_CUDA(cudaStreamSynchronize(stream));
      if (h & ERR_TOKEN) return fail(QW_ERR_TOKEN_RANGE, "token id outside [0, vocab) on the device");
      if (h & ERR_NONFINITE) return fail(QW_ERR_NUMERIC, "non-finite logits");
      if (h & ERR_RANGE)
        return fail(QW_ERR_NUMERIC, "a value outside the fp16 range of the KV cache or of a tensor-core operand");
      if (h & ERR_TIMEOUT) return fail(QW_ERR_TIMEOUT, "a bounded device-side wait gave up");
      if (h & ERR_LAYOUT) return fail(QW_ERR_CUDA, "a kernel found its shared memory misaligned");
    }
    return QW_OK;
  }

  void release() {
    for (auto& g : graphs)
      if (g) cudaGraphExecDestroy(g);
    graphs.clear();
    if (bgraph) cudaGraphExecDestroy(bgraph);
    bgraph = nullptr;
    if (bblock) cudaFree(bblock);
    if (battn_ws) cudaFree(battn_ws);
    void* bufs[] = {kv, x, q, attn, act, logits, rope, attn_ws, keys, lm_counter, pos, tok,
                    hist, hist_n, err, ids, pf_block, pf_ws, w16, tl_buf, mega_layers, mega_part,
                    mega_bar, mega_abort};
    for (void* b : bufs)
      if (b) cudaFree(b);
    if (pinned) cudaFreeHost(pinned);
    if (own_stream && stream) cudaStreamDestroy(stream);
  }
};

static qw_status validate(const qw_config* c, const qw_weights* w) {
  if (!c || !w) return fail(QW_ERR_INVALID_ARG, "null config or weights");
  if (c->n_layers < 1 || c->hidden < 1 || c->n_heads < 1 || c->n_kv_heads < 1 ||
      c->head_dim < 2 || c->intermediate < 1 || c->vocab < 1 || c->kv_capacity < 1 ||
      c->max_seqs < 1)
    return fail(QW_ERR_INVALID_ARG, "non-positive dimension in config");
  if (c->max_seqs > 16) return fail(QW_ERR_UNSUPPORTED, "max_seqs above 16");
  if (c->head_dim % 2) return fail(QW_ERR_INVALID_ARG, "head_dim must be even");
  if (c->n_heads % c->n_kv_heads) return fail(QW_ERR_INVALID_ARG, "n_heads not a multiple of n_kv_heads");
  if (c->n_heads * c->head_dim != c->hidden)
    return fail(QW_ERR_UNSUPPORTED, "head_dim must equal hidden / n_heads");
  if (c->n_heads / c->n_kv_heads > 8) return fail(QW_ERR_UNSUPPORTED, "more than 8 query heads per KV head");
  if (c->dtype != QW_F32 && c->dtype != QW_BF16) return fail(QW_ERR_INVALID_ARG, "unknown dtype");
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return fail(QW_ERR_INVALID_ARG, "bad eps or theta");
  const int hd = c->head_dim;
  if (hd != 16 && hd != 32 && hd != 64 && hd != 128) return fail(QW_ERR_UNSUPPORTED, "head_dim must be 16, 32, 64 or 128");
  const int vec = c->dtype == QW_BF16 ? 8 : 4;
  if (c->hidden % vec || c->intermediate % vec)
    return fail(QW_ERR_UNSUPPORTED, "hidden and intermediate must be multiples of 16 bytes of weights");
  if (c->hidden > 8 * 32 * 12 * vec || c->intermediate > 8 * 32 * 12 * vec)
    return fail(QW_ERR_UNSUPPORTED, "hidden or intermediate too large for the decode GEMV");
  if (!w->embed || !w->final_norm || !w->layers) return fail(QW_ERR_INVALID_ARG, "null weight pointer");
  if (!c->tied_embeddings && !w->lm_head) return fail(QW_ERR_INVALID_ARG, "untied model without lm_head");
  for (int l = 0; l < c->n_layers; ++l) {
    const qw_layer_weights& L = w->layers[l];
    const void* req[] = {L.in_norm, L.wq, L.wk, L.wv, L.wo, L.post_norm, L.w_gate, L.w_up, L.w_down};
    for (const void* p : req) {
      if (!p) return fail(QW_ERR_INVALID_ARG, "null layer weight pointer");
      if ((uintptr_t)p % 16) return fail(QW_ERR_INVALID_ARG, "layer weight not 16-byte aligned");
    }
    if (c->qkv_bias && (!L.bq || !L.bk || !L.bv)) return fail(QW_ERR_INVALID_ARG, "qkv_bias set but a bias is null");
  }
  if ((uintptr_t)w->embed % 16) return fail(QW_ERR_INVALID_ARG, "embedding not 16-byte aligned");
  if (w->lm_head && (uintptr_t)w->lm_head % 16) return fail(QW_ERR_INVALID_ARG, "lm_head not 16-byte aligned");
  return QW_OK;
}

static int op_attn_nsplit(int head_dim, int max_ctx, int kv_bytes) {
  return attn_nsplit_for(max_ctx, ATTN_CHUNK_MIN, head_dim, kv_bytes);
}

// Workspace bytes that qw_op_decode_attention uses for this shape and KV element type; its
// per-KV-head counters are the last n_kv_heads * 4 bytes of that range.
size_t qw::op_attn_workspace_exact(int kv_dtype, int n_heads, int n_kv_heads, int head_dim, int kv_stride) {
  const int nsplit = op_attn_nsplit(head_dim, kv_stride, kv_dtype == QW_F16 ? 2 : 4);
  return attn_workspace_bytes(n_heads, n_kv_heads, head_dim, nsplit);
}

extern "C" {

const char* qw_last_error(void) { return g_err.c_str(); }

qw_status qw_create(const qw_config* cfg, const qw_weights* w, void* cuda_stream, qw_model** out) {
  g_err.clear();
  if (!out) return fail(QW_ERR_INVALID_ARG, "null output pointer");
  *out = nullptr;
  qw_status st = validate(cfg, w);
  if (st) return st;
  if (fault_injected("alloc")) return fail(QW_ERR_FAULT_INJECTED, "QW_FAULT=alloc");
  qw_model* m = new qw_model();
  m->cfg = *cfg;
  Dims& d = m->d;
  d.L = cfg->n_layers; d.H = cfg->hidden; d.nq = cfg->n_heads; d.nkv = cfg->n_kv_heads;
  d.hd = cfg->head_dim; d.I = cfg->intermediate; d.V = cfg->vocab;
  d.eps = cfg->rms_eps; d.theta = cfg->rope_theta; d.dtype = cfg->dtype;
  d.cap = cfg->kv_capacity; d.max_seqs = cfg->max_seqs;
  m->esize = cfg->dtype == QW_BF16 ? 2 : 4;
  auto bail = [&](cudaError_t e, const char* where) {
    m->release();
    delete m;
    return cuda_fail(e, where);
  };
  cudaError_t e;
  if ((e = cudaGetDevice(&m->device))) return bail(e, "cudaGetDevice");
  if ((e = cudaDeviceGetAttribute(&d.nsm, cudaDevAttrMultiProcessorCount, m->device)))
    return bail(e, "cudaDeviceGetAttribute");
  {  // shortest context chunk of decode attention (tuning knob QW_ATTN_CHUNK_MIN)
    const char* cm = std::getenv("QW_ATTN_CHUNK_MIN");
    const int c = cm ? std::atoi(cm) : 0;
    d.attn_chunk_min = c >= 8 && c <= 1024 ? c : ATTN_CHUNK_MIN;
  }
  d.attn_nsplit = attn_nsplit_for(d.cap, d.attn_chunk_min, d.hd, cfg->dtype == QW_BF16 ? 2 : 4);
  m->attn_smem = attn_smem_bytes(d.nq / d.nkv, d.hd, d.cap, d.attn_nsplit, d.attn_chunk_min,
                                 cfg->dtype == QW_BF16 ? 2 : 4);
  if (cuda_stream) {
    m->stream = (cudaStream_t)cuda_stream;
  } else {
    if ((e = cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking))) return bail(e, "cudaStreamCreate");
    m->own_stream = true;
  }
  m->embed = w->embed;
  m->final_norm = w->final_norm;
  m->lm_head = cfg->tied_embeddings ? nullptr : w->lm_head;
  for (int l = 0; l < d.L; ++l) {
    const qw_layer_weights& L = w->layers[l];
    LayerPtrs p{L.in_norm, L.wq, cfg->qkv_bias ? L.bq : nullptr, L.wk, cfg->qkv_bias ? L.bk : nullptr,
                L.wv, cfg->qkv_bias ? L.bv : nullptr, L.wo, L.post_norm, L.w_gate, L.w_up, L.w_down,
                nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    m->layers.push_back(p);
  }
  const int S = d.max_seqs;
  const size_t kv_bytes = (size_t)S * m->seq_kv_elems() * m->esize;
  if ((e = cudaMalloc(&m->kv, kv_bytes))) return bail(e, "cudaMalloc(kv cache)");
  if ((e = cudaMemset(m->kv, 0, kv_bytes))) return bail(e, "cudaMemset(kv cache)");
  if ((e = cudaMalloc(&m->x, sizeof(float) * S * d.H))) return bail(e, "cudaMalloc");
  if ((e = cudaMalloc(&m->q, sizeof(float) * d.nq * d.hd))) return bail(e, "cudaMalloc");
  if ((e = cudaMalloc(&m->attn, sizeof(float) * d.nq * d.hd))) return bail(e, "cudaMalloc");
  if ((e = cudaMalloc(&m->act, sizeof(float) * d.I))) return bail(e, "cudaMalloc");
  if ((e = cudaMalloc(&m->logits, sizeof(float) * S * (size_t)d.V))) return bail(e, "cudaMalloc");
  if ((e = cudaMemset(m->logits, 0, sizeof(float) * S * (size_t)d.V))) return bail(e, "cudaMemset");
  const size_t ws = attn_workspace_bytes(d.nq, d.nkv, d.hd, d.attn_nsplit);
  if ((e = cudaMalloc(&m->attn_ws, ws))) return bail(e, "cudaMalloc");
  if ((e = cudaMemset(m->attn_ws, 0, ws))) return bail(e, "cudaMemset");
  if ((e = cudaMalloc(&m->keys, sizeof(unsigned long long) * S))) return bail(e, "cudaMalloc");
  if ((e = cudaMemset(m->keys, 0, sizeof(unsigned long long) * S))) return bail(e, "cudaMemset");
  if ((e = cudaMalloc(&m->lm_counter, sizeof(unsigned int) * S))) return bail(e, "cudaMalloc");
  if ((e = cudaMemset(m->lm_counter, 0, sizeof(unsigned int) * S))) return bail(e, "cudaMemset");
  if ((e = cudaMalloc(&m->pos, sizeof(int) * S))) return bail(e, "cudaMalloc");
  if ((e = cudaMalloc(&m->tok, sizeof(int) * S))) return bail(e, "cudaMalloc");
  if ((e = cudaMalloc(&m->hist_n, sizeof(int) * S))) return bail(e, "cudaMalloc");
  if ((e = cudaMalloc(&m->err, sizeof(int)))) return bail(e, "cudaMalloc");
  if ((e = cudaMalloc(&m->hist, sizeof(int) * S * (size_t)d.cap))) return bail(e, "cudaMalloc");
  if ((e = cudaMalloc(&m->ids, sizeof(int) * (size_t)d.cap))) return bail(e, "cudaMalloc");
  cudaMemset(m->pos, 0, sizeof(int) * S);
  cudaMemset(m->tok, 0, sizeof(int) * S);
  cudaMemset(m->hist_n, 0, sizeof(int) * S);
  cudaMemset(m->err, 0, sizeof(int));
  const size_t pin_n = (size_t)(d.cap > S ? d.cap : S);
  if ((e = cudaMallocHost(&m->pinned, sizeof(int) * pin_n))) return bail(e, "cudaMallocHost");
  // RoPE table: angle = pos * theta^(-2i/hd), evaluated in double precision
  {
    const int half = d.hd / 2;
    std::vector<float2> tab((size_t)d.cap * half);
    for (int p = 0; p < d.cap; ++p)
      for (int i = 0; i < half; ++i) {
        const double ang = (double)p * std::pow((double)cfg->rope_theta, -2.0 * i / d.hd);
        tab[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    if ((e = cudaMalloc(&m->rope, sizeof(float2) * tab.size()))) return bail(e, "cudaMalloc");
    if ((e = cudaMemcpy(m->rope, tab.data(), sizeof(float2) * tab.size(), cudaMemcpyHostToDevice)))
      return bail(e, "cudaMemcpy(rope)");
  }
  m->pf.use_tc = false;
  if (cfg->dtype == QW_BF16 && gemm_tc_available()) {
    const char* simt = std::getenv("QW_PREFILL_SIMT");
    m->pf.use_tc = !(simt && simt[0] == '1');
  }
  if (m->pf.use_tc) {
    // fp16 copies of the layer matrices: the tensor-core operands of the prefill GEMMs
    const size_t H = d.H, qd = (size_t)d.nq * d.hd, kvd = (size_t)d.nkv * d.hd, I = d.I;
    const size_t sizes[7] = {qd * H, kvd * H, kvd * H, H * qd, I * H, I * H, H * I};
    // q, k, v back to back (no padding between them: one fused projection); the rest on
    // 256-byte boundaries; then the concatenated q/k/v bias
    const size_t qkv_bytes = ((sizes[0] + sizes[1] + sizes[2]) * 2 + 255) & ~(size_t)255;
    const size_t bias_bytes = ((qd + 2 * kvd) * 2 + 255) & ~(size_t)255;
    size_t per_layer = qkv_bytes + bias_bytes;
    for (int i = 3; i < 7; ++i) per_layer += (sizes[i] * 2 + 255) & ~(size_t)255;
    if ((e = cudaMalloc(&m->w16, per_layer * d.L))) return bail(e, "cudaMalloc(fp16 weights)");
    char* p = (char*)m->w16;
    for (int l = 0; l < d.L; ++l) {
      LayerPtrs& L = m->layers[l];
      const void* src[7] = {L.wq, L.wk, L.wv, L.wo, L.w_gate, L.w_up, L.w_down};
      const void** dst[7] = {&L.wq16, &L.wk16, &L.wv16, &L.wo16, &L.wg16, &L.wu16, &L.wd16};
      char* q0 = p;
      for (int i = 0; i < 7; ++i) {
        *dst[i] = p;
        // q, k, v: each head's rows in RoPE-pair order (the projection's epilogue rotates
        // adjacent columns)
        e = i < 3 ? convert_bf16_to_half_pairs(src[i], p, sizes[i] / H, (int)H, d.hd, m->err, 0)
                  : convert_bf16_to_half(src[i], p, sizes[i], m->err, 0);
        if (e) return bail(e, "fp16 weight copy");
        p += i < 2 ? sizes[i] * 2 : i == 2 ? q0 + qkv_bytes - p : (sizes[i] * 2 + 255) & ~(size_t)255;
      }
      L.bqkv = nullptr;
      if (L.bq) {
        if ((e = copy_bias_pairs(L.bq, p, (int)qd, d.hd, 0)) ||
            (e = copy_bias_pairs(L.bk, p + qd * 2, (int)kvd, d.hd, 0)) ||
            (e = copy_bias_pairs(L.bv, p + (qd + kvd) * 2, (int)kvd, d.hd, 0)))
          return bail(e, "q/k/v bias copy");
        L.bqkv = p;
      }
      p += bias_bytes;
    }
    int h_err = 0;
    if ((e = cudaMemcpy(&h_err, m->err, sizeof(int), cudaMemcpyDeviceToHost))) return bail(e, "cudaMemcpy");
    if (h_err) {
      m->release();
      delete m;
      return fail(QW_ERR_NUMERIC, "a weight lies outside the fp16 range of the prefill operands");
    }
  }
  if ((e = decode_set_attributes(d))) return bail(e, "decode attributes");
  {
    // single-sequence decode steps of bf16 models as one persistent kernel (QW_MEGA=0: one
    // kernel per operation) when the shape has an instance and one CTA per SM can be
    // resident with its shared memory (cooperative launch)
    const char* mv = std::getenv("QW_MEGA");
    int coop = 0, per_sm = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, m->device);
    if (!(mv && mv[0] == '0') && coop && megastep_supported(d, d.nsm)) {
      if ((e = megastep_set_attributes(d))) return bail(e, "decode step attributes");
      if ((e = megastep_occupancy(d, &per_sm))) return bail(e, "decode step occupancy");
    }
    if (per_sm >= 1) {
      std::vector<unsigned char> recs(megastep_layer_bytes() * d.L);
      for (int l = 0; l < d.L; ++l) megastep_fill_layer(recs.data() + l * megastep_layer_bytes(), m->layers[l]);
      if ((e = cudaMalloc(&m->mega_layers, recs.size()))) return bail(e, "cudaMalloc");
      if ((e = cudaMemcpy(m->mega_layers, recs.data(), recs.size(), cudaMemcpyHostToDevice)))
        return bail(e, "cudaMemcpy");
      if ((e = cudaMalloc(&m->mega_part, megastep_work_floats(d) * sizeof(float)))) return bail(e, "cudaMalloc");
      // [0] grid-barrier counter, [1] its step base, [2, 18) attention arrival counters per KV
      // head, [18, 34) their step bases
      const size_t nbar = 2 + 2 * 16;
      if ((e = cudaMalloc(&m->mega_bar, nbar * sizeof(unsigned long long)))) return bail(e, "cudaMalloc");
      if ((e = cudaMemset(m->mega_bar, 0, nbar * sizeof(unsigned long long)))) return bail(e, "cudaMemset");
      if ((e = cudaMalloc(&m->mega_abort, sizeof(int)))) return bail(e, "cudaMalloc");
      if ((e = cudaMemset(m->mega_abort, 0, sizeof(int)))) return bail(e, "cudaMemset");
      m->use_mega = true;
    }
  }
  if (m->pf.use_tc && S > 1) {
    // batched decode: every weight matrix read once per step for all active sequences
    const char* bz = std::getenv("QW_BATCHED");
    // (the merge kernel holds one head's outputs in one 128-thread CTA, 32 chunks at most)
    if (!(bz && bz[0] == '0') && d.H % 8 == 0 && d.I % 8 == 0 && (d.nq * d.hd) % 8 == 0 && d.hd <= 128 &&
        attn_nsplit_for(d.cap, d.attn_chunk_min, d.hd, 2, 32) <= 32) {
      const size_t H = d.H, qd = (size_t)d.nq * d.hd, kvd = (size_t)d.nkv * d.hd, I = d.I;
      auto al = [](size_t b) { return (b + 255) & ~(size_t)255; };
      const size_t sz_q = al(16 * qd * 4), sz_x16 = al(16 * H * 2), sz_o16 = al(16 * qd * 2), sz_a16 = al(16 * I * 2),
                   sz_xb = al(16 * H * 2), sz_act = al(sizeof(int) * S);
      m->bplans.resize(d.L);
      bool ok = true;
      size_t part_floats = 0;
      // the fp16 activation rows live at fixed offsets of one block, so the plans can be made
      // before the allocation is known: make them against the final addresses afterwards
      char* blk = nullptr;
      size_t total = sz_q + sz_x16 + sz_o16 + sz_a16 + sz_xb + sz_act;
      // partial buffer: size from the plans' split counts (computed with a placeholder first)
      for (int pass = 0; pass < 2 && ok; ++pass) {
        if (pass == 1) {
          if ((e = cudaMalloc(&m->bblock, total + al(part_floats * 4)))) return bail(e, "cudaMalloc(batched)");
          if ((e = cudaMemset(m->bblock, 0, total + al(part_floats * 4)))) return bail(e, "cudaMemset(batched)");
          blk = (char*)m->bblock;
          m->bq = (float*)blk;
          m->bX16 = (__half*)(blk + sz_q);
          m->bO16 = (__half*)(blk + sz_q + sz_x16);
          m->bA16 = (__half*)(blk + sz_q + sz_x16 + sz_o16);
          m->bXb16 = (__nv_bfloat16*)(blk + sz_q + sz_x16 + sz_o16 + sz_a16);
          m->bactive = (int*)(blk + sz_q + sz_x16 + sz_o16 + sz_a16 + sz_xb);
          m->bpart = (float*)(blk + total);
        }
        // pass 0 plans against a 256-aligned placeholder address, only for the split counts
        const void* X16 = pass ? (const void*)m->bX16 : (const void*)(uintptr_t)4096;
        const void* O16 = pass ? (const void*)m->bO16 : X16;
        const void* A16 = pass ? (const void*)m->bA16 : X16;
        const void* Xb = pass ? (const void*)m->bXb16 : X16;
        for (int l = 0; l < d.L && ok; ++l) {
          const LayerPtrs& L = m->layers[l];
          BatchedLayerPlans& P = m->bplans[l];
          const void* wqkv[3] = {L.wq16, L.wk16, L.wv16};
          const int rqkv[3] = {(int)qd, (int)kvd, (int)kvd};
          const void* wo[1] = {L.wo16};
          const int ro[1] = {(int)H};
          const void* wgu[2] = {L.wg16, L.wu16};
          const int rgu[2] = {(int)I, (int)I};
          const void* wd[1] = {L.wd16};
          const char* fg = std::getenv("QW_BATCHED_GLU");  // 0: SwiGLU as its own kernel
          const bool glu = !(fg && fg[0] == '0') && skinny_plan_glu(&P.gu, L.wg16, L.wu16, (int)I, X16, (int)H, d.nsm);
          ok = skinny_plan(&P.qkv, 3, wqkv, rqkv, X16, (int)H, false, d.nsm) &&
               skinny_plan(&P.o, 1, wo, ro, O16, (int)qd, false, d.nsm) &&
               (glu || skinny_plan(&P.gu, 2, wgu, rgu, X16, (int)H, false, d.nsm)) &&
               skinny_plan(&P.down, 1, wd, ro, A16, (int)I, false, d.nsm);
          if (ok && pass == 0)
            for (const SkinnyPlan* sp : {&P.qkv, &P.o, &P.gu, &P.down})
              part_floats = std::max(part_floats, (size_t)sp->splits * 16 * sp->n_total);
        }
        const void* wlm[1] = {m->head_w()};
        const int rlm[1] = {d.V};
        ok = ok && skinny_plan(&m->blm, 1, wlm, rlm, Xb, (int)H, true, d.nsm);
      }
      if (ok) {
        // Context chunks per sequence and KV head (at most 32: the merge's limit).
        // The tensor-core kernel streams a chunk in 64-position tiles: chunks of 128
        // positions (two tiles), as many as a sequence needs, keep every CTA's work alike
        // across sequences of different lengths (16 sequences of 256-2048 positions: 10150
        // tok/s against 9610 with 8 chunks of any length). The one-pass CUDA-core kernel wants
        // short chunks (32). QW_BATCHED_SPLITS and QW_BATCHED_CHUNK override.
        const char* bm = std::getenv("QW_BATCHED_ATTN_MMA");  // 0: CUDA-core attention
        m->battn_mma = !(bm && bm[0] == '0') && (d.hd == 64 || d.hd == 128) && d.nq / d.nkv <= 16;
        const char* bs = std::getenv("QW_BATCHED_SPLITS");
        const int bmax = bs ? std::max(1, std::min(32, std::atoi(bs))) : 32;
        const char* bc = std::getenv("QW_BATCHED_CHUNK");
        const int bcv = bc ? std::atoi(bc) : 0;
        m->battn_chunk = bcv >= 8 && bcv <= 4096 ? bcv : (m->battn_mma ? 128 : d.attn_chunk_min);
        if (m->battn_mma)
          m->battn_nsplit = std::max(1, std::min(bmax, (d.cap + m->battn_chunk - 1) / m->battn_chunk));
        else
          m->battn_nsplit = attn_nsplit_for(d.cap, m->battn_chunk, d.hd, 2, bmax);
        m->battn_smem = m->battn_mma ? 0  // (the tensor-core kernel sizes its own tiles)
                                     : attn_smem_bytes(d.nq / d.nkv, d.hd, d.cap, m->battn_nsplit, m->battn_chunk, 2);
        const size_t aws = attn_batched_workspace_bytes(d.nq, d.nkv, d.hd, m->battn_nsplit, S);
        if ((e = cudaMalloc(&m->battn_ws, aws))) return bail(e, "cudaMalloc(batched attention)");
        if ((e = cudaMemset(m->battn_ws, 0, aws))) return bail(e, "cudaMemset(batched attention)");
        if ((e = batched_set_attributes())) return bail(e, "batched attributes");
        if (m->battn_mma && (e = attn_decode_mma_set_attributes())) return bail(e, "decode attention attributes");
        m->use_batched = true;
      }
    }
  }
  if ((e = attn_set_attributes(std::max(m->attn_smem, m->battn_smem)))) return bail(e, "attention attributes");
  if ((e = prefill_set_attributes(d))) return bail(e, "prefill attributes");
  if ((e = cudaDeviceSynchronize())) return bail(e, "cudaDeviceSynchronize");
  m->h_pos.assign(S, 0);
  m->active.assign(S, 0);
  m->graphs.assign(S, nullptr);
  const char* ng = std::getenv("QW_NO_GRAPH");
  m->use_graphs = !(ng && ng[0] == '1');
  m->merge_in_oproj = d.nq * d.hd <= 2048;
  {
    // tensor-core decode attention (QW_ATTN_MMA=0: CUDA cores); measured on the 1.5B shape:
    // equal at a 128-token context, 662 -> 688 tok/s at 4096-4351 positions
    const char* am = std::getenv("QW_ATTN_MMA");
    m->attn_mma = !(am && am[0] == '0') && m->merge_in_oproj && cfg->dtype == QW_BF16 && (d.hd == 64 || d.hd == 128) &&
                  d.nq / d.nkv <= 16;
    if (m->attn_mma) QW_CUDA(attn_decode_mma_set_attributes());
  }
  *out = m;
  return QW_OK;
}

void qw_destroy(qw_model* m) {
  if (!m) return;
  cudaStreamSynchronize(m->stream);
  m->release();
  delete m;
}

static qw_status prefill_common(qw_model* m, int32_t seq, int32_t n) {
  if (!m) return fail(QW_ERR_INVALID_ARG, "null model");
  if (seq < 0 || seq >= m->d.max_seqs) return fail(QW_ERR_INVALID_ARG, "sequence index out of range");
  if (n < 1) return fail(QW_ERR_INVALID_ARG, "empty prompt");
  if (n > m->d.cap) return fail(QW_ERR_CAPACITY, "prompt longer than kv_capacity");
  return QW_OK;
}

qw_status qw_prefill_device(qw_model* m, int32_t seq, const int32_t* ids_dev, int32_t n) {
  g_err.clear();
  qw_status st = prefill_common(m, seq, n);
  if (st) return st;
  if (!ids_dev) return fail(QW_ERR_INVALID_ARG, "null ids");
  QW_CUDA(m->enqueue_prefill(seq, ids_dev, n));
  m->h_pos[seq] = n;
  m->active[seq] = 1;
  m->bactive_dirty = true;
  return QW_OK;
}

qw_status qw_prefill(qw_model* m, int32_t seq, const int32_t* ids, int32_t n, int32_t* next_token) {
  g_err.clear();
  qw_status st = prefill_common(m, seq, n);
  if (st) return st;
  if (!ids) return fail(QW_ERR_INVALID_ARG, "null ids");
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= m->d.V) return fail(QW_ERR_TOKEN_RANGE, "prompt token id outside [0, vocab)");
  QW_CUDA(cudaStreamSynchronize(m->stream));  // the pinned staging buffer is reused
  std::memcpy(m->pinned, ids, sizeof(int) * n);
  QW_CUDA(cudaMemcpyAsync(m->ids, m->pinned, sizeof(int) * n, cudaMemcpyHostToDevice, m->stream));
  QW_CUDA(m->enqueue_prefill(seq, m->ids, n));
  m->h_pos[seq] = n;
  m->active[seq] = 1;
  m->bactive_dirty = true;
  if (next_token) {
    QW_CUDA(cudaMemcpyAsync(m->pinned, m->tok + seq, sizeof(int), cudaMemcpyDeviceToHost, m->stream));
    st = m->check_device_errors();
    if (st) return st;
    *next_token = m->pinned[0];
  }
  return QW_OK;
}

static qw_status decode_prepare(qw_model* m) {
  bool any = false;
  for (int s = 0; s < m->d.max_seqs; ++s) {
    if (!m->active[s]) continue;
    any = true;
    if (m->h_pos[s] + 1 > m->d.cap) return fail(QW_ERR_CAPACITY, "sequence reached kv_capacity");
  }
  if (!any) return fail(QW_ERR_INVALID_ARG, "no prefilled sequence");
  if (fault_injected("launch")) return fail(QW_ERR_FAULT_INJECTED, "QW_FAULT=launch");
  return QW_OK;
}

qw_status qw_decode_step(qw_model* m, const int32_t* feed, int32_t* next_tokens) {
  g_err.clear();
  if (!m) return fail(QW_ERR_INVALID_ARG, "null model");
  qw_status st = decode_prepare(m);
  if (st) return st;
  const int S = m->d.max_seqs;
  if (feed) {
    for (int s = 0; s < S; ++s)
      if (m->active[s] && (feed[s] < 0 || feed[s] >= m->d.V))
        return fail(QW_ERR_TOKEN_RANGE, "fed token id outside [0, vocab)");
    QW_CUDA(cudaStreamSynchronize(m->stream));
    for (int s = 0; s < S; ++s) m->pinned[s] = feed[s];
    for (int s = 0; s < S; ++s)
      if (m->active[s])
        QW_CUDA(cudaMemcpyAsync(m->tok + s, m->pinned + s, sizeof(int), cudaMemcpyHostToDevice, m->stream));
  }
  QW_CUDA(m->decode_all());
  if (next_tokens) {
    QW_CUDA(cudaStreamSynchronize(m->stream));
    QW_CUDA(cudaMemcpyAsync(m->pinned, m->tok, sizeof(int) * S, cudaMemcpyDeviceToHost, m->stream));
    st = m->check_device_errors();
    if (st) return st;
    for (int s = 0; s < S; ++s) next_tokens[s] = m->active[s] ? m->pinned[s] : -1;
  }
  return QW_OK;
}

qw_status qw_decode_steps(qw_model* m, int32_t n_steps) {
  g_err.clear();
  if (!m) return fail(QW_ERR_INVALID_ARG, "null model");
  if (n_steps < 0) return fail(QW_ERR_INVALID_ARG, "negative step count");
  for (int i = 0; i < n_steps; ++i) {
    qw_status st = decode_prepare(m);
    if (st) return st;
    QW_CUDA(m->decode_all());
  }
  return QW_OK;
}

static qw_status generate_impl(qw_model* m, const int32_t* ids, int32_t n, int32_t max_new,
                               const int32_t* stops, int32_t n_stops, int32_t* out, int32_t* n_out) {
  if (!m || !out || !n_out) return fail(QW_ERR_INVALID_ARG, "null argument");
  if (n_stops < 0 || (n_stops > 0 && !stops)) return fail(QW_ERR_INVALID_ARG, "bad stop-id set");
  if (max_new < 1) return fail(QW_ERR_INVALID_ARG, "max_new must be positive");
  qw_status st = prefill_common(m, 0, n);
  if (st) return st;
  if ((int64_t)n + max_new - 1 > m->d.cap) return fail(QW_ERR_CAPACITY, "prompt + max_new - 1 exceeds kv_capacity");
  for (int s = 1; s < m->d.max_seqs; ++s) m->active[s] = 0;
  m->bactive_dirty = true;
  st = qw_prefill(m, 0, ids, n, nullptr);
  if (st) return st;
  const int chunk = n_stops > 0 ? 16 : max_new;
  int done = 1;  // tokens produced so far
  int produced_total = 1;
  while (true) {
    const int steps = std::min(chunk, max_new - done);
    for (int i = 0; i < steps; ++i) {
      QW_CUDA(m->run_decode(0));
      m->h_pos[0] += 1;
    }
    done += steps;
    produced_total = done;
    QW_CUDA(cudaMemcpyAsync(m->pinned, m->hist, sizeof(int) * done, cudaMemcpyDeviceToHost, m->stream));
    st = m->check_device_errors();
    if (st) return st;
    int cut = -1;
    for (int i = 0; i < done && cut < 0; ++i)
      for (int k = 0; k < n_stops; ++k)
        if (m->pinned[i] == stops[k]) { cut = i + 1; break; }
    if (cut > 0 || done >= max_new) {
      const int k = cut > 0 ? cut : done;
      std::memcpy(out, m->pinned, sizeof(int) * k);
      *n_out = k;
      if (k < produced_total) {  // steps ran past eos: roll length and next token back
        const int len = n + k - 1;
        m->h_pos[0] = len;
        m->pinned[0] = len;
        m->pinned[1] = out[k - 1];
        QW_CUDA(cudaMemcpyAsync(m->pos, &m->pinned[0], sizeof(int), cudaMemcpyHostToDevice, m->stream));
        QW_CUDA(cudaMemcpyAsync(m->tok, &m->pinned[1], sizeof(int), cudaMemcpyHostToDevice, m->stream));
        QW_CUDA(cudaStreamSynchronize(m->stream));
      }
      return QW_OK;
    }
  }
}

qw_status qw_generate(qw_model* m, const int32_t* ids, int32_t n, int32_t max_new, int32_t eos,
                      int32_t* out, int32_t* n_out) {
  g_err.clear();
  return generate_impl(m, ids, n, max_new, &eos, eos >= 0 ? 1 : 0, out, n_out);
}

qw_status qw_generate_stops(qw_model* m, const int32_t* ids, int32_t n, int32_t max_new, const int32_t* stop_ids,
                            int32_t n_stop, int32_t* out, int32_t* n_out) {
  g_err.clear();
  return generate_impl(m, ids, n, max_new, stop_ids, n_stop, out, n_out);
}

qw_status qw_sync(qw_model* m) {
  g_err.clear();
  if (!m) return fail(QW_ERR_INVALID_ARG, "null model");
  return m->check_device_errors();
}

const float* qw_logits(const qw_model* m) { return m ? m->logits : nullptr; }
qw_status qw_set_trace(qw_model* m, int32_t kind, void* const* begin, void* const* end) {
  g_err.clear();
  if (!m) return fail(QW_ERR_INVALID_ARG, "null model");
  QW_CUDA(cudaStreamSynchronize(m->stream));
  m->drop_graphs();
  if (!begin || !end) {
    m->trace_kind = -1;
    m->trace_begin.clear();
    m->trace_end.clear();
    return QW_OK;
  }
  if (kind < 0 || kind > 5) return fail(QW_ERR_INVALID_ARG, "unknown kernel kind");
  const int n = kind == 5 ? 1 : m->d.L;
  m->trace_begin.assign((cudaEvent_t*)begin, (cudaEvent_t*)begin + n);
  m->trace_end.assign((cudaEvent_t*)end, (cudaEvent_t*)end + n);
  for (int i = 0; i < n; ++i)
    if (!m->trace_begin[i] || !m->trace_end[i]) return fail(QW_ERR_INVALID_ARG, "null event");
  m->trace_kind = kind;
  return QW_OK;
}

qw_status qw_set_timeline(qw_model* m, int32_t enable) {
  g_err.clear();
  if (!m) return fail(QW_ERR_INVALID_ARG, "null model");
  QW_CUDA(cudaStreamSynchronize(m->stream));
  m->drop_graphs();
  if (m->tl_buf) {
    cudaFree(m->tl_buf);
    m->tl_buf = nullptr;
  }
  if (!enable) return QW_OK;
  m->tl_n = 1 + 5 * m->d.L + 1;
  if (m->use_mega)  // three records per phase, then every CTA's arrival after layer 1's phases
    m->tl_n = std::max(m->tl_n, 3 * (5 * m->d.L + 1) + (5 * m->d.nsm + 8 * (5 * m->d.L + 1) + 2) / 3);
  if (m->use_batched) m->tl_n = std::max(m->tl_n, 3 + 10 * m->d.L);  // launches of a batched step
  m->tl_init.assign((size_t)3 * m->tl_n, ~0ull);
  for (int i = 0; i < m->tl_n; ++i) m->tl_init[3 * i + 2] = 0ull;
  QW_CUDA(cudaMalloc(&m->tl_buf, sizeof(unsigned long long) * 3 * m->tl_n));
  QW_CUDA(cudaMemcpy(m->tl_buf, m->tl_init.data(), sizeof(unsigned long long) * 3 * m->tl_n,
                     cudaMemcpyHostToDevice));
  return QW_OK;
}

qw_status qw_read_timeline(qw_model* m, uint64_t* out, int32_t max_launches, int32_t* n_launches) {
  g_err.clear();
  if (!m || !out || !n_launches) return fail(QW_ERR_INVALID_ARG, "null argument");
  if (!m->tl_buf) return fail(QW_ERR_INVALID_ARG, "timeline not enabled");
  const int n = m->tl_n < max_launches ? m->tl_n : max_launches;
  QW_CUDA(cudaMemcpyAsync(out, m->tl_buf, sizeof(unsigned long long) * 3 * n, cudaMemcpyDeviceToHost, m->stream));
  QW_CUDA(cudaStreamSynchronize(m->stream));
  *n_launches = n;
  return QW_OK;
}

qw_status qw_read_logits(qw_model* m, int32_t seq, float* host_out) {
  g_err.clear();
  if (!m || !host_out) return fail(QW_ERR_INVALID_ARG, "null argument");
  if (seq < 0 || seq >= m->d.max_seqs) return fail(QW_ERR_INVALID_ARG, "sequence index out of range");
  QW_CUDA(cudaMemcpyAsync(host_out, m->logits + (size_t)seq * m->d.V, sizeof(float) * m->d.V,
                          cudaMemcpyDeviceToHost, m->stream));
  return m->check_device_errors();
}

const int32_t* qw_tokens_device(const qw_model* m) { return m ? m->tok : nullptr; }

int32_t qw_decode_kernels_per_step(const qw_model* m) {
  if (!m) return 0;
  return m->use_mega ? 1 : 5 * m->d.L + 2;
}

qw_status qw_position(const qw_model* m, int32_t seq, int32_t* pos) {
  g_err.clear();
  if (!m || !pos) return fail(QW_ERR_INVALID_ARG, "null argument");
  if (seq < 0 || seq >= m->d.max_seqs) return fail(QW_ERR_INVALID_ARG, "sequence index out of range");
  *pos = m->active[seq] ? m->h_pos[seq] : 0;
  return QW_OK;
}

qw_status qw_reset(qw_model* m, int32_t seq) {
  g_err.clear();
  if (!m) return fail(QW_ERR_INVALID_ARG, "null model");
  if (seq < 0 || seq >= m->d.max_seqs) return fail(QW_ERR_INVALID_ARG, "sequence index out of range");
  m->active[seq] = 0;
  m->bactive_dirty = true;
  m->h_pos[seq] = 0;
  QW_CUDA(cudaMemsetAsync(m->pos + seq, 0, sizeof(int), m->stream));
  return QW_OK;
}

// ---- single-op entry points ----

size_t qw_op_decode_attention_workspace(int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                        int32_t max_ctx) {
  if (n_heads < 1 || n_kv_heads < 1 || head_dim < 2 || max_ctx < 1) return 0;
  // fp32 keys and values need the most chunks; the fp16 case fits the same workspace
  return attn_workspace_bytes(n_heads, n_kv_heads, head_dim, op_attn_nsplit(head_dim, max_ctx, 4));
}

qw_status qw_op_decode_attention(int32_t kv_dtype, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                 int32_t ctx, int32_t kv_stride, const float* q, const void* k,
                                 const void* v, float* out, void* workspace, size_t workspace_bytes,
                                 void* cuda_stream) {
  g_err.clear();
  if (!q || !k || !v || !out || !workspace) return fail(QW_ERR_INVALID_ARG, "null pointer");
  if (kv_dtype != QW_F32 && kv_dtype != QW_F16) return fail(QW_ERR_INVALID_ARG, "kv dtype must be QW_F32 or QW_F16");
  if (n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || head_dim < 2 || ctx < 1 || kv_stride < ctx)
    return fail(QW_ERR_INVALID_ARG, "bad attention shape");
  if (n_heads / n_kv_heads > 8) return fail(QW_ERR_UNSUPPORTED, "more than 8 query heads per KV head");
  if (head_dim % 8 || (n_heads / n_kv_heads) * head_dim > 1024)
    return fail(QW_ERR_UNSUPPORTED, "head_dim must be a multiple of 8 with (n_heads / n_kv_heads) * head_dim <= 1024");
  const int nsplit = op_attn_nsplit(head_dim, kv_stride, kv_dtype == QW_F16 ? 2 : 4);
  const size_t need = op_attn_workspace_exact(kv_dtype, n_heads, n_kv_heads, head_dim, kv_stride);
  if (workspace_bytes < need) return fail(QW_ERR_INVALID_ARG, "workspace too small");
  if ((uintptr_t)workspace % 16) return fail(QW_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  const size_t smem = attn_smem_bytes(n_heads / n_kv_heads, head_dim, kv_stride, nsplit, ATTN_CHUNK_MIN,
                                      kv_dtype == QW_F16 ? 2 : 4);
  if (smem > 220 * 1024) return fail(QW_ERR_UNSUPPORTED, "attention chunk too large for shared memory");
  cudaError_t e = attn_set_attributes(smem);
  if (e) return cuda_fail(e, "decode attention attributes");
  e = launch_attn(kv_dtype, n_heads, n_kv_heads, head_dim, nsplit, ATTN_CHUNK_MIN, smem, q, k, v,
                  kv_stride, nullptr, ctx, out, workspace, nullptr, (cudaStream_t)cuda_stream, false);
  if (e) return cuda_fail(e, "decode attention launch");
  return QW_OK;
}

static qw_status gemm_args(int32_t M, int32_t N, int32_t K, const void* A, const void* B) {
  if (M < 1 || N < 1 || K < 1) return fail(QW_ERR_INVALID_ARG, "non-positive GEMM size");
  if (!A || !B) return fail(QW_ERR_INVALID_ARG, "null pointer");
  if (N % 8 || K % 8) return fail(QW_ERR_UNSUPPORTED, "N and K must be multiples of 8");
  if (((uintptr_t)A | (uintptr_t)B) & 15) return fail(QW_ERR_INVALID_ARG, "operand not 16-byte aligned");
  if (!gemm_tc_available()) return fail(QW_ERR_UNSUPPORTED, "tensor-map encoder unavailable");
  return QW_OK;
}

qw_status qw_op_gemm_f16(int32_t M, int32_t N, int32_t K, const void* A, const void* B, const void* bias,
                          float* C, int32_t accumulate, int32_t* err_dev, void* cuda_stream) {
  g_err.clear();
  qw_status st = gemm_args(M, N, K, A, B);
  if (st) return st;
  if (!C || !err_dev) return fail(QW_ERR_INVALID_ARG, "null pointer");
  if ((uintptr_t)C & 15) return fail(QW_ERR_INVALID_ARG, "C not 16-byte aligned");
  cudaError_t e = gemm_tc_set_attributes();
  if (e) return cuda_fail(e, "gemm attributes");
  int dev = 0, nsm = 0;  // persistent CTAs, one per SM
  if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)))
    return cuda_fail(e, "device query");
  e = gemm_tc((const f16*)A, K, (const f16*)B, K, (const bf16*)bias, C, N, M, N, K, accumulate != 0,
              err_dev, (cudaStream_t)cuda_stream, nullptr, 0, nsm);
  if (e) return cuda_fail(e, "gemm launch");
  return QW_OK;
}

qw_status qw_op_gemm_swiglu_f16(int32_t M, int32_t N, int32_t K, const void* A, const void* Wg,
                                 const void* Wu, void* act, int32_t* err_dev, void* cuda_stream) {
  g_err.clear();
  qw_status st = gemm_args(M, N, K, A, Wg);
  if (st) return st;
  if (!Wu || !act || !err_dev) return fail(QW_ERR_INVALID_ARG, "null pointer");
  if (((uintptr_t)Wu | (uintptr_t)act) & 15) return fail(QW_ERR_INVALID_ARG, "operand not 16-byte aligned");
  cudaError_t e = gemm_tc_set_attributes();
  if (e) return cuda_fail(e, "gemm attributes");
  int dev = 0, nsm = 0;  // persistent CTAs, one per SM
  if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)))
    return cuda_fail(e, "device query");
  e = gemm_tc_swiglu((const f16*)A, K, (const f16*)Wg, (const f16*)Wu, K, (f16*)act, N, M, N, K, err_dev,
                     (cudaStream_t)cuda_stream, nullptr, 0, nsm);
  if (e) return cuda_fail(e, "gemm launch");
  return QW_OK;
}

}  // extern "C"
