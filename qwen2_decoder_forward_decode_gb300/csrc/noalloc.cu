// Decode attention with library-owned scratch: an entry point that allocates nothing.
//
// Some callers cannot allocate device memory on the path where they call attention: code
// embedded in another runtime whose memory is owned by that runtime's allocator, loops
// that must not hit cudaMalloc's implicit device synchronisation, or environments where a
// failed allocation mid-run is not acceptable. For them the split-context partials and
// the per-KV-head counters live in one fixed array below instead of a workspace argument.
#include "../../include/qw.h"
#include "internal.h"

#include <mutex>

namespace {

// Scratch of qw_op_decode_attention_noalloc. Every GPU that loads the library holds this
// array until the process exits. Calls share it and it keeps the last call's contents.
constexpr size_t NOALLOC_SCRATCH_BYTES = 1u << 20;  // 1 MiB
static __device__ __align__(256) unsigned char g_attn_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_scratch_addr[MAX_DEVICES] = {};  // device address of g_attn_scratch, per device

qw_status fail(qw_status s, const char* msg) {
  qw::set_error_message(msg);
  return s;
}

// Device address of the scratch array on the current device. The first call on a device
// looks it up (cudaGetSymbolAddress); that may not happen inside a stream capture.
qw_status scratch_on_current_device(cudaStream_t s, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(QW_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= MAX_DEVICES) return fail(QW_ERR_UNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess)
      return fail(QW_ERR_CUDA, "cudaStreamIsCapturing failed");
    if (cs != cudaStreamCaptureStatusNone)
      return fail(QW_ERR_INVALID_ARG,
                  "the first qw_op_decode_attention_noalloc call on a device must come before any stream capture");
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess || !p) return fail(QW_ERR_CUDA, cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return QW_OK;
}

}  // namespace

extern "C" {

size_t qw_op_decode_attention_noalloc_limit(void) { return NOALLOC_SCRATCH_BYTES; }

qw_status qw_op_decode_attention_noalloc(int32_t kv_dtype, int32_t n_heads, int32_t n_kv_heads,
                                         int32_t head_dim, int32_t ctx, int32_t kv_stride,
                                         const float* q, const void* k, const void* v, float* out,
                                         void* cuda_stream) {
  if (!q || !k || !v || !out) return fail(QW_ERR_INVALID_ARG, "null pointer");
  if (kv_dtype != QW_F32 && kv_dtype != QW_F16) return fail(QW_ERR_INVALID_ARG, "kv dtype must be QW_F32 or QW_F16");
  if (n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || head_dim < 2 || ctx < 1 || kv_stride < ctx)
    return fail(QW_ERR_INVALID_ARG, "bad attention shape");
  if (n_heads / n_kv_heads > 8) return fail(QW_ERR_UNSUPPORTED, "more than 8 query heads per KV head");
  // exactly the workspace the attention kernel will use for this KV type: its split count
  // (and so where its counters sit) depends on the element size
  const size_t need = qw::op_attn_workspace_exact(kv_dtype, n_heads, n_kv_heads, head_dim, kv_stride);
  if (need == 0 || need > NOALLOC_SCRATCH_BYTES)
    return fail(QW_ERR_UNSUPPORTED, "shape needs more scratch than the fixed 1 MiB array holds");
  cudaStream_t s = (cudaStream_t)cuda_stream;
  void* ws = nullptr;
  qw_status st = scratch_on_current_device(s, &ws);
  if (st) return st;
  // the per-KV-head arrival counters are the last bytes of that workspace and must start at
  // zero; an earlier call of another shape may have left partials there
  const size_t counters = (size_t)n_kv_heads * sizeof(unsigned int);
  if (cudaMemsetAsync((char*)ws + need - counters, 0, counters, s) != cudaSuccess)
    return fail(QW_ERR_CUDA, "cudaMemsetAsync of the scratch counters failed");
  return qw_op_decode_attention(kv_dtype, n_heads, n_kv_heads, head_dim, ctx, kv_stride, q, k, v, out, ws,
                                need, cuda_stream);
}

}  // extern "C"
