// Shared device helpers for the libqw kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qw {

typedef __nv_bfloat16 bf16;
typedef __half f16;

// Device-side error bits, OR-ed into the model's status word:
//   ERR_TOKEN     a token id outside [0, vocab)
//   ERR_NONFINITE non-finite logits
//   ERR_TIMEOUT   a bounded wait gave up
//   ERR_RANGE     a value written to an fp16 KV cache or fp16 tensor-core operand lay
//                 outside the fp16 range (or was not finite)
//   ERR_LAYOUT    a kernel found its shared-memory window misaligned and skipped its work
enum : int { ERR_TOKEN = 1, ERR_NONFINITE = 2, ERR_TIMEOUT = 4, ERR_RANGE = 8, ERR_LAYOUT = 16 };

// fp32 -> fp16 (round to nearest even) for data whose range the model does not bound: a
// value that would round to infinity, or a non-finite one, sets ERR_RANGE in *err.
__device__ __forceinline__ f16 to_half_checked(float v, int* err) {
  if (!(fabsf(v) < 65520.f)) atomicOr(err, ERR_RANGE);
  return __float2half_rn(v);
}
__device__ __forceinline__ __half2 to_half2_checked(float a, float b, int* err) {
  if (!(fabsf(a) < 65520.f) || !(fabsf(b) < 65520.f)) atomicOr(err, ERR_RANGE);
  return __floats2half2_rn(a, b);
}
// the KV-cache store of either element type (fp32 caches cannot overflow)
__device__ __forceinline__ void store_kv(float* dst, float v, int*) { *dst = v; }
__device__ __forceinline__ void store_kv(f16* dst, float v, int* err) { *dst = to_half_checked(v, err); }

// Programmatic dependent launch: wait for the upstream grid's completion and memory,
// and allow the downstream grid to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<bf16> { static constexpr int N = 8; };

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(f16 v) { return __half2float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }
template <> __device__ __forceinline__ f16 from_f32<f16>(float v) { return __float2half_rn(v); }

// 16-byte streaming load of read-only data (weights): no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// dot of one 16-byte vector of weights with VEC fp32 inputs
__device__ __forceinline__ float dotv(const uint4& w, const float* x, float acc, float) {
  acc = fmaf(__uint_as_float(w.x), x[0], acc);
  acc = fmaf(__uint_as_float(w.y), x[1], acc);
  acc = fmaf(__uint_as_float(w.z), x[2], acc);
  acc = fmaf(__uint_as_float(w.w), x[3], acc);
  return acc;
}
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float dotv(const uint4& w, const float* x, float acc, bf16) {
  acc = fmaf(bf_lo(w.x), x[0], acc);
  acc = fmaf(bf_hi(w.x), x[1], acc);
  acc = fmaf(bf_lo(w.y), x[2], acc);
  acc = fmaf(bf_hi(w.y), x[3], acc);
  acc = fmaf(bf_lo(w.z), x[4], acc);
  acc = fmaf(bf_hi(w.z), x[5], acc);
  acc = fmaf(bf_lo(w.w), x[6], acc);
  acc = fmaf(bf_hi(w.w), x[7], acc);
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over the block (any blockDim multiple of 32, <= 1024). All threads get the result.
__device__ __forceinline__ float block_sum(float v, float* scratch32) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch32[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += scratch32[i];  // fixed order: deterministic
  return t;
}

// Orderable 64-bit argmax key: larger value wins, then the lower index.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xffffffffu - (uint32_t)idx);
}
__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
  return (int)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
}

// ---- mbarrier and bulk-copy (TMA, 1-D) primitives ----------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// non-blocking test of phase `parity` (no suspension)
__device__ __forceinline__ bool mbar_test_now(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
constexpr long long WAIT_CYCLES = 4000000000ll;  // ~2 s at 2 GHz
// Wait for phase `parity` of the barrier; false if the budget ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_test(bar, parity))
    if (clock64() - t0 > WAIT_CYCLES) return false;
  return true;
}
// Order this thread's earlier generic-proxy shared-memory accesses before later async-proxy
// (bulk copy) writes.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// bytes (multiple of 16) from global src to shared dst (both 16-byte aligned); completion is
// counted on the barrier as transaction bytes
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Device timeline (profiling): globaltimer stamps reduced with atomics into per-launch slots.
__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// slots: [0] first CTA start, [1] first CTA past the dependency wait, [2] last CTA end
__device__ __forceinline__ void tl_stamp(unsigned long long* tl, int which) {
  if (tl && threadIdx.x == 0) {
    if (which < 2) atomicMin(tl + which, gtime());
    else atomicMax(tl + 2, gtime());
  }
}

// ---- warp-level tensor-core helpers (mma.sync m16n8k16, fp16 operands, fp32 accumulators) --
// Fragments follow the PTX ISA layout: with g = lane / 4 and t = lane % 4, A holds rows g and
// g + 8 at columns 2t, 2t + 1 (and + 8); B holds rows (k) 2t, 2t + 1 (and + 8) at column g;
// C holds rows g and g + 8 at columns 2t, 2t + 1.
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// four 8x8 b16 matrices, transposed: thread i gives the row address of row i % 8 of matrix
// i / 8; register j receives matrix j's elements (2t, g) and (2t + 1, g)
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t* r, const void* row_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(row_addr)));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16_s(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// The barrier's current phase counts one arrival when every cp.async this thread issued
// so far has landed (the barrier's expected count includes that arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Ask L2 to fetch bytes (multiple of 16) at src (16-byte aligned); no completion tracking.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

}  // namespace qw

// ---- host: kernel launch with optional programmatic dependent launch ----------------------
namespace qw {
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
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
}  // namespace qw
