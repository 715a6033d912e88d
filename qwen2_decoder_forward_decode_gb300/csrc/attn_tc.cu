// Causal prefill attention on the 5th-generation tensor cores (tcgen05, TMEM).
//
// "LLM Speedrun: Architecture" (Attention, Causal mask, Grouped Query Attention): query row t
// of head h (position pos0 + t) takes softmax over keys j <= pos0 + t of q . k_j / sqrt(d) and
// the weighted sum of the v_j; head h reads KV head h / (n_heads / n_kv_heads).
//
// One CTA per (128 query rows, head), the longest row blocks first. Keys stream in blocks of
// 128 in the online-softmax form:
//   warp 0, lane 0 / 1   TMA producers: the Q tile, then the key rows (lane 0) and value rows
//                        (lane 1) of each block into their own rings, straight from the fp16
//                        cache
//   warp 1, lane 0       MMA issuer: S_j = Q K_j^T (M 128, N 128 keys) into TMEM buffer j % 3;
//                        once the softmax has written P_j back over it, O += P_j V_j (M 128,
//                        N hd, K 128 keys) with P read straight from TMEM and V_j MN-major
//                        (head dimension contiguous), as the cache stores it. S_{j+2} is
//                        issued before waiting for P_j, so the tensor cores always hold work
//                        while the softmax runs.
//   warps 2..9           softmax. The warp pair (w, w + 4) shares TMEM lanes 32 (w % 4) ..
//                        +31, one query row per lane: warps 2..5 take keys 0..63 of every
//                        block, 6..9 keys 64..127, and the pair trades its halves' maxima
//                        (at the end its sums) through shared memory. Each thread masks keys
//                        past its row's position and writes P = 2^(S - m) as fp16 pairs over
//                        its half of S.
// The reference maximum m of a row moves only when a block's maximum exceeds it by more than
// 8 (base 2): then the warp rescales its half of O in TMEM (and l) by 2^(m_old - m_new) once
// P_{j-1} V_{j-1} is done, before P_j is released. Otherwise P stays below 2^8, which fp16
// holds with its full relative precision, and O accumulates in TMEM untouched. Every term of
// O and l carries the same factor 2^-m, so o / l is the softmax-weighted sum; it goes to the
// fp16 operand of the o_proj GEMM.
// Each CTA starts at its own key block and wraps around, so that CTAs do not all read the
// same lines at the same time.
// Q arrives in fp16, already multiplied by log2(e) / sqrt(d), so scores are in base 2.
// Launched with programmatic dependent launch (the prefill), the CTAs may start while the
// q/k/v projection finishes; they wait for it before reading anything.
// Every mbarrier wait is bounded: on expiry the thread flags ERR_TIMEOUT, the CTA stops
// issuing work, waits (bounded) for what it issued, and releases its TMEM.
#include <cuda.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace qw {
namespace fa {

constexpr int BQ = 128, BKEY = 128, THREADS = 320, TMEM_COLS = 512;

template <int HD>
struct L {
  static constexpr int KS = HD == 128 ? 3 : 4;    // depth of the key ring and of the value ring
  static constexpr int Q_BYTES = BQ * HD * 2;     // HD / 64 boxes [128 rows][64 columns]
  static constexpr int K_BYTES = BKEY * HD * 2;   // HD / 64 boxes [128 keys][64 columns]
  static constexpr int V_BYTES = BKEY * HD * 2;   // HD / 64 boxes [128 keys][64 columns]
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = OFF_K + KS * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + KS * V_BYTES;
  // q_full, k_full[KS], k_empty[KS], v_full[KS], v_empty[KS], s_full[3], p_full[3],
  // o_step[2], done, xb[4 warp pairs]
  static constexpr int NBAR = 1 + 4 * KS + 6 + 2 + 1 + 4;
  static constexpr int OFF_X = OFF_BAR + NBAR * 8 + 16;  // row maxima / sums [2][half][row]
  // the window must start 1024-byte aligned (the kernel checks): no slack is requested
  static constexpr int SMEM = OFF_X + 2 * 2 * BQ * 4;
  // TMEM columns: S (fp32) / P (fp16 pairs) buffers at 0, BKEY and 2 BKEY, O after them
  static constexpr int O_COL = 3 * BKEY;
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(3 * BKEY + HD <= TMEM_COLS, "TMEM");
};

constexpr float RESCALE_AT = 8.f;  // base-2 growth of a row maximum that moves its reference

struct Args {
  int T, pos0, nq, nkv, nqb;
  f16* Oh;  // [T][nq * HD]
  int* err;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// packed pairs of fp32 (one instruction for two lanes of arithmetic)
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  uint32_t a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(a), "=r"(b) : "l"(v));
  lo = __uint_as_float(a);
  hi = __uint_as_float(b);
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

template <int HD>
__global__ void __launch_bounds__(THREADS, 1)
attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const Args a) {
  using Lay = L<HD>;
  constexpr int KS = Lay::KS;
  pdl_trigger();  // the next kernel may be scheduled once every CTA of this one has started
  extern __shared__ __align__(1024) uint8_t fa_raw[];
  uint8_t* smem = fa_raw;
  uint64_t* bars = (uint64_t*)(smem + Lay::OFF_BAR);
  uint32_t* tmem_slot = (uint32_t*)(bars + Lay::NBAR);
  volatile int* s_abort = (volatile int*)(tmem_slot + 1);
  const uint32_t q_full = tc::smem_u32(bars);
  const uint32_t k_full0 = q_full + 8, k_empty0 = k_full0 + 8 * KS;
  const uint32_t v_full0 = k_empty0 + 8 * KS, v_empty0 = v_full0 + 8 * KS;
  const uint32_t s_full0 = v_empty0 + 8 * KS, p_full0 = s_full0 + 24, o_step0 = p_full0 + 24;
  const uint32_t done = o_step0 + 16, xb0 = done + 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int qb = a.nqb - 1 - (int)blockIdx.x / a.nq, h = (int)blockIdx.x % a.nq;
  const int g = h / (a.nq / a.nkv);
  const int q0 = qb * BQ;
  const int nb = (a.pos0 + min(a.T, q0 + BQ) - 1) / BKEY + 1;  // key blocks the tile sees
  // CTAs start at different key blocks (and wrap around), so they do not all read the same
  // lines at once; the streaming softmax takes the blocks in any order
  const int rot = (int)((blockIdx.x * 5u) % (unsigned)nb);
  auto key_block = [&](int j) { return j + rot < nb ? j + rot : j + rot - nb; };

  if (tc::smem_u32(fa_raw) & 1023) {  // the swizzled operand tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(a.err, ERR_LAYOUT);
    return;
  }
  pdl_wait();  // q and the caches come from the previous kernel
  // after a timeout anywhere on the stream the remaining CTAs do nothing
  if (threadIdx.x == 0) *s_abort = (*(volatile int*)a.err & ERR_TIMEOUT) != 0;
  __syncthreads();
  if (*s_abort) return;
  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < KS; ++s) {
      tc::mbar_init(k_full0 + 8 * s, 1);
      tc::mbar_init(k_empty0 + 8 * s, 1);
      tc::mbar_init(v_full0 + 8 * s, 1);
      tc::mbar_init(v_empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 3; ++b) {
      tc::mbar_init(s_full0 + 8 * b, 1);
      tc::mbar_init(p_full0 + 8 * b, 8);  // one arrival per softmax warp
    }
    tc::mbar_init(o_step0, 1);
    tc::mbar_init(o_step0 + 8, 1);
    tc::mbar_init(done, 1);
    for (int i = 0; i < 4; ++i) tc::mbar_init(xb0 + 8 * i, 2);  // the two warps of a pair
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane < 2) {
      // ---- lane 0: the Q tile, then key blocks; lane 1: value blocks
      const bool kl = lane == 0;
      const CUtensorMap* map = kl ? &tmK : &tmV;
      const uint32_t full0 = kl ? k_full0 : v_full0, empty0 = kl ? k_empty0 : v_empty0;
      const int off = kl ? Lay::OFF_K : Lay::OFF_V;
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
      if (kl) {
        tc::mbar_expect_tx(q_full, Lay::Q_BYTES);
        for (int c = 0; c < HD / 64; ++c)
          tc::tma_load_2d(tc::smem_u32(smem) + c * BQ * 128, &tmQ, q_full, h * HD + c * 64, q0);
      }
      int issued = 0;
      for (int j = 0; j < nb; ++j) {
        const int s = j % KS;
        if (j >= KS && !tc::mbar_wait(empty0 + 8 * s, ((j / KS) & 1) ^ 1, a.err)) {
          *s_abort = 1;
          break;
        }
        if (*s_abort) break;
        const uint32_t st = tc::smem_u32(smem + off + s * Lay::K_BYTES);
        tc::mbar_expect_tx(full0 + 8 * s, Lay::K_BYTES);
        for (int c = 0; c < HD / 64; ++c) tc::tma_load_3d(st + c * BKEY * 128, map, full0 + 8 * s, c * 64, key_block(j) * BKEY, g);
        ++issued;
      }
      // every copy issued lands before the shared memory is released
      if (kl) tc::mbar_wait(q_full, 0, a.err);
      for (int j = issued > KS ? issued - KS : 0; j < issued; ++j)
        tc::mbar_wait(full0 + 8 * (j % KS), (j / KS) & 1, a.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      constexpr uint32_t idS = tc::idesc_f16(BQ, BKEY), idO = tc::idesc_f16_bmn(BQ, HD);
      const uint32_t qbase = tc::smem_u32(smem);
      auto issue_s = [&](int j) -> bool {  // S_j into buffer j % 3; then K_j's slot is free
        const int s = j % KS;
        if (!tc::mbar_wait(k_full0 + 8 * s, (j / KS) & 1, a.err)) return false;
        tc::tc_fence_after();
        const uint32_t kbase = tc::smem_u32(smem + Lay::OFF_K + s * Lay::K_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc::mma_f16(tmem + (j % 3) * BKEY, tc::smem_desc_sw128(qbase + (kk >> 2) * BQ * 128 + (kk & 3) * 32),
                      tc::smem_desc_sw128(kbase + (kk >> 2) * BKEY * 128 + (kk & 3) * 32), idS, kk > 0);
        tc::mma_commit(s_full0 + 8 * (j % 3));
        tc::mma_commit(k_empty0 + 8 * s);
        return true;
      };
      bool ok = tc::mbar_wait(q_full, 0, a.err) && issue_s(0) && (nb < 2 || issue_s(1));
      for (int j = 0; j < nb && ok; ++j) {
        if (*s_abort) {
          ok = false;
          break;
        }
        // S_{j+2} into the buffer of P_{j-1}, which P_{j-1} V_{j-1} (issued before) reads
        if (j + 2 < nb && !(ok = issue_s(j + 2))) break;
        // P_j written over S_j (and O rescaled) by the softmax warps
        if (!(ok = tc::mbar_wait(p_full0 + 8 * (j % 3), (j / 3) & 1, a.err))) break;
        const int s = j % KS;
        if (!(ok = tc::mbar_wait(v_full0 + 8 * s, (j / KS) & 1, a.err))) break;
        tc::tc_fence_after();
        const uint32_t vbase = tc::smem_u32(smem + Lay::OFF_V + s * Lay::V_BYTES);
#pragma unroll
        for (int kk = 0; kk < BKEY / 16; ++kk)  // 16 keys: 8 TMEM columns of P, two 8-row atoms of V
          tc::mma_f16_tmem_a(tmem + Lay::O_COL, tmem + (j % 3) * BKEY + kk * 8,
                             tc::smem_desc_sw128_mn(vbase + kk * 2048, BKEY * 128, 1024), idO, (j | kk) > 0);
        tc::mma_commit(o_step0 + 8 * (j & 1));
        tc::mma_commit(v_empty0 + 8 * s);
      }
      if (!ok) *s_abort = 1;
      tc::mma_commit(done);  // arrives once every MMA issued above has completed
      tc::mbar_wait(done, 0, a.err);
    }
  } else {
    // ---- softmax: thread = query row r (TMEM lane), keys 64 half .. of every block
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int qpos = a.pos0 + q0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t xb = xb0 + 8 * quarter;
    float* xch = reinterpret_cast<float*>(smem + Lay::OFF_X);  // [block parity][half][row]
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      const int b = j % 3, x = j & 1;  // S/P buffer, exchange slot
      if (*s_abort || !tc::mbar_wait(s_full0 + 8 * b, (j / 3) & 1, a.err)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      uint32_t u[64];
      tc::tmem_ld32_nowait(lane_base + b * BKEY + 64 * half, u);
      tc::tmem_ld32_nowait(lane_base + b * BKEY + 64 * half + 32, u + 32);
      tc::tmem_wait_ld();
      const int k0 = key_block(j) * BKEY + 64 * half;
      if (k0 + 63 > qpos) {  // keys after the row's own position
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (k0 + c > qpos) u[c] = 0xff800000u;
      }
      float bm[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) bm[i] = __uint_as_float(u[i]);
#pragma unroll
      for (int c = 8; c < 64; ++c) bm[c & 7] = fmaxf(bm[c & 7], __uint_as_float(u[c]));
      const float hmx = fmaxf(fmaxf(fmaxf(bm[0], bm[1]), fmaxf(bm[2], bm[3])),
                              fmaxf(fmaxf(bm[4], bm[5]), fmaxf(bm[6], bm[7])));
      // the row maximum of the block: this half's and the partner warp's. A slot is written
      // again two blocks later, after the partner's next arrival, which follows its read.
      xch[(2 * x + half) * BQ + r] = hmx;
      __syncwarp();
      if (lane == 0) mbar_arrive(xb);
      if (!tc::mbar_wait(xb, j & 1, a.err)) {
        ok = false;
        break;
      }
      const float mx = fmaxf(hmx, xch[(2 * x + (half ^ 1)) * BQ + r]);
      // m stays -inf until the row has seen a visible key (then the move, with f = 0, clears
      // the zeros gathered so far)
      const bool move = mx > m + RESCALE_AT;
      if (__any_sync(0xffffffffu, move)) {
        const float f = move ? ex2(m - mx) : 1.f;
        if (j > 0) {
          // O = P_0 V_0 + ... + P_{j-1} V_{j-1} once the last of them is done. Products
          // alternate between two barriers: P_{j-3} V_{j-3} finished before S_j, so the one of
          // P_{j-1} V_{j-1} is at most one phase behind and the parity names it.
          if (!tc::mbar_wait(o_step0 + 8 * ((j - 1) & 1), ((j - 1) >> 1) & 1, a.err)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll
          for (int c = 0; c < HD / 2; c += 32) {
            const uint32_t oc = lane_base + Lay::O_COL + half * (HD / 2) + c;
            uint32_t o[32];
            tc::tmem_ld32_nowait(oc, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
            tc::tmem_st32(oc, o);
          }
        }
        if (move) {
          l *= f;
          m = mx;
        }
      }
      // P = 2^(S - m) as fp16 pairs (key 2c of the half in the low half of column c), written
      // over S (m is -inf only while every key so far was masked: P is 0 then)
      const float mr = m == -INFINITY ? 0.f : m;
      const uint64_t m2 = f2_pack(__float_as_uint(mr), __float_as_uint(mr));
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float d0, d1;
        f2_unpack(f2_sub(f2_pack(u[2 * c], u[2 * c + 1]), m2), d0, d1);
        const float p0 = ex2(d0), p1 = ex2(d1);
        acc[c & 3] = f2_add(acc[c & 3], f2_pack(__float_as_uint(p0), __float_as_uint(p1)));
        u[c] = pack_half2(p0, p1);
      }
      tc::tmem_st32(lane_base + b * BKEY + 32 * half, u);
      float a0, a1, b0, b1, c0, c1, e0, e1;
      f2_unpack(acc[0], a0, a1);
      f2_unpack(acc[1], b0, b1);
      f2_unpack(acc[2], c0, c1);
      f2_unpack(acc[3], e0, e1);
      l += ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (e0 + e1));
      tc::tmem_wait_st();  // P (and a rescaled O) in TMEM before the MMA reads them
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full0 + 8 * b);
    }
    if (ok) ok = tc::mbar_wait(done, 0, a.err);  // the last P V product
    if (ok) {
      tc::tc_fence_after();
      // the row sum: this half's and the partner's (phase nb of the pair's barrier)
      const int b = nb & 1;
      xch[(2 * b + half) * BQ + r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(xb);
      ok = tc::mbar_wait(xb, nb & 1, a.err);
      const float inv = 1.f / (l + xch[(2 * b + (half ^ 1)) * BQ + r]);
      const int row = q0 + r;
      f16* dst = a.Oh + (size_t)row * a.nq * HD + (size_t)h * HD + half * (HD / 2);
#pragma unroll
      for (int c = 0; c < HD / 2; c += 32) {
        uint32_t o[32];
        tc::tmem_ld32_nowait(lane_base + Lay::O_COL + half * (HD / 2) + c, o);
        tc::tmem_wait_ld();
        if (ok && row < a.T) {
#pragma unroll
          for (int d = 0; d < 32; d += 8) {
            uint4 pk;
            pk.x = pack_half2(__uint_as_float(o[d]) * inv, __uint_as_float(o[d + 1]) * inv);
            pk.y = pack_half2(__uint_as_float(o[d + 2]) * inv, __uint_as_float(o[d + 3]) * inv);
            pk.z = pack_half2(__uint_as_float(o[d + 4]) * inv, __uint_as_float(o[d + 5]) * inv);
            pk.w = pack_half2(__uint_as_float(o[d + 6]) * inv, __uint_as_float(o[d + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + c + d) = pk;
          }
        }
      }
    }
    if (!ok) *s_abort = 1;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace fa

bool attn_prefill_tc_supported(int hd) { return hd == 64 || hd == 128; }

cudaError_t attn_prefill_tc_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(fa::attn_prefill_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       fa::L<128>::SMEM);
  if (e) return e;
  return cudaFuncSetAttribute(fa::attn_prefill_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              fa::L<64>::SMEM);
}

cudaError_t attn_prefill_tc(const Dims& d, int T, int pos0, const f16* Qh, const f16* kc, const f16* vc, f16* Oh,
                            int* err, cudaStream_t s) {
  if (!attn_prefill_tc_supported(d.hd) || T < 1 || pos0 < 0 || pos0 + T > d.cap || d.nq % d.nkv)
    return cudaErrorInvalidValue;
  alignas(64) unsigned char mq[128], mk[128], mv[128];
  if (!make_map(mq, Qh, T, d.nq * d.hd, d.nq * d.hd, fa::BQ) ||
      !make_map_kv(mk, kc, d.hd, pos0 + T, d.nkv, d.cap, fa::BKEY) ||
      !make_map_kv(mv, vc, d.hd, pos0 + T, d.nkv, d.cap, fa::BKEY))
    return cudaErrorInvalidValue;
  const int nqb = (T + fa::BQ - 1) / fa::BQ;
  const fa::Args a{T, pos0, d.nq, d.nkv, nqb, Oh, err};
  const CUtensorMap& q = *reinterpret_cast<const CUtensorMap*>(mq);
  const CUtensorMap& k = *reinterpret_cast<const CUtensorMap*>(mk);
  const CUtensorMap& v = *reinterpret_cast<const CUtensorMap*>(mv);
  if (d.hd == 128)
    return launch_k(fa::attn_prefill_tc_kernel<128>, dim3(nqb * d.nq), dim3(fa::THREADS), fa::L<128>::SMEM, s,
                    tc_pdl(), q, k, v, a);
  return launch_k(fa::attn_prefill_tc_kernel<64>, dim3(nqb * d.nq), dim3(fa::THREADS), fa::L<64>::SMEM, s, tc_pdl(),
                  q, k, v, a);
}

}  // namespace qw
