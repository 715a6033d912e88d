// Causal prefill attention on the 5th-generation tensor cores (tcgen05, TMEM).
//
// "LLM Speedrun: Architecture" (Attention, Causal mask, Grouped Query Attention): query row t
// of head h (position pos0 + t) takes softmax over keys j <= pos0 + t of q . k_j / sqrt(d) and
// the weighted sum of the v_j; head h reads KV head h / (n_heads / n_kv_heads).
//
// One CTA per (128 query rows, head); keys stream in blocks of 64 in the online-softmax form
// (running maximum m and sum l per row):
//   warp 0, one lane   TMA producer: the Q tile once, then the key and value rows of each
//                      block into a KSTAGES-deep ring, straight from the fp16 cache
//   warp 1, one lane   MMA issuer: S_j = Q K_j^T (M 128, N 64) into one of two TMEM buffers;
//                      after the softmax has written P_j, O_j = P_j V_j (M 128, N hd) into one
//                      of two more. S_{j+1} is issued before waiting for P_j, so the tensor
//                      cores work while the softmax runs. V_j is read MN-major (head
//                      dimension contiguous), as the cache stores it.
//   warps 2..5         softmax, one query row per thread (its TMEM lane): read S_j, mask keys
//                      past the row's position, update m and l, write P_j = 2^(S_j - m) as
//                      fp16 into shared memory in the 128-byte-swizzled K-major layout the
//                      MMA reads, and fold O_{j-1} into registers: o = o * 2^(m_old - m) + O.
//                      At the end o / l goes to the fp16 operand of the o_proj GEMM.
// Q arrives in fp16, already multiplied by log2(e) / sqrt(d), so scores are in base 2.
// Every mbarrier wait is bounded: on expiry the thread flags ERR_TIMEOUT, the CTA stops
// issuing work, waits (bounded) for what it issued, and releases its TMEM.
#include <cuda.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace qw {
namespace fa {

constexpr int BQ = 128, BKEY = 64, KSTAGES = 3, THREADS = 192;

template <int HD>
struct L {
  static constexpr int Q_BYTES = BQ * HD * 2;     // HD / 64 boxes [128 rows][64 columns]
  static constexpr int K_BYTES = BKEY * HD * 2;   // HD / 64 boxes [64 keys][64 columns]
  static constexpr int V_BYTES = BKEY * HD * 2;   // HD / 64 boxes [64 keys][64 columns]
  static constexpr int STAGE = K_BYTES + V_BYTES;
  static constexpr int P_BYTES = BQ * BKEY * 2;   // [128 rows][64 keys]
  static constexpr int OFF_STAGE = Q_BYTES;
  static constexpr int OFF_P = OFF_STAGE + KSTAGES * STAGE;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  // q_full, kv_full[KSTAGES], kv_empty[KSTAGES], s_full[2], p_full[2], o_full[2], done
  static constexpr int NBAR = 2 + 2 * KSTAGES + 6;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
  // TMEM columns: S buffers at 0 and BKEY, O buffers at 2 BKEY and 2 BKEY + HD
  static constexpr int S_COL = 0, O_COL = 2 * BKEY;
  static constexpr int TMEM_COLS = 2 * BKEY + 2 * HD <= 256 ? 256 : 512;
};

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

template <int HD>
__global__ void __launch_bounds__(THREADS, 1)
attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const Args a) {
  using Lay = L<HD>;
  extern __shared__ uint8_t fa_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)fa_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + Lay::OFF_BAR);
  uint32_t* tmem_slot = (uint32_t*)(bars + Lay::NBAR);
  volatile int* s_abort = (volatile int*)(tmem_slot + 1);
  const uint32_t q_full = tc::smem_u32(bars);
  const uint32_t kv_full0 = q_full + 8, kv_empty0 = kv_full0 + 8 * KSTAGES;
  const uint32_t s_full0 = kv_empty0 + 8 * KSTAGES, p_full0 = s_full0 + 16, o_full0 = p_full0 + 16;
  const uint32_t done = o_full0 + 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the longest (last) query blocks of every head first
  const int qb = a.nqb - 1 - (int)blockIdx.x / a.nq, h = (int)blockIdx.x % a.nq;
  const int g = h / (a.nq / a.nkv);
  const int q0 = qb * BQ;
  const int last_pos = a.pos0 + min(a.T, q0 + BQ) - 1;
  const int nblk = last_pos / BKEY + 1;  // key blocks some row of this tile sees

  // after a timeout anywhere on the stream the remaining CTAs do nothing
  if (threadIdx.x == 0) *s_abort = (*(volatile int*)a.err & ERR_TIMEOUT) != 0;
  __syncthreads();
  if (*s_abort) return;
  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < KSTAGES; ++s) {
      tc::mbar_init(kv_full0 + 8 * s, 1);
      tc::mbar_init(kv_empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(s_full0 + 8 * b, 1);
      tc::mbar_init(p_full0 + 8 * b, 128);
      tc::mbar_init(o_full0 + 8 * b, 1);
    }
    tc::mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_slot), Lay::TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmQ) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmK) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmV) : "memory");
      tc::mbar_expect_tx(q_full, Lay::Q_BYTES);
      for (int c = 0; c < HD / 64; ++c)
        tc::tma_load_2d(tc::smem_u32(smem) + c * BQ * 128, &tmQ, q_full, h * HD + c * 64, q0);
      int issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int s = j % KSTAGES;
        if (j >= KSTAGES && !tc::mbar_wait(kv_empty0 + 8 * s, ((j / KSTAGES) & 1) ^ 1, a.err)) {
          *s_abort = 1;
          break;
        }
        if (*s_abort) break;
        const uint32_t st = tc::smem_u32(smem + Lay::OFF_STAGE + s * Lay::STAGE);
        tc::mbar_expect_tx(kv_full0 + 8 * s, Lay::STAGE);
        for (int c = 0; c < HD / 64; ++c) {
          tc::tma_load_3d(st + c * BKEY * 128, &tmK, kv_full0 + 8 * s, c * 64, j * BKEY, g);
          tc::tma_load_3d(st + Lay::K_BYTES + c * BKEY * 128, &tmV, kv_full0 + 8 * s, c * 64, j * BKEY, g);
        }
        ++issued;
      }
      // every copy this CTA issued lands before its shared memory is released
      tc::mbar_wait(q_full, 0, a.err);
      for (int j = issued > KSTAGES ? issued - KSTAGES : 0; j < issued; ++j)
        tc::mbar_wait(kv_full0 + 8 * (j % KSTAGES), (j / KSTAGES) & 1, a.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      constexpr uint32_t idS = tc::idesc_f16(BQ, BKEY), idO = tc::idesc_f16_bmn(BQ, HD);
      const uint32_t qbase = tc::smem_u32(smem);
      bool ok = tc::mbar_wait(q_full, 0, a.err);
      auto issue_s = [&](int j) -> bool {  // S_j into S buffer j % 2
        const int s = j % KSTAGES;
        if (!tc::mbar_wait(kv_full0 + 8 * s, (j / KSTAGES) & 1, a.err)) return false;
        tc::tc_fence_after();
        const uint32_t kbase = tc::smem_u32(smem + Lay::OFF_STAGE + s * Lay::STAGE);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc::mma_f16(tmem + Lay::S_COL + (j & 1) * BKEY,
                      tc::smem_desc_sw128(qbase + (kk >> 2) * BQ * 128 + (kk & 3) * 32),
                      tc::smem_desc_sw128(kbase + (kk >> 2) * BKEY * 128 + (kk & 3) * 32), idS, kk > 0);
        tc::mma_commit(s_full0 + 8 * (j & 1));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nblk && ok; ++j) {
        if (*s_abort) {
          ok = false;
          break;
        }
        if (j + 1 < nblk && !(ok = issue_s(j + 1))) break;
        // P_j written, S_j and O_{j-2} read by all 128 softmax threads
        if (!(ok = tc::mbar_wait(p_full0 + 8 * (j & 1), (j >> 1) & 1, a.err))) break;
        tc::tc_fence_after();
        const uint32_t pbase = tc::smem_u32(smem + Lay::OFF_P + (j & 1) * Lay::P_BYTES);
        const uint32_t vbase = tc::smem_u32(smem + Lay::OFF_STAGE + (j % KSTAGES) * Lay::STAGE + Lay::K_BYTES);
#pragma unroll
        for (int kk = 0; kk < BKEY / 16; ++kk)  // 16 keys: two 8-row atoms of every column box
          tc::mma_f16(tmem + Lay::O_COL + (j & 1) * HD, tc::smem_desc_sw128(pbase + kk * 32),
                      tc::smem_desc_sw128_mn(vbase + kk * 2048, BKEY * 128, 1024), idO, kk > 0);
        tc::mma_commit(o_full0 + 8 * (j & 1));
        tc::mma_commit(kv_empty0 + 8 * (j % KSTAGES));
      }
      if (!ok) *s_abort = 1;
      tc::mma_commit(done);  // arrives once every MMA issued above has completed
      tc::mbar_wait(done, 0, a.err);
    }
  } else {
    // ---- softmax: thread = query row r, TMEM lane 32 (warp % 4) + lane
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qpos = a.pos0 + q0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    float o[HD];
#pragma unroll
    for (int d = 0; d < HD; ++d) o[d] = 0.f;
    float m = -INFINITY, l = 0.f, corr_pend = 0.f;
    bool ok = true;
    auto take_o = [&](int j) -> bool {  // o = o * corr(j) + O_j
      if (!tc::mbar_wait(o_full0 + 8 * (j & 1), (j >> 1) & 1, a.err)) return false;
      tc::tc_fence_after();
#pragma unroll
      for (int c = 0; c < HD; c += 32) {
        float v[32];
        tc::tmem_ld32(lane_base + Lay::O_COL + (j & 1) * HD + c, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c + i] = fmaf(o[c + i], corr_pend, v[i]);
      }
      return true;
    };
    for (int j = 0; j < nblk; ++j) {
      if (*s_abort || !tc::mbar_wait(s_full0 + 8 * (j & 1), (j >> 1) & 1, a.err)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      float sv[BKEY];
      tc::tmem_ld32(lane_base + Lay::S_COL + (j & 1) * BKEY, sv);
      tc::tmem_ld32(lane_base + Lay::S_COL + (j & 1) * BKEY + 32, sv + 32);
      const int k0 = j * BKEY;
      if (k0 + BKEY - 1 > qpos) {  // keys after the row's own position
#pragma unroll
        for (int c = 0; c < BKEY; ++c)
          if (k0 + c > qpos) sv[c] = -INFINITY;
      }
      float mx = m;
#pragma unroll
      for (int c = 0; c < BKEY; ++c) mx = fmaxf(mx, sv[c]);
      // block 0 holds key 0, which every row sees: m is finite from then on
      const float corr = ex2(m - mx);  // 0 on block 0 (m = -inf)
      float sum = 0.f;
      uint8_t* prow = smem + Lay::OFF_P + (j & 1) * Lay::P_BYTES + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int c8 = 0; c8 < BKEY / 8; ++c8) {
        float pv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          pv[i] = ex2(sv[c8 * 8 + i] - mx);
          sum += pv[i];
        }
        uint4 pk;
        pk.x = pack_half2(pv[0], pv[1]);
        pk.y = pack_half2(pv[2], pv[3]);
        pk.z = pack_half2(pv[4], pv[5]);
        pk.w = pack_half2(pv[6], pv[7]);
        *reinterpret_cast<uint4*>(prow + ((c8 ^ (r & 7)) << 4)) = pk;  // 128-byte swizzle
      }
      l = fmaf(l, corr, sum);
      m = mx;
      // P stores visible to the tensor cores; S and O reads complete
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc::tc_fence_before();
      mbar_arrive(p_full0 + 8 * (j & 1));
      if (j >= 1 && !(ok = take_o(j - 1))) break;
      corr_pend = corr;
    }
    if (ok) ok = take_o(nblk - 1);
    if (ok && q0 + r < a.T) {
      const float inv = 1.f / l;
      f16* dst = a.Oh + (size_t)(q0 + r) * a.nq * HD + (size_t)h * HD;
#pragma unroll
      for (int d = 0; d < HD; d += 8) {
        uint4 pk;
        pk.x = pack_half2(o[d] * inv, o[d + 1] * inv);
        pk.y = pack_half2(o[d + 2] * inv, o[d + 3] * inv);
        pk.z = pack_half2(o[d + 4] * inv, o[d + 5] * inv);
        pk.w = pack_half2(o[d + 6] * inv, o[d + 7] * inv);
        *reinterpret_cast<uint4*>(dst + d) = pk;
      }
    }
    if (!ok) *s_abort = 1;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, Lay::TMEM_COLS);
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
  if (!make_map(mq, Qh, T, d.nq * d.hd, d.nq * d.hd, fa::BQ) || !make_map_kv(mk, kc, d.hd, pos0 + T, d.nkv, d.cap) ||
      !make_map_kv(mv, vc, d.hd, pos0 + T, d.nkv, d.cap))
    return cudaErrorInvalidValue;
  const int nqb = (T + fa::BQ - 1) / fa::BQ;
  const fa::Args a{T, pos0, d.nq, d.nkv, nqb, Oh, err};
  const dim3 grid(nqb * d.nq), block(fa::THREADS);
  const CUtensorMap& q = *reinterpret_cast<const CUtensorMap*>(mq);
  const CUtensorMap& k = *reinterpret_cast<const CUtensorMap*>(mk);
  const CUtensorMap& v = *reinterpret_cast<const CUtensorMap*>(mv);
  if (d.hd == 128)
    fa::attn_prefill_tc_kernel<128><<<grid, block, fa::L<128>::SMEM, s>>>(q, k, v, a);
  else
    fa::attn_prefill_tc_kernel<64><<<grid, block, fa::L<64>::SMEM, s>>>(q, k, v, a);
  return cudaGetLastError();
}

}  // namespace qw
