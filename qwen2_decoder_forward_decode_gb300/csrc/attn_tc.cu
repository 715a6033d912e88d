// Causal prefill attention on the 5th-generation tensor cores (tcgen05, TMEM).
//
// "LLM Speedrun: Architecture" (Attention, Causal mask, Grouped Query Attention): query row t
// of head h (position pos0 + t) takes softmax over keys j <= pos0 + t of q . k_j / sqrt(d) and
// the weighted sum of the v_j; head h reads KV head h / (n_heads / n_kv_heads).
//
// One CTA holds two query tiles of 128 rows that read the same keys: two heads of one KV
// group (same rows), or, when a group holds an odd number of heads, two consecutive row
// blocks of one head. Keys stream in blocks of 128 in the online-softmax form:
//   warp 0, lane 0 / 1   TMA producers: the Q tiles, then the key rows (lane 0) and value
//                        rows (lane 1) of each block into their own rings, straight from the
//                        fp16 cache
//   warp 1, lane 0       MMA issuer. Per tile and block j: S_j = Q K_j^T (M 128, N 128 keys)
//                        into the tile's TMEM buffer; once the softmax has written P_j back
//                        over it, O += P_j V_j (M 128, N hd, K 128 keys) with P read straight
//                        from TMEM and V_j MN-major (head dimension contiguous), as the cache
//                        stores it; then S_{j+1} of that tile. The two tiles alternate, so
//                        one tile's products run while the other tile's softmax works.
//   warps 2..5, 6..9     softmax of tile 0 and tile 1, one query row per thread (its TMEM
//                        lane): read S_j, mask keys past the row's position, write P_j =
//                        2^(S_j - m) as fp16 pairs into the first 64 columns of the buffer,
//                        add its row sum to l.
// The reference maximum m of a row moves only when a block's maximum exceeds it by more than
// 8 (base 2): then the warp rescales its rows of O in TMEM (and l) by 2^(m_old - m_new)
// before P_j is released (S_j is complete only after P_{j-1} V_{j-1}, so O is settled).
// Otherwise P stays below 2^8, which fp16 holds with its full relative precision, and O
// accumulates in TMEM untouched. Every term of O and l carries the same factor 2^-m, so
// o / l is the softmax-weighted sum; it goes to the fp16 operand of the o_proj GEMM.
// Each CTA starts at its own key block and wraps around, so that CTAs do not all read the
// same lines at the same time.
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

constexpr int BQ = 128, BKEY = 128, THREADS = 320, TILE_COLS = 256, TMEM_COLS = 512;

template <int HD>
struct L {
  static constexpr int KS_K = HD == 128 ? 3 : 4, KS_V = HD == 128 ? 2 : 3;  // ring depths
  static constexpr int Q_BYTES = BQ * HD * 2;     // per tile: HD / 64 boxes [128 rows][64 columns]
  static constexpr int K_BYTES = BKEY * HD * 2;   // HD / 64 boxes [128 keys][64 columns]
  static constexpr int V_BYTES = BKEY * HD * 2;   // HD / 64 boxes [128 keys][64 columns]
  static constexpr int OFF_K = 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + KS_K * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + KS_V * V_BYTES;
  // q_full, k_full[KS_K], k_empty[KS_K], v_full[KS_V], v_empty[KS_V], s_full[2], p_full[2],
  // done, xb[2 tiles][4 warp pairs]
  static constexpr int NBAR = 1 + 2 * KS_K + 2 * KS_V + 5 + 8;
  static constexpr int OFF_X = OFF_BAR + NBAR * 8 + 16;  // row maxima / sums [tile][half][row]
  // the window must start 1024-byte aligned (the kernel checks): no slack is requested
  static constexpr int SMEM = OFF_X + 2 * 2 * BQ * 4;
  // TMEM columns of tile t, from t * TILE_COLS: S (fp32) / P (fp16 pairs) at 0, O at 128
  static constexpr int SP_COL = 0, O_COL = BKEY;
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(BKEY + HD <= TILE_COLS, "TMEM tile");
};

constexpr float RESCALE_AT = 8.f;  // base-2 growth of a row maximum that moves its reference

struct Args {
  int T, pos0, nq, nkv, nqb;
  int head_pairs;  // 1: tiles are heads 2p, 2p+1 of one row block; 0: row blocks 2p, 2p+1 of one head
  f16* Oh;         // [T][nq * HD]
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
  constexpr int KS_K = Lay::KS_K, KS_V = Lay::KS_V;
  extern __shared__ __align__(1024) uint8_t fa_raw[];
  uint8_t* smem = fa_raw;
  uint64_t* bars = (uint64_t*)(smem + Lay::OFF_BAR);
  uint32_t* tmem_slot = (uint32_t*)(bars + Lay::NBAR);
  volatile int* s_abort = (volatile int*)(tmem_slot + 1);
  const uint32_t q_full = tc::smem_u32(bars);
  const uint32_t k_full0 = q_full + 8, k_empty0 = k_full0 + 8 * KS_K;
  const uint32_t v_full0 = k_empty0 + 8 * KS_K, v_empty0 = v_full0 + 8 * KS_V;
  const uint32_t s_full0 = v_empty0 + 8 * KS_V, p_full0 = s_full0 + 16, done = p_full0 + 16;
  const uint32_t xb0 = done + 8;  // [tile][warp pair]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // the two tiles: head and first row of each; the longest row blocks first
  const int nunit = a.head_pairs ? a.nq / 2 : a.nq;
  const int unit = (int)blockIdx.x % nunit;
  const int pb = (a.head_pairs ? a.nqb : (a.nqb + 1) / 2) - 1 - (int)blockIdx.x / nunit;
  const int head0 = a.head_pairs ? 2 * unit : unit, head1 = a.head_pairs ? 2 * unit + 1 : unit;
  const int q00 = (a.head_pairs ? pb : 2 * pb) * BQ, q01 = (a.head_pairs ? pb : 2 * pb + 1) * BQ;
  // key blocks the CTA reads: up to the last active row; both active tiles take all of them
  // (a row-block pair's first tile finds its last block fully masked)
  const int nb = (a.pos0 + min(a.T, max(q00, q01 < a.T ? q01 : q00) + BQ) - 1) / BKEY + 1;
  const int nblk0 = nb, nblk1 = q01 < a.T ? nb : 0;
  const int g = head0 / (a.nq / a.nkv);
  // CTAs start at different key blocks (and wrap around), so they do not all read the same
  // lines at once; the streaming softmax takes the blocks in any order
  const int rot = (int)((blockIdx.x * 5u) % (unsigned)nb);
  auto key_block = [&](int j) { return j + rot < nb ? j + rot : j + rot - nb; };

  if (tc::smem_u32(fa_raw) & 1023) {  // the swizzled operand tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(a.err, ERR_LAYOUT);
    return;
  }
  // after a timeout anywhere on the stream the remaining CTAs do nothing
  if (threadIdx.x == 0) *s_abort = (*(volatile int*)a.err & ERR_TIMEOUT) != 0;
  __syncthreads();
  if (*s_abort) return;
  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < KS_K; ++s) {
      tc::mbar_init(k_full0 + 8 * s, 1);
      tc::mbar_init(k_empty0 + 8 * s, 1);
    }
    for (int s = 0; s < KS_V; ++s) {
      tc::mbar_init(v_full0 + 8 * s, 1);
      tc::mbar_init(v_empty0 + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      tc::mbar_init(s_full0 + 8 * t, 1);
      tc::mbar_init(p_full0 + 8 * t, 8);  // one arrival per softmax warp
    }
    for (int i = 0; i < 8; ++i) tc::mbar_init(xb0 + 8 * i, 2);  // the two warps of a pair
    tc::mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_slot), TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---- Q tiles, then key blocks
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmQ) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmK) : "memory");
      tc::mbar_expect_tx(q_full, (nblk0 > 0) * Lay::Q_BYTES + (nblk1 > 0) * Lay::Q_BYTES);
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if ((t ? nblk1 : nblk0) > 0)
          for (int c = 0; c < HD / 64; ++c)
            tc::tma_load_2d(tc::smem_u32(smem) + t * Lay::Q_BYTES + c * BQ * 128, &tmQ, q_full,
                            (t ? head1 : head0) * HD + c * 64, t ? q01 : q00);
      int issued = 0;
      for (int j = 0; j < nb; ++j) {
        const int s = j % KS_K;
        if (j >= KS_K && !tc::mbar_wait(k_empty0 + 8 * s, ((j / KS_K) & 1) ^ 1, a.err)) {
          *s_abort = 1;
          break;
        }
        if (*s_abort) break;
        const uint32_t st = tc::smem_u32(smem + Lay::OFF_K + s * Lay::K_BYTES);
        tc::mbar_expect_tx(k_full0 + 8 * s, Lay::K_BYTES);
        for (int c = 0; c < HD / 64; ++c) tc::tma_load_3d(st + c * BKEY * 128, &tmK, k_full0 + 8 * s, c * 64, key_block(j) * BKEY, g);
        ++issued;
      }
      // every copy issued lands before the shared memory is released
      tc::mbar_wait(q_full, 0, a.err);
      for (int j = issued > KS_K ? issued - KS_K : 0; j < issued; ++j)
        tc::mbar_wait(k_full0 + 8 * (j % KS_K), (j / KS_K) & 1, a.err);
    } else if (lane == 1) {
      // ---- value blocks
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmV) : "memory");
      int issued = 0;
      for (int j = 0; j < nb; ++j) {
        const int s = j % KS_V;
        if (j >= KS_V && !tc::mbar_wait(v_empty0 + 8 * s, ((j / KS_V) & 1) ^ 1, a.err)) {
          *s_abort = 1;
          break;
        }
        if (*s_abort) break;
        const uint32_t st = tc::smem_u32(smem + Lay::OFF_V + s * Lay::V_BYTES);
        tc::mbar_expect_tx(v_full0 + 8 * s, Lay::V_BYTES);
        for (int c = 0; c < HD / 64; ++c) tc::tma_load_3d(st + c * BKEY * 128, &tmV, v_full0 + 8 * s, c * 64, key_block(j) * BKEY, g);
        ++issued;
      }
      for (int j = issued > KS_V ? issued - KS_V : 0; j < issued; ++j)
        tc::mbar_wait(v_full0 + 8 * (j % KS_V), (j / KS_V) & 1, a.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      constexpr uint32_t idS = tc::idesc_f16(BQ, BKEY), idO = tc::idesc_f16_bmn(BQ, HD);
      auto issue_s = [&](int t, int j) {  // S_j of tile t (the key block is resident)
        const uint32_t kbase = tc::smem_u32(smem + Lay::OFF_K + (j % KS_K) * Lay::K_BYTES);
        const uint32_t qbase = tc::smem_u32(smem + t * Lay::Q_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc::mma_f16(tmem + t * TILE_COLS + Lay::SP_COL,
                      tc::smem_desc_sw128(qbase + (kk >> 2) * BQ * 128 + (kk & 3) * 32),
                      tc::smem_desc_sw128(kbase + (kk >> 2) * BKEY * 128 + (kk & 3) * 32), idS, kk > 0);
        tc::mma_commit(s_full0 + 8 * t);
      };
      bool ok = tc::mbar_wait(q_full, 0, a.err) && tc::mbar_wait(k_full0, 0, a.err);
      if (ok) {
        tc::tc_fence_after();
        if (nblk0 > 0) issue_s(0, 0);
        if (nblk1 > 0) issue_s(1, 0);
        tc::mma_commit(k_empty0);  // K_0 is free once both products are done
      }
      for (int j = 0; j < nb && ok; ++j) {
        if (*s_abort) {
          ok = false;
          break;
        }
        const bool next = j + 1 < nb;
        const uint32_t vbase = tc::smem_u32(smem + Lay::OFF_V + (j % KS_V) * Lay::V_BYTES);
        bool v_in = false, k_in = false;  // V_j / K_{j+1} waited for
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nbt = t ? nblk1 : nblk0;
          if (!ok || j >= nbt) continue;
          // P_j of tile t written over S_j (and O rescaled) by the softmax warps
          if (!(ok = tc::mbar_wait(p_full0 + 8 * t, j & 1, a.err))) break;
          if (!v_in && !(ok = v_in = tc::mbar_wait(v_full0 + 8 * (j % KS_V), (j / KS_V) & 1, a.err))) break;
          tc::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BKEY / 16; ++kk)  // 16 keys: 8 TMEM columns of P, two 8-row atoms of V
            tc::mma_f16_tmem_a(tmem + t * TILE_COLS + Lay::O_COL, tmem + t * TILE_COLS + Lay::SP_COL + kk * 8,
                               tc::smem_desc_sw128_mn(vbase + kk * 2048, BKEY * 128, 1024), idO, (j | kk) > 0);
          if (j + 1 < nbt) {  // after P_j V_j, which reads the same columns
            if (!k_in) {
              if (!(ok = k_in = tc::mbar_wait(k_full0 + 8 * ((j + 1) % KS_K), ((j + 1) / KS_K) & 1, a.err))) break;
              tc::tc_fence_after();
            }
            issue_s(t, j + 1);
          }
        }
        if (!ok) break;
        tc::mma_commit(v_empty0 + 8 * (j % KS_V));
        if (next) tc::mma_commit(k_empty0 + 8 * ((j + 1) % KS_K));
      }
      if (!ok) *s_abort = 1;
      tc::mma_commit(done);  // arrives once every MMA issued above has completed
      tc::mbar_wait(done, 0, a.err);
    }
  } else {
    // ---- softmax: warps 2..9. The warp pair (w, w + 4) shares TMEM lanes 32 (w % 4) ..
    // +31, one query row per lane: warps 2..5 take keys 0..63 of every block, 6..9 keys
    // 64..127, and the pair trades its halves' maxima (then, at the end, its sums) through
    // shared memory. Both tiles' blocks go through the same warps in turn.
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    float* xch = reinterpret_cast<float*>(smem + Lay::OFF_X);  // [tile][half][row]
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    bool ok = true;
    for (int j = 0; j < nb && ok; ++j) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!ok || j >= (t ? nblk1 : nblk0)) continue;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16) + t * TILE_COLS;
        const int qpos = a.pos0 + (t ? q01 : q00) + r;
        const uint32_t xb = xb0 + 8 * (4 * t + quarter);
        if (*s_abort || !tc::mbar_wait(s_full0 + 8 * t, j & 1, a.err)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        uint32_t u[64];
        tc::tmem_ld32_nowait(lane_base + Lay::SP_COL + 64 * half, u);
        tc::tmem_ld32_nowait(lane_base + Lay::SP_COL + 64 * half + 32, u + 32);
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
        // the row maximum of the block: this half's and the partner warp's. The slot is
        // written again only after every softmax warp released P_j of this tile, which the
        // partner does after reading it.
        xch[(2 * t + half) * BQ + r] = hmx;
        __syncwarp();
        if (lane == 0) mbar_arrive(xb);
        if (!tc::mbar_wait(xb, j & 1, a.err)) {
          ok = false;
          break;
        }
        const float mx = fmaxf(hmx, xch[(2 * t + (half ^ 1)) * BQ + r]);
        // m stays -inf until the row has seen a visible key (then the move, with f = 0, clears
        // the zeros gathered so far)
        const bool move = mx > m[t] + RESCALE_AT;
        if (__any_sync(0xffffffffu, move)) {
          const float f = move ? ex2(m[t] - mx) : 1.f;
          if (j > 0) {  // O holds P_0 V_0 + ... + P_{j-1} V_{j-1}: settled before S_j completed
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
            l[t] *= f;
            m[t] = mx;
          }
        }
        // P = 2^(S - m) as fp16 pairs (key 2c of the half in the low half of column c),
        // written over S (m is -inf only while every key so far was masked: P is 0 then)
        const float mr = m[t] == -INFINITY ? 0.f : m[t];
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
        tc::tmem_st32(lane_base + Lay::SP_COL + 32 * half, u);
        float a0, a1, b0, b1, c0, c1, e0, e1;
        f2_unpack(acc[0], a0, a1);
        f2_unpack(acc[1], b0, b1);
        f2_unpack(acc[2], c0, c1);
        f2_unpack(acc[3], e0, e1);
        l[t] += ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (e0 + e1));
        tc::tmem_wait_st();  // P (and a rescaled O) in TMEM before the MMA reads them
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full0 + 8 * t);
      }
    }
    if (ok) ok = tc::mbar_wait(done, 0, a.err);  // the last P V products
    if (ok) tc::tc_fence_after();
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (!ok || (t ? nblk1 : nblk0) == 0) continue;
      // the row sum: this half's and the partner's (phase nb of the pair's barrier)
      const uint32_t xb = xb0 + 8 * (4 * t + quarter);
      xch[(2 * t + half) * BQ + r] = l[t];
      __syncwarp();
      if (lane == 0) mbar_arrive(xb);
      if (!(ok = tc::mbar_wait(xb, nb & 1, a.err))) break;
      const float inv = 1.f / (l[t] + xch[(2 * t + (half ^ 1)) * BQ + r]);
      const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16) + t * TILE_COLS;
      const int row = (t ? q01 : q00) + r;
      f16* dst = a.Oh + (size_t)row * a.nq * HD + (size_t)(t ? head1 : head0) * HD + half * (HD / 2);
#pragma unroll
      for (int c = 0; c < HD / 2; c += 32) {
        uint32_t o[32];
        tc::tmem_ld32_nowait(lane_base + Lay::O_COL + half * (HD / 2) + c, o);
        tc::tmem_wait_ld();
        if (row < a.T) {
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
  // two heads of a KV group per CTA when the group holds an even number, else two row blocks
  const int head_pairs = (d.nq / d.nkv) % 2 == 0;
  const fa::Args a{T, pos0, d.nq, d.nkv, nqb, head_pairs, Oh, err};
  const int grid = head_pairs ? nqb * (d.nq / 2) : ((nqb + 1) / 2) * d.nq;
  const CUtensorMap& q = *reinterpret_cast<const CUtensorMap*>(mq);
  const CUtensorMap& k = *reinterpret_cast<const CUtensorMap*>(mk);
  const CUtensorMap& v = *reinterpret_cast<const CUtensorMap*>(mv);
  if (d.hd == 128)
    fa::attn_prefill_tc_kernel<128><<<grid, fa::THREADS, fa::L<128>::SMEM, s>>>(q, k, v, a);
  else
    fa::attn_prefill_tc_kernel<64><<<grid, fa::THREADS, fa::L<64>::SMEM, s>>>(q, k, v, a);
  return cudaGetLastError();
}

}  // namespace qw
