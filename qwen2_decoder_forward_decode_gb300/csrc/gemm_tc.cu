// Prefill GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   C[M, N] = A[M, K] . B[N, K]^T     A: fp16 activations, B: fp16 weights, both K-major
//
// A persistent CTA per SM computes 128 x BN tiles into two TMEM fp32 accumulators:
//   warp 0 (one lane)  TMA producer: 128-byte-swizzled A and B tiles of 64 K-elements into
//                      a shared-memory ring of 4 to 8 stages, as many as fit (mbarrier
//                      full/empty pairs)
//   warp 1 (one lane)  MMA issuer: tcgen05.mma.cta_group::1.kind::f16, M=128, N=BN, K=16,
//                      four per stage; tcgen05.commit frees a stage when its MMAs retire
//   warps 2..9         epilogue: tcgen05.ld of their 32 TMEM lanes (= tile rows; warps w and
//                      w + 4 split the columns), fused bias / residual-add / SwiGLU / q|k|v
//                      RoPE and KV append, stores to global memory, while the next tile
//                      accumulates in the other buffer
// With two or more row tiles, CTA pairs (clusters of two) run the same roles on 256 x BN
// tiles with the pair form of the MMA (cta_group::2), each CTA staging half of B.
// Launched with programmatic dependent launch (the prefill), a CTA requests the B (weight)
// tiles of its first stages before it waits for the previous kernel, then A.
// Every mbarrier wait is bounded (clock budget); on expiry the CTA flags ERR_TIMEOUT,
// stops issuing work, and still releases its TMEM.
#include <cuda.h>

#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace qw {

namespace tc {

constexpr int BM = 128, BK = 64;
constexpr int THREADS = 320;  // producer, MMA issuer, eight epilogue warps

}  // namespace tc

// Epilogues
enum : int { EPI_STORE = 0, EPI_ADD = 1, EPI_SWIGLU = 2, EPI_QKV = 3 };

struct TcEpi {
  float* C;          // EPI_STORE: C = acc (+ bias); EPI_ADD: C += acc   (fp32, ld = ldc)
  const bf16* bias;  // [N] or null (EPI_STORE, EPI_QKV)
  f16* Cb;           // EPI_SWIGLU: Cb[m][n] = silu(gate) * up as fp16, ld = ldc
  int ldc;
  QkvOut qkv;        // EPI_QKV: + bias, RoPE of adjacent column pairs, fp16 q and K/V rows
};

// Persistent: grid = min(units, SMs); CTA c takes work units c, c + grid, ... in order, a unit
// being one 128 x BN output tile (of one K range under split-K). The producer streams the
// A and B blocks of consecutive units through one ring without a pause, the MMA warp
// accumulates unit i into TMEM buffer i % 2 (2 x BN columns), and the epilogue warps drain
// unit i while the MMAs of unit i + 1 run.
// BN columns per tile. For EPI_SWIGLU the B ring holds BN/2 gate rows then BN/2 up rows of
// the same output columns, so one N = BN product leaves gate in accumulator columns
// [0, BN/2) and up in [BN/2, BN).
// Split-K (splits > 1): unit z of a tile covers a contiguous range of K blocks and stores its
// raw fp32 tile to ws[z]; a reduce kernel then adds the splits in order and applies the bias,
// the residual add, SwiGLU, or the q|k|v bias, RoPE and KV append (deterministic).
// CL = 2: a cluster of two CTAs (one per SM) computes a 256 x BN tile with the pair form of
// the MMA (tcgen05 cta_group::2, M = 256): each CTA stages its 128 rows of A and its half of
// the BN rows of B, so an SM takes in a third fewer operand bytes per FLOP, and the stage
// ring gets deeper. The even CTA's MMA thread issues for both; its full barriers count the
// bytes landing in both CTAs, its commits free both CTAs' stages and hand each CTA's
// epilogue its 128 accumulator rows, and both CTAs' epilogue warps release its
// accumulators.
struct TcGrid {
  int tiles_m, tiles_n, splits;
};

template <int BN, int CL>
__host__ __device__ constexpr size_t tc_stage_bytes() {
  return (size_t)tc::BM * tc::BK * 2 + (size_t)(CL == 2 ? BN / 2 : BN) * tc::BK * 2;
}
// as many stages as fit beside the barriers, the epilogue scratch and the alignment slack (at
// most 8): narrow tiles keep more weight bytes in flight
template <int BN, int CL>
__host__ __device__ constexpr int tc_stages() {
  return (232448 - 256 - 8 * 32 * 33 * 4 - 1024) / tc_stage_bytes<BN, CL>() < 8
             ? (int)((232448 - 256 - 8 * 32 * 33 * 4 - 1024) / tc_stage_bytes<BN, CL>())
             : 8;
}
// ring, barriers (256 B), epilogue scratch (8 warps x 32 x 33 floats), 1024-B alignment slack
template <int BN, int CL>
__host__ __device__ constexpr size_t tc_smem() {
  return tc_stages<BN, CL>() * tc_stage_bytes<BN, CL>() + 256 + 8 * 32 * 33 * 4 + 1024;
}

// EPI_QKV epilogue of one thread: v holds row `row` of the 32 columns col0 .. col0 + 31 (of
// q | k | v, pair order: columns 2i and 2i + 1 of a head are the rotation pair (a, b) of
// head columns i and i + hd/2). Adds the bias, rotates q and k rows by the position's
// (cos, sin): a' = a cos - b sin, b' = b cos + a sin, and stores fp16 at head columns i and
// i + hd/2 of Qh (times qscale) or of the K or V cache row at position pos0 + row.
__device__ __forceinline__ void qkv_row(const TcEpi& ep, const float* v, int col0, int N, int row, int M,
                                        int* err) {
  const QkvOut& o = ep.qkv;
  if (row >= M) return;
  const int hd = o.hd, half = hd >> 1;
  bool bad = false;  // a value fp16 cannot hold
  if ((hd & 31) == 0) {  // the 32 columns lie in one head: 16 pairs, vector loads and stores
    if (col0 >= N) return;
    const int head = col0 / hd, i0 = (col0 - head * hd) >> 1;
    const bool rot = head < o.nq + o.nkv;
    float a[16], b[16];
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      a[p] = v[2 * p];
      b[p] = v[2 * p + 1];
    }
    if (ep.bias) {
      const uint4* bp = reinterpret_cast<const uint4*>(ep.bias + col0);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 w = __ldg(bp + q4);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[k]));
          a[4 * q4 + k] += f.x;
          b[4 * q4 + k] += f.y;
        }
      }
    }
    float scale = 1.f;
    f16* dst;
    if (head < o.nq) {
      dst = o.Qh + (size_t)row * o.nq * hd + (size_t)head * hd;
      scale = o.qscale;
    } else {
      const int hh = rot ? head - o.nq : head - o.nq - o.nkv;
      dst = (rot ? o.kc : o.vc) + ((size_t)hh * o.cap + o.pos0 + row) * hd;
    }
    if (rot) {
      const float4* cp = reinterpret_cast<const float4*>(o.rope + (size_t)(o.pos0 + row) * half + i0);
#pragma unroll
      for (int q2 = 0; q2 < 8; ++q2) {
        const float4 c2 = __ldg(cp + q2);  // (cos, sin) of pairs 2 q2 and 2 q2 + 1
        const int p = 2 * q2;
        const float ra = a[p] * c2.x - b[p] * c2.y, rb = b[p] * c2.x + a[p] * c2.y;
        const float sa = a[p + 1] * c2.z - b[p + 1] * c2.w, sb = b[p + 1] * c2.z + a[p + 1] * c2.w;
        a[p] = ra;
        b[p] = rb;
        a[p + 1] = sa;
        b[p + 1] = sb;
      }
    }
    uint32_t ha[8], hb[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float x0 = a[2 * k] * scale, x1 = a[2 * k + 1] * scale;
      const float y0 = b[2 * k] * scale, y1 = b[2 * k + 1] * scale;
      bad |= !(fabsf(x0) < 65520.f) || !(fabsf(x1) < 65520.f) || !(fabsf(y0) < 65520.f) || !(fabsf(y1) < 65520.f);
      const __half2 hx = __floats2half2_rn(x0, x1), hy = __floats2half2_rn(y0, y1);
      ha[k] = *reinterpret_cast<const uint32_t*>(&hx);
      hb[k] = *reinterpret_cast<const uint32_t*>(&hy);
    }
    uint4* da = reinterpret_cast<uint4*>(dst + i0);
    uint4* db = reinterpret_cast<uint4*>(dst + i0 + half);
    da[0] = make_uint4(ha[0], ha[1], ha[2], ha[3]);
    da[1] = make_uint4(ha[4], ha[5], ha[6], ha[7]);
    db[0] = make_uint4(hb[0], hb[1], hb[2], hb[3]);
    db[1] = make_uint4(hb[4], hb[5], hb[6], hb[7]);
  } else {  // any even head size: pair by pair
    for (int p = 0; p < 16; ++p) {
      const int col = col0 + 2 * p;
      if (col >= N) break;
      float x = v[2 * p], y = v[2 * p + 1];
      if (ep.bias) {
        x += to_f32(ep.bias[col]);
        y += to_f32(ep.bias[col + 1]);
      }
      const int head = col / hd, i = (col - head * hd) >> 1;
      float scale = 1.f;
      f16* dst;
      if (head < o.nq + o.nkv) {
        const float2 cs = o.rope[(size_t)(o.pos0 + row) * half + i];
        const float rx = x * cs.x - y * cs.y, ry = y * cs.x + x * cs.y;
        x = rx;
        y = ry;
      }
      if (head < o.nq) {
        dst = o.Qh + (size_t)row * o.nq * hd + (size_t)head * hd;
        scale = o.qscale;
      } else {
        const bool is_k = head < o.nq + o.nkv;
        const int hh = is_k ? head - o.nq : head - o.nq - o.nkv;
        dst = (is_k ? o.kc : o.vc) + ((size_t)hh * o.cap + o.pos0 + row) * hd;
      }
      x *= scale;
      y *= scale;
      bad |= !(fabsf(x) < 65520.f) || !(fabsf(y) < 65520.f);
      dst[i] = __float2half_rn(x);
      dst[i + half] = __float2half_rn(y);
    }
  }
  if (bad) atomicOr(err, ERR_RANGE);
}

template <int BN, int EPI, int CL>
__global__ void __launch_bounds__(tc::THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmB2, TcEpi ep, int M, int N, int K, int* err, TcGrid g,
               float* ws) {
  using namespace tc;
  constexpr int A_BYTES = BM * BK * 2;
  constexpr int B_BYTES = (CL == 2 ? BN / 2 : BN) * BK * 2;  // this CTA's rows of B
  constexpr int STAGE = A_BYTES + B_BYTES;
  constexpr int STAGES = tc_stages<BN, CL>();
  static_assert(tc_smem<BN, CL>() <= 232448, "shared memory");
  constexpr int NOUT = EPI == EPI_SWIGLU ? BN / 2 : BN;  // output columns per tile
  extern __shared__ uint8_t smem_raw[];
  // launched with programmatic dependent launch: the next kernel may be scheduled once every
  // CTA of this one runs (it waits for this grid's completion before touching its outputs)
  pdl_trigger();
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + STAGES * STAGE);
  uint32_t* tmem_slot = (uint32_t*)(bars + 2 * STAGES + 4);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t acc_full0 = smem_u32(bars + 2 * STAGES), acc_empty0 = acc_full0 + 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CL = 2: a unit is a pair of row tiles, the cluster's CTAs take one each (rank)
  const int rank = CL == 2 ? (int)tc::cluster_ctarank() : 0;
  const int tiles_mu = (g.tiles_m + CL - 1) / CL;  // row units
  const int tiles = tiles_mu * g.tiles_n, units = tiles * g.splits;
  const int first = (int)blockIdx.x / CL, step = (int)gridDim.x / CL;
  const int nk_all = (K + BK - 1) / BK;
  // unit -> first row, first output column, split index, K block range
  auto unit_of = [&](int u, int& m0, int& n0, int& z, int& kb_lo, int& kb_hi) {
    z = u / tiles;
    const int t = u - z * tiles;
    m0 = ((t % tiles_mu) * CL + rank) * BM;
    n0 = (t / tiles_mu) * NOUT;
    kb_lo = (int)((long long)z * nk_all / g.splits);
    kb_hi = (int)((long long)(z + 1) * nk_all / g.splits);
  };
  __shared__ int s_abort;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(full0 + 8 * s, 1);
      tc::mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(acc_full0 + 8 * b, 1);
      tc::mbar_init(acc_empty0 + 8 * b, 8 * CL);  // one arrival per epilogue warp of the pair
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  constexpr uint32_t TCOLS = 2 * BN <= 256 ? 256 : 512;  // two accumulators, a power of two
  if (warp == 0) {
    if (CL == 2) tc::tmem_alloc_pair(smem_u32(tmem_slot), TCOLS);
    else tc::tmem_alloc(smem_u32(tmem_slot), TCOLS);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (CL == 2) tc::cluster_sync();  // the pair's barriers exist before either CTA signals one
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer: the K blocks of this CTA's units, back to back
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
    // stage s of K block kb of the unit at (m0, n0): the byte count, then A and/or B
    auto issue = [&](int s, int kb, int m0, int n0, bool load_a, bool load_b) {
      const uint32_t a_dst = smem_u32(smem + s * STAGE);
      const uint32_t b_dst = a_dst + A_BYTES;
      if (CL == 2) {  // bytes counted on the even CTA's barrier (SwiGLU: rank 0 gate, rank 1 up)
        const uint32_t bar = tc::mapa_shared(full0 + 8 * s, 0);
        if (load_b && rank == 0) tc::mbar_expect_tx(full0 + 8 * s, 2 * STAGE);
        if (load_a) tc::tma_load_2d_pair(a_dst, &tmA, bar, kb * BK, m0);
        if (load_b) {
          if (EPI == EPI_SWIGLU)
            tc::tma_load_2d_pair(b_dst, rank ? &tmB2 : &tmB, bar, kb * BK, n0);
          else
            tc::tma_load_2d_pair(b_dst, &tmB, bar, kb * BK, n0 + rank * (BN / 2));
        }
        return;
      }
      if (load_b) tc::mbar_expect_tx(full0 + 8 * s, STAGE);
      if (load_a) tc::tma_load_2d(a_dst, &tmA, full0 + 8 * s, kb * BK, m0);
      if (load_b) {
        if (EPI == EPI_SWIGLU) {
          tc::tma_load_2d(b_dst, &tmB, full0 + 8 * s, kb * BK, n0);
          tc::tma_load_2d(b_dst + B_BYTES / 2, &tmB2, full0 + 8 * s, kb * BK, n0);
        } else {
          tc::tma_load_2d(b_dst, &tmB, full0 + 8 * s, kb * BK, n0);
        }
      }
    };
    // The weights (B) of the first stages are requested before waiting for the kernel that
    // writes A; A follows once that kernel's grid is complete.
    int pre = 0, pre_m0[STAGES], pre_n0[STAGES], pre_kb[STAGES];
    for (int u = first; u < units && pre < STAGES; u += step) {
      int m0, n0, z, kb_lo, kb_hi;
      unit_of(u, m0, n0, z, kb_lo, kb_hi);
      for (int kb = kb_lo; kb < kb_hi && pre < STAGES; ++kb, ++pre) {
        pre_m0[pre] = m0;
        pre_n0[pre] = n0;
        pre_kb[pre] = kb;
        issue(pre, kb, m0, n0, false, true);
      }
    }
    pdl_wait();
    for (int j = 0; j < pre; ++j) issue(j, pre_kb[j], pre_m0[j], pre_n0[j], true, false);
    int it = 0;  // K blocks issued
    for (int u = first; u < units && !s_abort; u += step) {
      int m0, n0, z, kb_lo, kb_hi;
      unit_of(u, m0, n0, z, kb_lo, kb_hi);
      for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
        if (it < pre) continue;  // issued above
        const int s = it % STAGES;
        if (it >= STAGES && !tc::mbar_wait(empty0 + 8 * s, ((it / STAGES) & 1) ^ 1, err)) { s_abort = 1; break; }
        if (s_abort) break;
        issue(s, kb, m0, n0, true, true);
      }
    }
    // drain: every issued stage must land before the CTA may exit (the odd CTA's bytes are
    // counted on the even CTA's barriers, which drains them before the closing cluster barrier)
    if (rank == 0)
      for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
        tc::mbar_wait(full0 + 8 * (j % STAGES), (j / STAGES) & 1, err);
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---- MMA issuer: one N = BN product per 16 K (gate and up together for SwiGLU)
    constexpr uint32_t idesc = tc::idesc_f16(CL * BM, BN);
    int it = 0, i = 0;  // K blocks consumed, units done
    bool ok = true;
    for (int u = first; u < units && ok; u += step, ++i) {
      int m0, n0, z, kb_lo, kb_hi;
      unit_of(u, m0, n0, z, kb_lo, kb_hi);
      const int b = i & 1;
      // the epilogue has drained this accumulator's previous unit
      if (i >= 2 && !tc::mbar_wait(acc_empty0 + 8 * b, ((i >> 1) & 1) ^ 1, err)) { ok = false; break; }
      tc::tc_fence_after();
      for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
        const int s = it % STAGES;
        if (!tc::mbar_wait(full0 + 8 * s, (it / STAGES) & 1, err)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t a_base = smem_u32(smem + s * STAGE);
        const uint32_t b_base = a_base + A_BYTES;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t da = tc::smem_desc_sw128(a_base + 32 * k), db = tc::smem_desc_sw128(b_base + 32 * k);
          if (CL == 2) tc::mma_f16_pair(tmem + b * BN, da, db, idesc, (kb > kb_lo) || k);
          else tc::mma_f16(tmem + b * BN, da, db, idesc, (kb > kb_lo) || k);
        }
        if (CL == 2) tc::mma_commit_pair(empty0 + 8 * s, 3);  // the stage is free in both CTAs
        else tc::mma_commit(empty0 + 8 * s);
      }
      if (!ok) break;
      if (CL == 2) tc::mma_commit_pair(acc_full0 + 8 * b, 3);
      else tc::mma_commit(acc_full0 + 8 * b);
    }
    if (!ok) s_abort = 1;
  } else if (warp >= 2) {
    // ---- epilogue: warp w reads TMEM lanes 32*(w%4) .. +31, columns of half (w-2)/4
    const int q = warp & 3, eh = (warp - 2) >> 2;
    pdl_wait();  // outputs (and C) belong to this kernel only once the previous grid is done
    int i = 0;
    for (int u = first; u < units; u += step, ++i) {
      int m0, n0, z, kb_lo, kb_hi;
      unit_of(u, m0, n0, z, kb_lo, kb_hi);
      const int b = i & 1;
      if (!tc::mbar_wait(acc_full0 + 8 * b, (i >> 1) & 1, err)) break;
      tc::tc_fence_after();
      const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + b * BN;
      // Each 32 x 32 block goes through the warp's shared-memory scratch (row stride 33 words,
      // conflict-free both ways) so that every store instruction writes 32 consecutive
      // columns of one row.
      float* stg = reinterpret_cast<float*>(smem + STAGES * STAGE + 256) + (warp - 2) * 32 * 33;
      const int rbase = m0 + q * 32;
      constexpr bool GLU_OUT = EPI == EPI_SWIGLU;  // SwiGLU applied here (no split)
      const int ncol = GLU_OUT && g.splits == 1 ? BN / 2 : BN;
      for (int c = eh * ncol / 2; c < (eh + 1) * ncol / 2; c += 32) {
        float v[32];
        if (GLU_OUT && g.splits == 1) {
          float gv[32], uv[32];
          tc::tmem_ld32(lane_base + c, gv);
          tc::tmem_ld32(lane_base + BN / 2 + c, uv);
#pragma unroll
          for (int i1 = 0; i1 < 32; ++i1) v[i1] = __fdividef(gv[i1], 1.f + __expf(-gv[i1])) * uv[i1];
        } else {
          tc::tmem_ld32(lane_base + c, v);
        }
        if (EPI == EPI_QKV && g.splits == 1) {  // row per thread: the pairs sit in adjacent registers
          qkv_row(ep, v, n0 + c, N, rbase + lane, M, err);
          continue;
        }
        __syncwarp();
#pragma unroll
        for (int i1 = 0; i1 < 32; ++i1) stg[lane * 33 + i1] = v[i1];
        __syncwarp();
        // this lane's output column and where the block's rows go
        int col = n0 + c + lane;
        size_t base_off = 0;
        if (GLU_OUT && g.splits > 1) {  // raw gate then up partials: ws[z][M][2N]
          const bool up = c >= BN / 2;
          col = n0 + (up ? c - BN / 2 : c) + lane;
          base_off = up ? (size_t)N : 0;
        }
        if (col < N) {
          const float bias = EPI == EPI_STORE && g.splits == 1 && ep.bias ? to_f32(ep.bias[col]) : 0.f;
          const int nr = min(32, M - rbase);
          if (EPI == EPI_ADD && g.splits == 1) {  // residual add: all loads first
            float old[32];
#pragma unroll
            for (int rr = 0; rr < 32; ++rr)
              old[rr] = rr < nr ? ep.C[(size_t)(rbase + rr) * ep.ldc + col] : 0.f;
#pragma unroll
            for (int rr = 0; rr < 32; ++rr)
              if (rr < nr) ep.C[(size_t)(rbase + rr) * ep.ldc + col] = old[rr] + stg[rr * 33 + lane];
          } else {
            bool bad = false;  // fp16 range (SwiGLU output), raised once after the block
#pragma unroll 4
            for (int rr = 0; rr < nr; ++rr) {
              const float x = stg[rr * 33 + lane];
              const int row = rbase + rr;
              if (g.splits > 1) {
                if (GLU_OUT)
                  ws[((size_t)z * M + row) * 2 * N + base_off + col] = x;
                else
                  ws[((size_t)z * M + row) * N + col] = x;
              } else if (GLU_OUT) {
                bad |= !(fabsf(x) < 65520.f);
                ep.Cb[(size_t)row * ep.ldc + col] = __float2half_rn(x);
              } else {
                ep.C[(size_t)row * ep.ldc + col] = x + bias;
              }
            }
            if (bad) atomicOr(err, ERR_RANGE);
          }
        }
      }
      // the accumulator is free for unit i + 2
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CL == 2) tc::mbar_arrive_cluster(tc::mapa_shared(acc_empty0 + 8 * b, 0));
        else mbar_arrive(acc_empty0 + 8 * b);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (CL == 2) tc::cluster_sync();  // the pair's MMAs and loads are all done
  if (warp == 0) {
    tc::tc_fence_after();
    if (CL == 2) tc::tmem_dealloc_pair(tmem, TCOLS);
    else tc::tmem_dealloc(tmem, TCOLS);
  }
}

// ---- skinny GEMM of a batched decode step ------------------------------------------------
//
//   P[split][b][col_off + r] = sum over the split's K range of W[r, k] X[b, k]
//
// for up to three weight matrices W (selected per CTA, e.g. q/k/v or gate/up) against the
// (at most 16) activation rows X of the sequences. The weight rows take the MMA's M side
// (128 per CTA) and the sequences its N side (N = 16), so every weight byte is read once
// for all sequences. K is split over grid.y so that about one CTA per SM streams weights;
// the fp32 partials are summed by the consuming kernel in split order (deterministic).
// The LM-head variant (one split) stores the logits of active sequences and folds each
// warp's rows into per-sequence packed argmax keys.
namespace sk {
constexpr int BM = 128, BN = 16, BK = 64, STAGES = 6, THREADS = 192;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE = A_BYTES + B_BYTES;
constexpr size_t SMEM = (size_t)STAGES * STAGE + 1024 + 256;
}  // namespace sk

struct SkinnyArgs {
  int nz;
  int tile_start[3];  // first tile of each weight matrix (grid.x = all tiles)
  int rows[3];        // rows of each matrix
  int col_off[3];     // partial column of its first row
  int K, splits, n_total;
  float* part;        // [splits][16][n_total]
  // LM head
  float* logits;      // [nseq][V]
  int V, nseq;
  const int* active;
  unsigned long long* keys;  // [nseq]
  int* err;
  unsigned long long* tl;    // timeline slots or null
  // fused SwiGLU (MODE 2): w0 / w1 = gate / up maps of 64-row boxes; act[b][i] fp16
  f16* act;
  int n_act;
};

// MODE 0: split-K partials; 1: LM head (logits and argmax keys); 2: gate/up with SwiGLU
// (a tile holds 64 gate rows then the 64 up rows of the same outputs; one split)
template <int MODE>
__global__ void __launch_bounds__(sk::THREADS, 1)
skinny_tc_kernel(const __grid_constant__ CUtensorMap w0, const __grid_constant__ CUtensorMap w1,
                 const __grid_constant__ CUtensorMap w2, const __grid_constant__ CUtensorMap xm,
                 const SkinnyArgs a) {
  using namespace sk;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + STAGES * STAGE);
  uint32_t* tmem_slot = (uint32_t*)(bars + 2 * STAGES + 1);
  const uint32_t full0 = tc::smem_u32(bars), empty0 = tc::smem_u32(bars + STAGES),
                 accum = tc::smem_u32(bars + 2 * STAGES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  constexpr bool LM = MODE == 1, GLU = MODE == 2;
  const int z = GLU ? 0 : (a.nz > 1 && tile >= a.tile_start[1]) + (a.nz > 2 && tile >= a.tile_start[2]);
  const CUtensorMap* wm = z == 0 ? &w0 : z == 1 ? &w1 : &w2;
  const int m0 = GLU ? tile * (BM / 2) : (tile - a.tile_start[z]) * BM;
  const int nk = (a.K + BK - 1) / BK;
  const int kb0 = (int)((long long)blockIdx.y * nk / a.splits);
  const int kb1 = (int)((long long)(blockIdx.y + 1) * nk / a.splits);
  __shared__ int s_abort;
  tl_stamp(a.tl, 0);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(full0 + 8 * s, 1);
      tc::mbar_init(empty0 + 8 * s, 1);
    }
    tc::mbar_init(accum, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_slot), 32);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer: 128 weight rows and the 16 activation rows per 64-wide K block.
    // The weights of the first stages do not depend on the preceding kernels: they are
    // requested before the dependency wait, their activation rows after it.
    const int pre = min(STAGES, kb1 - kb0);
    for (int j = 0; j < pre; ++j) {
      const uint32_t a_dst = tc::smem_u32(smem + j * STAGE);
      tc::mbar_expect_tx(full0 + 8 * j, STAGE);
      if (GLU) {
        tc::tma_load_2d(a_dst, &w0, full0 + 8 * j, (kb0 + j) * BK, m0);
        tc::tma_load_2d(a_dst + A_BYTES / 2, &w1, full0 + 8 * j, (kb0 + j) * BK, m0);
      } else {
        tc::tma_load_2d(a_dst, wm, full0 + 8 * j, (kb0 + j) * BK, m0);
      }
    }
    pdl_wait();
    pdl_trigger();
    tl_stamp(a.tl, 1);
    for (int j = 0; j < pre; ++j)
      tc::tma_load_2d(tc::smem_u32(smem + j * STAGE) + A_BYTES, &xm, full0 + 8 * j, (kb0 + j) * BK, 0);
    int issued = pre;
    for (int kb = kb0 + pre; kb < kb1; ++kb) {
      const int j = kb - kb0, s = j % STAGES;
      if (!tc::mbar_wait(empty0 + 8 * s, ((j / STAGES) & 1) ^ 1, a.err)) { s_abort = 1; break; }
      if (s_abort) break;
      const uint32_t a_dst = tc::smem_u32(smem + s * STAGE);
      tc::mbar_expect_tx(full0 + 8 * s, STAGE);
      if (GLU) {
        tc::tma_load_2d(a_dst, &w0, full0 + 8 * s, kb * BK, m0);
        tc::tma_load_2d(a_dst + A_BYTES / 2, &w1, full0 + 8 * s, kb * BK, m0);
      } else {
        tc::tma_load_2d(a_dst, wm, full0 + 8 * s, kb * BK, m0);
      }
      tc::tma_load_2d(a_dst + A_BYTES, &xm, full0 + 8 * s, kb * BK, 0);
      ++issued;
    }
    for (int j = (issued > STAGES ? issued - STAGES : 0); j < issued; ++j)
      tc::mbar_wait(full0 + 8 * (j % STAGES), (j / STAGES) & 1, a.err);
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    constexpr uint32_t idesc = LM ? tc::idesc_bf16(BM, BN) : tc::idesc_f16(BM, BN);
    bool ok = true;
    for (int kb = kb0; kb < kb1; ++kb) {
      const int j = kb - kb0, s = j % STAGES;
      if (!tc::mbar_wait(full0 + 8 * s, (j / STAGES) & 1, a.err)) { ok = false; s_abort = 1; break; }
      tc::tc_fence_after();
      const uint32_t a_base = tc::smem_u32(smem + s * STAGE);
      const uint32_t b_base = a_base + A_BYTES;
#pragma unroll
      for (int k = 0; k < BK / 16; ++k)
        tc::mma_f16(tmem, tc::smem_desc_sw128(a_base + 32 * k), tc::smem_desc_sw128(b_base + 32 * k), idesc,
                    (j | k) != 0);
      tc::mma_commit(empty0 + 8 * s);
    }
    if (ok && kb1 > kb0) tc::mma_commit(accum);
  } else if (warp >= 2) {
    // ---- epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 = weight rows of the tile
    pdl_wait();  // the partial buffer and the flags belong to the preceding kernels until then
    const int q = warp & 3;
    const int r = m0 + q * 32 + lane;
    float v[16];
    bool have = false;
    if (kb1 > kb0 && tc::mbar_wait(accum, 0, a.err)) {
      tc::tc_fence_after();
      tc::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16), v);
      have = true;
    } else if (kb1 == kb0) {
#pragma unroll
      for (int b = 0; b < 16; ++b) v[b] = 0.f;
      have = true;
    }
    if (GLU) {
      // TMEM lanes 0-63: gate rows m0.., lanes 64-127: the up rows of the same outputs. The
      // gate warps park their values in shared memory (the drained stage buffers), the up
      // warps form silu(gate) * up for the 16 activation rows.
      float* gbuf = reinterpret_cast<float*>(smem);  // [64][17]
      if (q < 2 && have) {
#pragma unroll
        for (int b = 0; b < 16; ++b) gbuf[(q * 32 + lane) * 17 + b] = v[b];
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
      if (q >= 2 && have) {
        const int i = m0 + (q - 2) * 32 + lane;
        if (i < a.n_act) {
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            const float g = gbuf[((q - 2) * 32 + lane) * 17 + b];
            a.act[(size_t)b * a.n_act + i] = to_half_checked((g / (1.f + expf(-g))) * v[b], a.err);
          }
        }
      }
    } else if (have) {
      const bool in = r < a.rows[z];
      if (!LM) {
        if (in) {
          float* dst = a.part + (size_t)blockIdx.y * 16 * a.n_total + a.col_off[z] + r;
#pragma unroll
          for (int b = 0; b < 16; ++b) dst[(size_t)b * a.n_total] = v[b];
        }
      } else {
        bool bad = false;
#pragma unroll
        for (int b = 0; b < 16; ++b) {
          if (b < a.nseq && a.active[b]) {  // uniform over the warp
            unsigned long long k = 0ull;
            if (in) {
              a.logits[(size_t)b * a.V + r] = v[b];
              if (!isfinite(v[b])) bad = true;
              k = argmax_key(v[b], r);
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
              const unsigned long long t = __shfl_xor_sync(0xffffffffu, k, o);
              k = t > k ? t : k;
            }
            if (lane == 0 && k) atomicMax(a.keys + b, k);
          }
        }
        if (bad) atomicOr(a.err, ERR_NONFINITE);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 32);
  }
  tl_stamp(a.tl, 2);
}

// Act[m][n] = fp16(silu(g) * u), g and u the split sums (in split order) of ws[s][m][n] and
// ws[s][m][N + n]
__global__ void splitk_swiglu_kernel(const float* ws, int splits, int M, int N, f16* Act, int ldc, int* err) {
  pdl_trigger();
  pdl_wait();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)M * N) return;
  const int m = (int)(i / N), n = (int)(i - (size_t)m * N);
  float g = 0.f, u = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float* row = ws + ((size_t)s * M + m) * 2 * N;
    g += __ldcg(row + n);
    u += __ldcg(row + N + n);
  }
  Act[(size_t)m * ldc + n] = to_half_checked((g / (1.f + expf(-g))) * u, err);
}

// C[m][n] = (add ? C[m][n] : 0) + sum over splits of ws[s][m][n] (in split order) + bias[n]
__global__ void splitk_reduce_kernel(const float* ws, int splits, int M, int N, const bf16* bias, float* C, int ldc,
                                     int add) {
  pdl_trigger();
  pdl_wait();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)M * N) return;
  const int m = (int)(i / N), n = (int)(i - (size_t)m * N);
  float v[16];
#pragma unroll
  for (int s = 0; s < 16; ++s) v[s] = s < splits ? __ldcg(ws + (size_t)s * M * N + i) : 0.f;
  float acc = add ? C[(size_t)m * ldc + n] : 0.f;
#pragma unroll
  for (int s = 0; s < 16; ++s) acc += v[s];
  if (bias) acc += __bfloat162float(bias[n]);
  C[(size_t)m * ldc + n] = acc;
}

// EPI_QKV after split-K: one thread per (row, rotation pair), the splits added in order
__global__ void splitk_qkv_kernel(const float* ws, int splits, int M, int N, const bf16* bias, QkvOut o, int* err) {
  pdl_trigger();
  pdl_wait();
  const int np = N >> 1;
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)M * np) return;
  const int m = (int)(idx / np), col = 2 * (int)(idx - (size_t)m * np);
  float a = 0.f, b = 0.f;
  for (int z = 0; z < splits; ++z) {
    const float2 v = __ldcg(reinterpret_cast<const float2*>(ws + ((size_t)z * M + m) * N + col));
    a += v.x;
    b += v.y;
  }
  if (bias) {
    a += __bfloat162float(bias[col]);
    b += __bfloat162float(bias[col + 1]);
  }
  const int head = col / o.hd, half = o.hd >> 1, i = (col - head * o.hd) >> 1;
  f16* dst;
  if (head < o.nq + o.nkv) {
    const float2 cs = o.rope[(size_t)(o.pos0 + m) * half + i];
    const float ra = a * cs.x - b * cs.y, rb = b * cs.x + a * cs.y;
    a = ra;
    b = rb;
  }
  if (head < o.nq) {
    dst = o.Qh + (size_t)m * o.nq * o.hd + (size_t)head * o.hd;
    a *= o.qscale;
    b *= o.qscale;
  } else {
    const bool is_k = head < o.nq + o.nkv;
    const int hh = is_k ? head - o.nq : head - o.nq - o.nkv;
    dst = (is_k ? o.kc : o.vc) + ((size_t)hh * o.cap + o.pos0 + m) * o.hd;
  }
  dst[i] = to_half_checked(a, err);
  dst[i + half] = to_half_checked(b, err);
}

// ---- host side ------------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

// 2-D fp16 (or bf16) row-major [rows][cols] (row pitch ld elements), box 64 x box_rows,
// 128B swizzle
bool make_map(void* mv, const void* base, int rows, int cols, int ld, int box_rows, bool bf) {
  CUtensorMap* m = reinterpret_cast<CUtensorMap*>(mv);
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  if (((uintptr_t)base & 15) || ((size_t)ld * 2) % 16) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)tc::BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return f(m, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
           const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of one layer's fp16 key or value cache [nkv][cap][hd]: dims {hd, keys, nkv}
// (keys = the positions written so far, so boxes past them read zeros), boxes of 64 head
// columns x box_keys positions of one KV head, 128-byte swizzle.
bool make_map_kv(void* mv, const void* base, int hd, int keys, int nkv, int cap, int box_keys) {
  CUtensorMap* m = reinterpret_cast<CUtensorMap*>(mv);
  EncodeTiledFn f = encode_fn();
  if (!f || ((uintptr_t)base & 15) || hd % 64 || keys < 1 || keys > cap || box_keys < 8 || box_keys > 256) return false;
  cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)keys, (cuuint64_t)nkv};
  cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)cap * hd * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_keys, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


constexpr int TC_BN = 256;

template <int BN, int EPI, int CL>
static cudaError_t set_tc_attr() {
  return cudaFuncSetAttribute(gemm_tc_kernel<BN, EPI, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)tc_smem<BN, CL>());
}

cudaError_t gemm_tc_set_attributes() {
  cudaError_t e;
  if ((e = set_tc_attr<TC_BN, EPI_STORE, 1>()) || (e = set_tc_attr<TC_BN, EPI_STORE, 2>())) return e;
  if ((e = set_tc_attr<TC_BN, EPI_ADD, 1>()) || (e = set_tc_attr<TC_BN, EPI_ADD, 2>())) return e;
  if ((e = set_tc_attr<TC_BN, EPI_SWIGLU, 1>()) || (e = set_tc_attr<TC_BN, EPI_SWIGLU, 2>())) return e;
  if ((e = set_tc_attr<192, EPI_STORE, 1>()) || (e = set_tc_attr<192, EPI_STORE, 2>())) return e;
  if ((e = set_tc_attr<192, EPI_ADD, 1>()) || (e = set_tc_attr<192, EPI_ADD, 2>())) return e;
  if ((e = set_tc_attr<64, EPI_STORE, 1>()) || (e = set_tc_attr<64, EPI_ADD, 1>())) return e;
  if ((e = set_tc_attr<TC_BN, EPI_QKV, 1>()) || (e = set_tc_attr<TC_BN, EPI_QKV, 2>())) return e;
  if ((e = set_tc_attr<192, EPI_QKV, 1>()) || (e = set_tc_attr<192, EPI_QKV, 2>())) return e;
  if ((e = set_tc_attr<64, EPI_QKV, 1>())) return e;
  return set_tc_attr<128, EPI_SWIGLU, 1>();
}

// QW_PREFILL_PDL=0: launch the prefill kernels without programmatic dependent launch
bool tc_pdl() {
  static const bool v = [] {
    const char* e = std::getenv("QW_PREFILL_PDL");
    return !(e && e[0] == '0');
  }();
  return v;
}

// One launch of the persistent GEMM: clusters of CL CTAs, as many as fit one per SM (at most
// one per unit)
template <int BN, int EPI, int CL>
static cudaError_t launch_tc(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mb2, const TcEpi& ep,
                             int M, int N, int K, int* err, const TcGrid& g, float* ws, int nsm, cudaStream_t s,
                             bool pdl) {
  const int units = ((g.tiles_m + CL - 1) / CL) * g.tiles_n * g.splits;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(tc::THREADS);
  cfg.dynamicSmemBytes = tc_smem<BN, CL>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CL > 1 ? 1 : 0;
  // the pairs that can be resident at once (an SM left over in a GPC takes none)
  static int resident = -1;
  if (resident < 0) {
    int n = 0;
    cfg.gridDim = dim3(CL);
    if (CL == 1 || cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, EPI, CL>, &cfg) != cudaSuccess || n <= 0)
      n = nsm / CL;
    resident = n;
  }
  int clusters = nsm > 0 ? std::min(resident, nsm / CL) : units;
  if (clusters > units || clusters <= 0) clusters = units;
  cfg.gridDim = dim3(clusters * CL);
  // programmatic dependent launch: the CTAs may start (and request their weights) while the
  // previous kernel finishes
  cudaLaunchAttribute attrs[2] = {attr[0], {}};
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = CL > 1 ? attrs : attrs + 1;
  cfg.numAttrs = (CL > 1 ? 1 : 0) + (pdl ? 1 : 0);
  if (cfg.numAttrs == 0) cfg.attrs = nullptr;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, EPI, CL>, ma, mb, mb2, ep, M, N, K, err, g, ws);
}

// QW_GEMM_CLUSTER=0: no CTA pairs (for comparison)
static bool gemm_pairs() {
  static const bool v = [] {
    const char* e = std::getenv("QW_GEMM_CLUSTER");
    return !(e && e[0] == '0');
  }();
  return v;
}


bool gemm_tc_available() { return encode_fn() != nullptr; }

cudaError_t skinny_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(skinny_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sk::SMEM);
  if (e) return e;
  if ((e = cudaFuncSetAttribute(skinny_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sk::SMEM)))
    return e;
  return cudaFuncSetAttribute(skinny_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sk::SMEM);
}

// Fused gate/up + SwiGLU: tiles of 64 gate rows and the 64 up rows of the same outputs
// (64-row boxes), one split; false unless that keeps at least half the SMs busy.
bool skinny_plan_glu(SkinnyPlan* p, const void* Wg, const void* Wu, int I, const void* X, int K, int nsm) {
  std::memset(p, 0, sizeof(*p));
  const int tiles = (I + sk::BM / 2 - 1) / (sk::BM / 2);
  if (2 * tiles < nsm) return false;
  if (!make_map(reinterpret_cast<CUtensorMap*>(p->wmap[0]), Wg, I, K, K, sk::BM / 2) ||
      !make_map(reinterpret_cast<CUtensorMap*>(p->wmap[1]), Wu, I, K, K, sk::BM / 2) ||
      !make_map(reinterpret_cast<CUtensorMap*>(p->wmap[2]), Wu, I, K, K, sk::BM / 2) ||
      !make_map(reinterpret_cast<CUtensorMap*>(p->xmap), X, 16, K, K, sk::BN))
    return false;
  p->nz = 2;
  p->K = K;
  p->tiles = tiles;
  p->splits = 1;
  p->n_total = I;
  p->glu = true;
  return true;
}

// Tensor maps of one skinny GEMM: nz weight matrices [rows_z][K] (fp16, or bf16 for the LM
// head) and the activation rows X [16][K] of the same type.
bool skinny_plan(SkinnyPlan* p, int nz, const void* const* W, const int* rows, const void* X, int K, bool bf,
                 int nsm) {
  if (nz < 1 || nz > 3) return false;
  std::memset(p, 0, sizeof(*p));
  p->nz = nz;
  p->K = K;
  p->lm = bf;
  int tiles = 0, col = 0;
  for (int i = 0; i < 3; ++i) {
    const int zi = i < nz ? i : nz - 1;
    if (!make_map(reinterpret_cast<CUtensorMap*>(p->wmap[i]), W[zi], rows[zi], K, K, sk::BM, bf)) return false;
    if (i < nz) {
      p->tile_start[i] = tiles;
      p->rows[i] = rows[i];
      p->col_off[i] = col;
      tiles += (rows[i] + sk::BM - 1) / sk::BM;
      col += rows[i];
    }
  }
  if (!make_map(reinterpret_cast<CUtensorMap*>(p->xmap), X, 16, K, K, sk::BN, bf)) return false;
  p->tiles = tiles;
  p->n_total = col;
  const int nk = (K + sk::BK - 1) / sk::BK;
  int splits = bf ? 1 : nsm / tiles;
  if (splits < 1) splits = 1;
  if (splits > nk) splits = nk;
  if (splits > SKINNY_MAX_SPLITS) splits = SKINNY_MAX_SPLITS;  // the consumers sum at most this many
  p->splits = splits;
  return true;
}

cudaError_t skinny_run(const SkinnyPlan& p, float* part, float* logits, int V, int nseq, const int* active,
                       unsigned long long* keys, int* err, unsigned long long* tl, cudaStream_t s, __half* act) {
  SkinnyArgs a{};
  a.nz = p.nz;
  for (int i = 0; i < 3; ++i) {
    a.tile_start[i] = p.tile_start[i];
    a.rows[i] = p.rows[i];
    a.col_off[i] = p.col_off[i];
  }
  a.K = p.K;
  a.splits = p.splits;
  a.n_total = p.n_total;
  a.part = part;
  a.logits = logits;
  a.V = V;
  a.nseq = nseq;
  a.active = active;
  a.keys = keys;
  a.err = err;
  a.tl = tl;
  const CUtensorMap* wm = reinterpret_cast<const CUtensorMap*>(p.wmap);
  const CUtensorMap* xm = reinterpret_cast<const CUtensorMap*>(p.xmap);
  const dim3 grid(p.tiles, p.splits);
  a.act = act;
  a.n_act = p.n_total;
  const bool pdl = batched_pdl();
  if (p.lm) return launch_k(skinny_tc_kernel<1>, grid, dim3(sk::THREADS), sk::SMEM, s, pdl, wm[0], wm[1], wm[2], *xm, a);
  if (p.glu) return launch_k(skinny_tc_kernel<2>, grid, dim3(sk::THREADS), sk::SMEM, s, pdl, wm[0], wm[1], wm[2], *xm, a);
  return launch_k(skinny_tc_kernel<0>, grid, dim3(sk::THREADS), sk::SMEM, s, pdl, wm[0], wm[1], wm[2], *xm, a);
}

// C[M][N] (fp32, ldc) = / += A[M][K] (fp16, lda) . B[N][K]^T (fp16, ldb) (+ bias[N], bf16)
template <int BN, int CL>
static cudaError_t launch_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const TcEpi& ep, int M, int N, int K,
                               bool add, int* err, const TcGrid& g, float* ws, int nsm, cudaStream_t s, bool pdl) {
  if (add) return launch_tc<BN, EPI_ADD, CL>(ma, mb, mb, ep, M, N, K, err, g, ws, nsm, s, pdl);
  return launch_tc<BN, EPI_STORE, CL>(ma, mb, mb, ep, M, N, K, err, g, ws, nsm, s, pdl);
}

// Tile width, K splits and CTA pairing of a C[M, N] = A . B^T launch
struct TcPlan {
  int bn, splits, tiles_m;
  bool pair;
};
static TcPlan tc_plan(int M, int N, int K, const float* ws, size_t ws_floats, int nsm) {
  const int tiles_m = (M + tc::BM - 1) / tc::BM;
  const int nk = (K + tc::BK - 1) / tc::BK;
  // tile width: 256 or 192 columns, whichever finishes first when the tiles go round the
  // SMs in whole rounds (time of a round ~ tile width); 64 for short prompts (M <= 256),
  // whose GEMMs stream weights: narrow tiles give the SMs work with fewer K splits
  int bn = TC_BN;
  if (nsm > 0 && tiles_m <= 2) {
    bn = 64;
  } else if (nsm > 0) {
    auto rounds = [&](int w) { const int u = tiles_m * ((N + w - 1) / w); return (u + nsm - 1) / nsm; };
    if ((long long)rounds(192) * 192 < (long long)rounds(TC_BN) * TC_BN) bn = 192;
  }
  const int tiles = ((N + bn - 1) / bn) * tiles_m;
  // too few tiles to stream the weights from every SM: split K (up to 16 ways, at least two
  // K blocks per split, as far as the workspace holds the partial tiles)
  int splits = 1;
  if (ws && nsm > 0 && 2 * tiles < nsm) {
    splits = nsm / tiles;
    if (splits > 16) splits = 16;
    if (splits > nk / 2) splits = nk / 2;
    const size_t per = (size_t)M * N;
    if ((size_t)splits * per > ws_floats) splits = (int)(ws_floats / per);
    if (splits < 2) splits = 1;
  }
  // CTA pairs (M = 256 products, each CTA staging half of B) when there are row tiles to pair
  const bool pair = bn != 64 && tiles_m >= 2 && nsm >= 2 && gemm_pairs();
  return TcPlan{bn, splits, tiles_m, pair};
}

cudaError_t gemm_tc(const f16* A, int lda, const f16* B, int ldb, const bf16* bias, float* C, int ldc,
                    int M, int N, int K, bool accumulate, int* err, cudaStream_t s, float* ws, size_t ws_floats,
                    int nsm, bool pdl) {
  const TcPlan pl = tc_plan(M, N, K, ws, ws_floats, nsm);
  const int bn = pl.bn, splits = pl.splits, tiles_m = pl.tiles_m;
  const bool pair = pl.pair;
  CUtensorMap ma, mb;
  if (!make_map(&ma, A, M, K, lda, tc::BM) || !make_map(&mb, B, N, K, ldb, pair ? bn / 2 : bn))
    return cudaErrorInvalidValue;
  TcEpi ep{C, bias, nullptr, ldc, {}};
  const TcGrid g{tiles_m, (N + bn - 1) / bn, splits};
  const bool add = accumulate && splits == 1;
  cudaError_t e;
  if (bn == 192) e = pair ? launch_gemm<192, 2>(ma, mb, ep, M, N, K, add, err, g, ws, nsm, s, pdl)
                          : launch_gemm<192, 1>(ma, mb, ep, M, N, K, add, err, g, ws, nsm, s, pdl);
  else if (bn == 64) e = launch_gemm<64, 1>(ma, mb, ep, M, N, K, add, err, g, ws, nsm, s, pdl);
  else e = pair ? launch_gemm<TC_BN, 2>(ma, mb, ep, M, N, K, add, err, g, ws, nsm, s, pdl)
                : launch_gemm<TC_BN, 1>(ma, mb, ep, M, N, K, add, err, g, ws, nsm, s, pdl);
  if (e) return e;
  if (splits > 1) {
    const size_t n = (size_t)M * N;
    if ((e = launch_k(splitk_reduce_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, pdl,
                      (const float*)ws, splits, M, N, bias, C, ldc, accumulate ? 1 : 0)))
      return e;
  }
  return cudaGetLastError();
}

// q | k | v = A . B^T (+ bias), rotated and stored in fp16 (QkvOut)
cudaError_t gemm_tc_qkv(const f16* A, int lda, const f16* B, int ldb, const bf16* bias, int M, int N, int K,
                        const QkvOut& o, int* err, cudaStream_t s, float* ws, size_t ws_floats, int nsm, bool pdl) {
  if (o.hd <= 0 || (o.hd & 1) || N != (o.nq + 2 * o.nkv) * o.hd) return cudaErrorInvalidValue;
  const TcPlan pl = tc_plan(M, N, K, ws, ws_floats, nsm);
  CUtensorMap ma, mb;
  if (!make_map(&ma, A, M, K, lda, tc::BM) || !make_map(&mb, B, N, K, ldb, pl.pair ? pl.bn / 2 : pl.bn))
    return cudaErrorInvalidValue;
  TcEpi ep{nullptr, bias, nullptr, 0, o};
  const TcGrid g{pl.tiles_m, (N + pl.bn - 1) / pl.bn, pl.splits};
  cudaError_t e;
  if (pl.bn == 192)
    e = pl.pair ? launch_tc<192, EPI_QKV, 2>(ma, mb, mb, ep, M, N, K, err, g, ws, nsm, s, pdl)
                : launch_tc<192, EPI_QKV, 1>(ma, mb, mb, ep, M, N, K, err, g, ws, nsm, s, pdl);
  else if (pl.bn == 64)
    e = launch_tc<64, EPI_QKV, 1>(ma, mb, mb, ep, M, N, K, err, g, ws, nsm, s, pdl);
  else
    e = pl.pair ? launch_tc<TC_BN, EPI_QKV, 2>(ma, mb, mb, ep, M, N, K, err, g, ws, nsm, s, pdl)
                : launch_tc<TC_BN, EPI_QKV, 1>(ma, mb, mb, ep, M, N, K, err, g, ws, nsm, s, pdl);
  if (e) return e;
  if (pl.splits > 1) {
    const size_t n = (size_t)M * (N / 2);
    if ((e = launch_k(splitk_qkv_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, pdl,
                      (const float*)ws, pl.splits, M, N, bias, o, err)))
      return e;
  }
  return cudaGetLastError();
}

// Act[M][N] (fp16, ldc) = silu(A . Wg^T) * (A . Wu^T)
cudaError_t gemm_tc_swiglu(const f16* A, int lda, const f16* Wg, const f16* Wu, int ldb, f16* Act,
                           int ldc, int M, int N, int K, int* err, cudaStream_t s, float* ws, size_t ws_floats,
                           int nsm, bool pdl) {
  // 128 output columns per tile (128 gate + 128 up rows); 64 for short prompts, whose gate/up
  // then fills the SMs without K splits
  const int tiles_m = (M + tc::BM - 1) / tc::BM;
  const int bn = nsm > 0 && tiles_m <= 2 ? 128 : TC_BN;
  CUtensorMap ma, mg, mu;
  if (!make_map(&ma, A, M, K, lda, tc::BM) || !make_map(&mg, Wg, N, K, ldb, bn / 2) ||
      !make_map(&mu, Wu, N, K, ldb, bn / 2))
    return cudaErrorInvalidValue;
  TcEpi ep{nullptr, nullptr, Act, ldc, {}};
  const int tiles = ((N + bn / 2 - 1) / (bn / 2)) * tiles_m;
  const int nk = (K + tc::BK - 1) / tc::BK;
  int splits = 1;  // as in gemm_tc: split K when the tiles leave SMs idle
  if (ws && nsm > 0 && 2 * tiles < 2 * nsm && tiles < nsm / 2) {
    splits = nsm / tiles;
    if (splits > 16) splits = 16;
    if (splits > nk / 2) splits = nk / 2;
    const size_t per = (size_t)M * 2 * N;
    if ((size_t)splits * per > ws_floats) splits = (int)(ws_floats / per);
    if (splits < 2) splits = 1;
  }
  const TcGrid g{tiles_m, (N + bn / 2 - 1) / (bn / 2), splits};
  cudaError_t e;
  if (bn == 128)
    e = launch_tc<128, EPI_SWIGLU, 1>(ma, mg, mu, ep, M, N, K, err, g, ws, nsm, s, pdl);
  else if (tiles_m >= 2 && nsm >= 2 && gemm_pairs())  // CTA pairs: rank 0 stages gate, rank 1 up
    e = launch_tc<TC_BN, EPI_SWIGLU, 2>(ma, mg, mu, ep, M, N, K, err, g, ws, nsm, s, pdl);
  else
    e = launch_tc<TC_BN, EPI_SWIGLU, 1>(ma, mg, mu, ep, M, N, K, err, g, ws, nsm, s, pdl);
  if (e) return e;
  if (splits > 1) {
    const size_t n = (size_t)M * N;
    if ((e = launch_k(splitk_swiglu_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, pdl,
                      (const float*)ws, splits, M, N, Act, ldc, err)))
      return e;
  }
  return cudaGetLastError();
}

}  // namespace qw
