// bwd_sm103a.cu — attention backward (dQ, dK, dV) on tcgen05 / TMEM / TMA.
//
// "Why Fast GPUs Still Wait for Memory", section "FlashAttention is an IO
// algorithm": the backward pass keeps the forward's tiling and recomputes S
// from Q and K instead of storing it, trading extra arithmetic for traffic.
// With the forward's log-sum-exp L_i saved, each tile recomputes
//     P_ij = exp(s_ij - L_i)                  (s = scale q_i . k_j, masked)
// exactly, with no running maximum, and the gradients follow from the chain
// rule through the row softmax:
//     dV = P^T dO,   dP = dO V^T,   dS = P * (dP - delta),
//     delta_i = sum_k dO_ik O_ik  (= sum_j P_ij dP_ij),
//     dQ = scale dS K,   dK = scale dS^T Q.
//
// Three launches:
//   1. prep:  delta_i and L_i log2(e) per query row, into a workspace padded
//             to whole 128-row tiles (padding: delta = 0, L = +inf, so padded
//             query rows get P = 0 in every tile that reads them);
//   2. dK/dV: one CTA per (K/V head, 128-key tile).  K and V stay in shared
//             memory; the query tiles of every query head of the group stream
//             through a two-stage TMA ring (Q, dO, L, delta).  Per query tile
//             the MMA warp computes S^T = K Q^T and dP^T = V dO^T into TMEM,
//             eight compute warps turn them into P^T and dS^T (bf16, written
//             back over S^T and dP^T), and the MMA warp accumulates
//             dV += P^T dO and dK += dS^T Q in TMEM.  Summing over the group's
//             query heads in the loop gives grouped-query K/V gradients
//             without atomics.
//   3. dQ:    one CTA per (query head, 128-query tile); K/V tiles stream
//             through the ring; S = Q K^T and dP = dO V^T into TMEM, dS back
//             over S, dQ += dS K in TMEM.
// dQ is computed by its own kernel (recomputing S and dP once more) rather
// than accumulated with atomics across the dK/dV CTAs: the gradient
// reduction stays deterministic and free of the atomic contention that the
// "Validating Memory-Optimal Transformer Kernels on Real Hardware" paper
// (section 4, the fused forward+backward kernel) measured on GPUs.
//
// Warp roles (320 threads): warps 0-7 compute (warp w owns TMEM lanes
// 32 (w % 4) .. +31, i.e. those tile rows, and columns half w / 4 of each
// 128-wide score tile), warp 8 issues MMAs, warp 9 issues TMA.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace ea {
namespace bwd {

constexpr int BT = 128;                        // rows per tile (queries or keys)
constexpr int kThreads = 320;
constexpr int kComputeWarps = 8;
constexpr int kWarpMMA = 8;
constexpr int kWarpTMA = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBoxBytes = 64 * BT * 2;    // one TMA box: 64 columns x 128 rows bf16
constexpr float kLog2e = 1.44269504088896340736f;

// dK/dV kernel: shared memory K | V | stages (Q, dO, L, delta); TMEM
// dV | dK | S^T (P^T) | dP^T (dS^T).
template <int D>
struct CfgKV {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int KB = D / 64;
  static constexpr uint32_t TILE = BT * D * 2;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = TILE;
  static constexpr uint32_t OFF_STAGE = 2 * TILE;
  static constexpr uint32_t ST_Q = 0;
  static constexpr uint32_t ST_DO = TILE;
  static constexpr uint32_t ST_LSE = 2 * TILE;          // 128 fp32
  static constexpr uint32_t ST_DELTA = 2 * TILE + 512;  // 128 fp32
  static constexpr uint32_t STAGE_BYTES = 2 * TILE + 1024;
  static constexpr uint32_t STAGE_TX = 2 * TILE + 1024;
  static constexpr int NST = (D == 64) ? 4 : 2;          // query-tile ring depth
  static constexpr uint32_t OFF_BAR = OFF_STAGE + NST * STAGE_BYTES;
  // kv, full[NST], empty[NST], s[2], dp[2], p[2], done, drain
  static constexpr int NBAR = 1 + 2 * NST + 8;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;   // tmem slot, abort flag
  // At least 116 KB so that one CTA runs per SM: each allocates all 512 TMEM
  // columns, and a second CTA would only wait for them.
  static constexpr uint32_t SMEM_ALLOC =
      SMEM_BYTES + 1024 > 118784u ? SMEM_BYTES + 1024 : 118784u;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  static constexpr uint32_t TM_DV = 0;
  static constexpr uint32_t TM_DK = D;
  static constexpr uint32_t TM_ST = 2 * D;
  static constexpr uint32_t TM_DPT = 2 * D + BT;
  static_assert(TM_DPT + BT <= kTmemCols, "tensor memory budget");
};

// dQ kernel: shared memory = a ring of (K, V) tiles; TMEM S (dS) | dP | dQ |
// Q | dO.  The query tile's Q and dO sit in TMEM as the A operands of
// S = Q K^T and dP = dO V^T, so those products read only K / V from shared
// memory (half the shared-memory operand traffic of two SS products).
template <int D>
struct CfgQ {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int KB = D / 64;
  static constexpr uint32_t TILE = BT * D * 2;
  static constexpr uint32_t OFF_STAGE = 0;
  static constexpr uint32_t ST_K = 0;
  static constexpr uint32_t ST_V = TILE;
  static constexpr uint32_t STAGE_BYTES = 2 * TILE;
  static constexpr int NST = (D == 64) ? 4 : 3;          // K/V ring depth
  static constexpr uint32_t OFF_BAR = OFF_STAGE + NST * STAGE_BYTES;
  // q (Q, dO in TMEM), full[NST], empty[NST], s[2], dp[2], p[2], done, drain
  static constexpr int NBAR = 1 + 2 * NST + 8;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;
  static constexpr uint32_t SMEM_ALLOC =
      SMEM_BYTES + 1024 > 118784u ? SMEM_BYTES + 1024 : 118784u;   // one CTA per SM
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_DP = BT;
  static constexpr uint32_t TM_DQ = 2 * BT;
  static constexpr uint32_t TM_Q = 2 * BT + D;           // bf16 pairs: D / 2 columns
  static constexpr uint32_t TM_DO = TM_Q + D / 2;
  static_assert(TM_DO + D / 2 <= kTmemCols, "tensor memory budget");
};

// ------------------------------------------------------------------ prep
// delta = sum_k dO O (fp32) and L log2(e) per (head, padded row).  D / 8
// threads per row, 16-byte loads, two rows per thread (both loads issued
// before either is used).
constexpr int kPrepThreads = 256;
template <int D>
__global__ void __launch_bounds__(kPrepThreads)
    attn_bwd_prep_kernel(const __nv_bfloat16 *__restrict__ O, const __nv_bfloat16 *__restrict__ dO,
                         const float *__restrict__ LSE, float *__restrict__ lse2,
                         float *__restrict__ delta, int N, int N_pad) {
  constexpr int TPR = D / 8;                          // threads per row
  constexpr int RPB = kPrepThreads / TPR;             // rows per block and pass
  const int sub = threadIdx.x % TPR;
  const size_t bh = blockIdx.x;                       // one head per grid row
  const __nv_bfloat16 *Oh = O + bh * N * D;
  const __nv_bfloat16 *dOh = dO + bh * N * D;
  for (int i0 = static_cast<int>(blockIdx.y) * 2 * RPB; i0 < N_pad;
       i0 += static_cast<int>(gridDim.y) * 2 * RPB) {
    int ii[2];
    uint4 o[2], g[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      ii[u] = i0 + u * RPB + static_cast<int>(threadIdx.x) / TPR;
      o[u] = make_uint4(0, 0, 0, 0);
      g[u] = o[u];
      if (ii[u] < N) {
        const size_t off = static_cast<size_t>(ii[u]) * D + sub * 8;
        o[u] = *reinterpret_cast<const uint4 *>(Oh + off);
        g[u] = *reinterpret_cast<const uint4 *>(dOh + off);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t ow[4] = {o[u].x, o[u].y, o[u].z, o[u].w};
      const uint32_t gw[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        acc += bf16lo(ow[e]) * bf16lo(gw[e]) + bf16hi(ow[e]) * bf16hi(gw[e]);
#pragma unroll
      for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (sub == 0 && ii[u] < N_pad) {
        const size_t r = bh * N_pad + ii[u];
        if (ii[u] < N) {
          delta[r] = acc;
          lse2[r] = LSE[bh * N + ii[u]] * kLog2e;
        } else {   // padding row: P = 0 wherever it is read
          delta[r] = 0.f;
          lse2[r] = INFINITY;
        }
      }
    }
  }
}

// Stages 32 fp32 accumulator columns (times `mul`) of tile row `row` as bf16
// at columns col0.. of a [128 rows][D] tile laid out as the 128-byte-swizzled
// 64-column boxes of a TMA map (box b at stage + b * kBoxBytes), for a TMA
// store of the whole tile (rows past N are dropped by the map).
__device__ __forceinline__ void stage_row32(uint32_t stage, int row, int col0,
                                            const uint32_t (&r)[32], float mul) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = pack_bf16x2(__uint_as_float(r[8 * v + 2 * e]) * mul,
                         __uint_as_float(r[8 * v + 2 * e + 1]) * mul);
    const int col = col0 + 8 * v;
    const uint32_t chunk = static_cast<uint32_t>((col & 63) >> 3) ^ static_cast<uint32_t>(row & 7);
    st_shared_v4(stage + (col >> 6) * kBoxBytes + static_cast<uint32_t>(row) * 128 + (chunk << 4),
                 w[0], w[1], w[2], w[3]);
  }
}
constexpr uint32_t kEpiBar = 1;   // named barrier of the compute warps (epilogue)

// Both kernels run two independent pipelines, one per half of the 128-wide
// score tile (query columns 0-63 / 64-127 in the dK/dV kernel, key columns
// in the dQ kernel).  Compute warps 4h..4h+3 own half h; the MMA warp issues
// each half's score products (N = 64) as soon as that half's region is free
// and each half's gradient products as soon as that half's P / dS are in.
// While one half's warps compute, the tensor pipe works on the other half.

// ------------------------------------------------------------------ dK / dV
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmdO,
                         const __grid_constant__ CUtensorMap tmdK,
                         const __grid_constant__ CUtensorMap tmdV, const float *__restrict__ lse2,
                         const float *__restrict__ delta, int N, int N_pad, int H, int H_kv,
                         int n_blk, float scale_log2, float scale, unsigned *status) {
  using C = CfgKV<D>;
  constexpr int NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Causal: K/V heads vary fastest and key tiles go in ascending order (the
  // first key tiles are seen by the most query tiles: longest first).
  // Non-causal: key tiles vary fastest, so co-resident CTAs share their
  // head's Q and dO through L2.
  const int BHkv = static_cast<int>(gridDim.x) / n_blk;
  const int bkv = CAUSAL ? static_cast<int>(blockIdx.x % BHkv) : static_cast<int>(blockIdx.x / n_blk);
  const int jt = CAUSAL ? static_cast<int>(blockIdx.x / BHkv) : static_cast<int>(blockIdx.x % n_blk);
  const int group = H / H_kv;
  const int b = bkv / H_kv;
  const int hk = bkv % H_kv;
  const int it0 = CAUSAL ? jt : 0;
  const int n_q = n_blk - it0;                 // query tiles per query head
  const int n_it = group * n_q;                // (query head of the group, query tile) pairs
  auto q_head = [&](int t) { return b * H + hk * group + t / n_q; };
  auto q_tile = [&](int t) { return it0 + t % n_q; };

  const uint32_t bar0 = sb + C::OFF_BAR;
  const uint32_t B_KV = bar0;
  auto B_FULL = [&](int s) { return bar0 + 8u * (1 + s); };
  auto B_EMPTY = [&](int s) { return bar0 + 8u * (1 + NST + s); };
  const uint32_t bar1 = bar0 + 8u * (1 + 2 * NST);
  auto B_S = [&](int h) { return bar1 + 8u * h; };          // S^T half h in TMEM
  auto B_DP = [&](int h) { return bar1 + 8u * (2 + h); };   // dP^T half h in TMEM
  auto B_P = [&](int h) { return bar1 + 8u * (4 + h); };    // P^T, dS^T half h written
  const uint32_t B_DONE = bar1 + 48;
  const uint32_t B_DRAIN = bar1 + 56;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == kWarpTMA * 32) {
    mbar_init(B_KV, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(B_FULL(s), 1);
      mbar_init(B_EMPTY(s), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(B_S(h), 1);
      mbar_init(B_DP(h), 1);
      mbar_init(B_P(h), kComputeWarps / 2);
    }
    mbar_init(B_DONE, 1);
    mbar_init(B_DRAIN, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    mbar_arrive_expect_tx(B_KV, 2 * C::TILE);
    for (int kb = 0; kb < C::KB; ++kb) {
      tma_load_3d(sb + C::OFF_K + kb * kBoxBytes, &tmK, kb * 64, jt * BT, bkv, B_KV);
      tma_load_3d(sb + C::OFF_V + kb * kBoxBytes, &tmV, kb * 64, jt * BT, bkv, B_KV);
    }
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTMA) {
    // ------------------------------------------------------------ TMA
    const bool leader = elect_one();
    int issued = 0;
    for (int t = 0; t < n_it; ++t) {
      const int s = t % NST;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(B_EMPTY(s), ((t / NST) & 1) ^ 1u, status, abort_flag)))
        break;
      if (leader) {
        const int bh = q_head(t);
        const int it = q_tile(t);
        const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(B_FULL(s), C::STAGE_TX);
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_3d(st + C::ST_Q + kb * kBoxBytes, &tmQ, kb * 64, it * BT, bh, B_FULL(s));
          tma_load_3d(st + C::ST_DO + kb * kBoxBytes, &tmdO, kb * 64, it * BT, bh, B_FULL(s));
        }
        const size_t row0 = static_cast<size_t>(bh) * N_pad + static_cast<size_t>(it) * BT;
        bulk_load_1d(st + C::ST_LSE, lse2 + row0, BT * 4, B_FULL(s));
        bulk_load_1d(st + C::ST_DELTA, delta + row0, BT * 4, B_FULL(s));
      }
      issued = t + 1;
    }
    if (leader && *abort_flag) {
      mbar_wait_drain(B_KV, 0, 100000000ull);
      for (int j = 0; j < NST && j < issued; ++j) {
        const int tt = issued - 1 - j;
        mbar_wait_drain(B_FULL(tt % NST), (tt / NST) & 1, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------------ MMA
    const bool leader = elect_one();
    constexpr uint32_t kIdescS = make_idesc_bf16(BT, BT / 2, 0, 0);
    constexpr uint32_t kIdescG = make_idesc_bf16(BT, D, 0, 1);
    // Low words of the shared-memory descriptors (one common high word):
    // K-major (head dim contiguous, 16-element k-steps inside a 64-column
    // box) and MN-major (the stage's Q / dO as B operands with the query
    // index as the reduction dimension: 16-row k-steps, 64-column boxes
    // kBoxBytes apart).
    const uint64_t dK0 = make_sdesc_sw128(sb + C::OFF_K, 16, 1024);
    const uint32_t hi = static_cast<uint32_t>(dK0 >> 32);
    const uint32_t k_lo = static_cast<uint32_t>(dK0);
    const uint32_t v_lo = static_cast<uint32_t>(make_sdesc_sw128(sb + C::OFF_V, 16, 1024));
    const uint32_t stk_lo = static_cast<uint32_t>(make_sdesc_sw128(sb + C::OFF_STAGE, 16, 1024));
    const uint32_t stm_lo =
        static_cast<uint32_t>(make_sdesc_sw128(sb + C::OFF_STAGE, kBoxBytes, 1024));
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort_flag));
    };
    // Half h of S^T = K Q^T and of dP^T = V dO^T: queries 64h..64h+63 (rows
    // 64h.. of the stage's tiles, 64 rows x 128 B = 8 KB into each box).
    auto issue_scores = [&](int s, int h) {
      const uint32_t so = (s * C::STAGE_BYTES + h * 64 * 128) >> 4;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
        mma_bf16_ss_lo(tmem + C::TM_ST + 64 * h, k_lo + koff, stk_lo + so + (C::ST_Q >> 4) + koff,
                       hi, kIdescS, kk > 0 ? 1u : 0u);
      }
      mma_commit(B_S(h));
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
        mma_bf16_ss_lo(tmem + C::TM_DPT + 64 * h, v_lo + koff, stk_lo + so + (C::ST_DO >> 4) + koff,
                       hi, kIdescS, kk > 0 ? 1u : 0u);
      }
      mma_commit(B_DP(h));
    };
    // Half h of dV += P^T dO and dK += dS^T Q: the 16-query steps 4h..4h+3,
    // A from TMEM (8 columns per step; half h's P^T / dS^T sit in columns
    // 64h..64h+31 of their regions), B = the stage's dO / Q, MN-major.
    auto issue_grads = [&](int s, int h, bool acc) {
      const uint32_t so = (s * C::STAGE_BYTES) >> 4;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int kk = 4 * h + u;
        const uint32_t boff = (kk * 16 * 128) >> 4;
        mma_bf16_ts_lo(tmem + C::TM_DV, tmem + C::TM_ST + 64 * h + 8 * u,
                       stm_lo + so + (C::ST_DO >> 4) + boff, hi, kIdescG, (acc || u > 0) ? 1u : 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int kk = 4 * h + u;
        const uint32_t boff = (kk * 16 * 128) >> 4;
        mma_bf16_ts_lo(tmem + C::TM_DK, tmem + C::TM_DPT + 64 * h + 8 * u,
                       stm_lo + so + (C::ST_Q >> 4) + boff, hi, kIdescG, (acc || u > 0) ? 1u : 0u);
      }
    };
    bool ok = wait_all(B_KV, 0) && wait_all(B_FULL(0), 0);
    if (ok) {
      tc_fence_after();
      if (leader) {
        issue_scores(0, 0);
        issue_scores(0, 1);
      }
      __syncwarp();
    }
    for (int t = 0; ok && t < n_it; ++t) {
      const int s = t % NST;
      for (int h = 0; h < 2; ++h) {
        // Half h's warps have read S^T / dP^T and written P^T / dS^T over
        // them: accumulate, then reuse the half's regions for the next tile
        // (MMAs from one thread run in issue order).
        if (!(ok = wait_all(B_P(h), t & 1))) break;
        tc_fence_after();
        if (leader) {
          issue_grads(s, h, t > 0 || h > 0);
          if (h == 1) mma_commit(t + 1 < n_it ? B_EMPTY(s) : B_DONE);
        }
        __syncwarp();
        if (t + 1 < n_it) {
          if (h == 0 && !(ok = wait_all(B_FULL((t + 1) % NST), ((t + 1) / NST) & 1)))
            break;
          tc_fence_after();
          if (leader) issue_scores((t + 1) % NST, h);
          __syncwarp();
        }
      }
    }
    if (leader) {
      mma_commit(B_DRAIN);
      mbar_wait_drain(B_DRAIN, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- compute
    const int q = warp & 3;                  // TMEM lanes 32q..32q+31 = key rows
    const int h = warp >> 2;                 // query columns 64h .. 64h + 63
    const int row = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    bool ok = true;
    for (int t = 0; t < n_it; ++t) {
      const int s = t % NST;
      const int it = q_tile(t);
      ok = __all_sync(0xffffffffu, mbar_wait(B_FULL(s), (t / NST) & 1, status, abort_flag)) &&
           __all_sync(0xffffffffu, mbar_wait(B_S(h), t & 1, status, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const float *lse_s =
          reinterpret_cast<const float *>(smem + C::OFF_STAGE + s * C::STAGE_BYTES + C::ST_LSE);
      const float *del_s =
          reinterpret_cast<const float *>(smem + C::OFF_STAGE + s * C::STAGE_BYTES + C::ST_DELTA);
      const bool diag = CAUSAL && it == jt;
      // P^T for the half's 64 queries while the dP^T product is still running.
      float p[64];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col0 = 64 * h + 32 * c;
        uint32_t sr[32];
        tmem_ld_32cols(tmem + lane_base + C::TM_ST + col0, sr);
        tmem_ld_wait_regs(sr);
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          const float4 lv = *reinterpret_cast<const float4 *>(lse_s + col0 + k);
          const float lsev[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float pe = ex2_approx(fmaf(__uint_as_float(sr[k + e]), scale_log2, -lsev[e]));
            if (diag && col0 + k + e < row) pe = 0.f;   // query before key: masked
            p[32 * c + k + e] = pe;
          }
        }
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(B_DP(h), t & 1, status, abort_flag)))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col0 = 64 * h + 32 * c;
        uint32_t dp[32];
        tmem_ld_32cols(tmem + lane_base + C::TM_DPT + col0, dp);
        tmem_ld_wait_regs(dp);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          const float4 dv = *reinterpret_cast<const float4 *>(del_s + col0 + k);
          const float delv[4] = {dv.x, dv.y, dv.z, dv.w};
          float ds[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            ds[e] = p[32 * c + k + e] * (__uint_as_float(dp[k + e]) - delv[e]);
          pk[k / 2] = pack_bf16x2(p[32 * c + k], p[32 * c + k + 1]);
          pk[k / 2 + 1] = pack_bf16x2(p[32 * c + k + 2], p[32 * c + k + 3]);
          dk[k / 2] = pack_bf16x2(ds[0], ds[1]);
          dk[k / 2 + 1] = pack_bf16x2(ds[2], ds[3]);
        }
        tmem_st_16cols(tmem + lane_base + C::TM_ST + 64 * h + 16 * c, pk);
        tmem_st_16cols(tmem + lane_base + C::TM_DPT + 64 * h + 16 * c, dk);
      }
      tmem_st_wait();
      // The stage's L / delta were read through the generic proxy and the
      // next TMA refill writes them through the async proxy.
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B_P(h));
    }
    // Epilogue: dV and dK staged as bf16 in stage 0's Q and dO slots (every
    // load into the ring has been consumed once the last products are done)
    // and stored by TMA; the compute warps agree first, so that they all
    // take part in the barrier or all skip it.
    const bool okd = ok && __all_sync(0xffffffffu, mbar_wait(B_DONE, 0, status, abort_flag));
    if (!named_bar_any(kEpiBar, 32 * kComputeWarps, !okd)) {
      tc_fence_after();
      const uint32_t st_dv = sb + C::OFF_STAGE + C::ST_Q;
      const uint32_t st_dk = sb + C::OFF_STAGE + C::ST_DO;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(tmem + lane_base + C::TM_DV + h * (D / 2) + 32 * c, r);
        tmem_ld_wait_regs(r);
        stage_row32(st_dv, row, h * (D / 2) + 32 * c, r, 1.f);
        tmem_ld_32cols(tmem + lane_base + C::TM_DK + h * (D / 2) + 32 * c, r);
        tmem_ld_wait_regs(r);
        stage_row32(st_dk, row, h * (D / 2) + 32 * c, r, scale);
      }
      fence_proxy_async_smem();
      named_bar_sync(kEpiBar, 32 * kComputeWarps);
      if (threadIdx.x == 0) {
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_store_3d(&tmdV, kb * 64, jt * BT, bkv, st_dv + kb * kBoxBytes);
          tma_store_3d(&tmdK, kb * 64, jt * BT, bkv, st_dk + kb * kBoxBytes);
        }
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ dQ
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmdQ,
                       const __nv_bfloat16 *__restrict__ Q, const __nv_bfloat16 *__restrict__ dO,
                       const float *__restrict__ lse2, const float *__restrict__ delta,
                       int N, int N_pad, int H, int H_kv,
                       int n_blk, float scale_log2, float scale, unsigned *status) {
  using C = CfgQ<D>;
  constexpr int NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Causal: heads fastest, query tiles in descending order (longest first).
  // Non-causal: query tiles fastest (co-resident CTAs share K/V through L2).
  const int BH = static_cast<int>(gridDim.x) / n_blk;
  const int bh = CAUSAL ? static_cast<int>(blockIdx.x % BH) : static_cast<int>(blockIdx.x / n_blk);
  const int it = CAUSAL ? n_blk - 1 - static_cast<int>(blockIdx.x / BH)
                        : static_cast<int>(blockIdx.x % n_blk);
  const int group = H / H_kv;
  const int kvh = (bh / H) * H_kv + (bh % H) / group;
  const int n_j = CAUSAL ? it + 1 : n_blk;

  const uint32_t bar0 = sb + C::OFF_BAR;
  const uint32_t B_Q = bar0;   // the compute warps have put Q and dO into TMEM
  auto B_FULL = [&](int s) { return bar0 + 8u * (1 + s); };
  auto B_EMPTY = [&](int s) { return bar0 + 8u * (1 + NST + s); };
  const uint32_t bar1 = bar0 + 8u * (1 + 2 * NST);
  auto B_S = [&](int h) { return bar1 + 8u * h; };          // S half h in TMEM
  auto B_DP = [&](int h) { return bar1 + 8u * (2 + h); };   // dP half h in TMEM
  auto B_P = [&](int h) { return bar1 + 8u * (4 + h); };    // dS half h written
  const uint32_t B_DONE = bar1 + 48;
  const uint32_t B_DRAIN = bar1 + 56;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == kWarpTMA * 32) {
    mbar_init(B_Q, kComputeWarps);
    for (int s = 0; s < NST; ++s) {
      mbar_init(B_FULL(s), 1);
      mbar_init(B_EMPTY(s), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(B_S(h), 1);
      mbar_init(B_DP(h), 1);
      mbar_init(B_P(h), kComputeWarps / 2);
    }
    mbar_init(B_DONE, 1);
    mbar_init(B_DRAIN, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTMA) {
    // ------------------------------------------------------------ TMA
    const bool leader = elect_one();
    int issued = 0;
    for (int j = 0; j < n_j; ++j) {
      const int s = j % NST;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(B_EMPTY(s), ((j / NST) & 1) ^ 1u, status, abort_flag)))
        break;
      if (leader) {
        const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(B_FULL(s), 2 * C::TILE);
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_3d(st + C::ST_K + kb * kBoxBytes, &tmK, kb * 64, j * BT, kvh, B_FULL(s));
          tma_load_3d(st + C::ST_V + kb * kBoxBytes, &tmV, kb * 64, j * BT, kvh, B_FULL(s));
        }
      }
      issued = j + 1;
    }
    if (leader && *abort_flag) {
      for (int u = 0; u < NST && u < issued; ++u) {
        const int jj = issued - 1 - u;
        mbar_wait_drain(B_FULL(jj % NST), (jj / NST) & 1, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------------ MMA
    const bool leader = elect_one();
    constexpr uint32_t kIdescS = make_idesc_bf16(BT, BT / 2, 0, 0);
    constexpr uint32_t kIdescG = make_idesc_bf16(BT, D, 0, 1);
    const uint64_t dst0 = make_sdesc_sw128(sb + C::OFF_STAGE, 16, 1024);
    const uint32_t hi = static_cast<uint32_t>(dst0 >> 32);
    const uint32_t stk_lo = static_cast<uint32_t>(dst0);
    const uint32_t stm_lo =
        static_cast<uint32_t>(make_sdesc_sw128(sb + C::OFF_STAGE, kBoxBytes, 1024));
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort_flag));
    };
    // Half h of S = Q K^T and of dP = dO V^T: keys 64h..64h+63 of the tile;
    // Q / dO from TMEM (8 columns per 16-element step of the head dim).
    auto issue_scores = [&](int s, int h) {
      const uint32_t so = (s * C::STAGE_BYTES + h * 64 * 128) >> 4;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
        mma_bf16_ts_lo(tmem + C::TM_S + 64 * h, tmem + C::TM_Q + 8 * kk,
                       stk_lo + so + (C::ST_K >> 4) + koff, hi, kIdescS, kk > 0 ? 1u : 0u);
      }
      mma_commit(B_S(h));
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
        mma_bf16_ts_lo(tmem + C::TM_DP + 64 * h, tmem + C::TM_DO + 8 * kk,
                       stk_lo + so + (C::ST_V >> 4) + koff, hi, kIdescS, kk > 0 ? 1u : 0u);
      }
      mma_commit(B_DP(h));
    };
    // Half h of dQ += dS K: key steps 4h..4h+3, dS from TMEM (columns
    // 64h..64h+31 of the S region), K MN-major (16-key steps).
    auto issue_dq = [&](int s, int h, bool acc) {
      const uint32_t so = (s * C::STAGE_BYTES) >> 4;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int kk = 4 * h + u;
        const uint32_t boff = (kk * 16 * 128) >> 4;
        mma_bf16_ts_lo(tmem + C::TM_DQ, tmem + C::TM_S + 64 * h + 8 * u,
                       stm_lo + so + (C::ST_K >> 4) + boff, hi, kIdescG, (acc || u > 0) ? 1u : 0u);
      }
    };
    bool ok = wait_all(B_Q, 0) && wait_all(B_FULL(0), 0);
    if (ok) {
      tc_fence_after();
      if (leader) {
        issue_scores(0, 0);
        issue_scores(0, 1);
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < n_j; ++j) {
      const int s = j % NST;
      for (int h = 0; h < 2; ++h) {
        if (!(ok = wait_all(B_P(h), j & 1))) break;
        tc_fence_after();
        if (leader) {
          issue_dq(s, h, j > 0 || h > 0);
          if (h == 1) mma_commit(j + 1 < n_j ? B_EMPTY(s) : B_DONE);
        }
        __syncwarp();
        if (j + 1 < n_j) {
          if (h == 0 && !(ok = wait_all(B_FULL((j + 1) % NST), ((j + 1) / NST) & 1)))
            break;
          tc_fence_after();
          if (leader) issue_scores((j + 1) % NST, h);
          __syncwarp();
        }
      }
    }
    if (leader) {
      mma_commit(B_DRAIN);
      mbar_wait_drain(B_DRAIN, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- compute
    const int q = warp & 3;                  // TMEM lanes 32q..32q+31 = query rows
    const int h = warp >> 2;                 // key columns 64h .. 64h + 63
    const int row = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const size_t prow = static_cast<size_t>(bh) * N_pad + static_cast<size_t>(it) * BT + row;
    const float l2 = lse2[prow];
    const float dl = delta[prow];
    {
      // Warps of half 0 put this tile's Q rows into TMEM, warps of half 1
      // its dO rows (row = lane, bf16 pairs along the columns; rows past N
      // are zero).
      const int qi = it * BT + row;
      const __nv_bfloat16 *src = (h == 0 ? Q : dO) + (static_cast<size_t>(bh) * N + qi) * D;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint4 x = make_uint4(0, 0, 0, 0);
          if (qi < N) x = *reinterpret_cast<const uint4 *>(src + 64 * c + 8 * v);
          w[4 * v] = x.x;
          w[4 * v + 1] = x.y;
          w[4 * v + 2] = x.z;
          w[4 * v + 3] = x.w;
        }
        tmem_st_32cols(tmem + lane_base + (h == 0 ? C::TM_Q : C::TM_DO) + 32 * c, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B_Q);
    }
    bool ok = true;
    for (int j = 0; j < n_j; ++j) {
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(B_S(h), j & 1, status, abort_flag)))) break;
      tc_fence_after();
      const bool diag = CAUSAL && j == it;
      const int kmax = N - j * BT;            // keys past the sequence are masked
      float p[64];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col0 = 64 * h + 32 * c;
        uint32_t sr[32];
        tmem_ld_32cols(tmem + lane_base + C::TM_S + col0, sr);
        tmem_ld_wait_regs(sr);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int col = col0 + k;
          float pe = ex2_approx(fmaf(__uint_as_float(sr[k]), scale_log2, -l2));
          if ((diag && col > row) || col >= kmax) pe = 0.f;
          p[32 * c + k] = pe;
        }
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(B_DP(h), j & 1, status, abort_flag)))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col0 = 64 * h + 32 * c;
        uint32_t dp[32];
        tmem_ld_32cols(tmem + lane_base + C::TM_DP + col0, dp);
        tmem_ld_wait_regs(dp);
        uint32_t dk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2)
          dk[k / 2] = pack_bf16x2(p[32 * c + k] * (__uint_as_float(dp[k]) - dl),
                                  p[32 * c + k + 1] * (__uint_as_float(dp[k + 1]) - dl));
        tmem_st_16cols(tmem + lane_base + C::TM_S + 64 * h + 16 * c, dk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B_P(h));
    }
    // Epilogue: dQ staged as bf16 in stage 0's K slot (every K/V load has
    // been consumed once the last products are done) and stored by TMA.
    const bool okd = ok && __all_sync(0xffffffffu, mbar_wait(B_DONE, 0, status, abort_flag));
    if (!named_bar_any(kEpiBar, 32 * kComputeWarps, !okd)) {
      tc_fence_after();
      const uint32_t st_dq = sb + C::OFF_STAGE + C::ST_K;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(tmem + lane_base + C::TM_DQ + h * (D / 2) + 32 * c, r);
        tmem_ld_wait_regs(r);
        stage_row32(st_dq, row, h * (D / 2) + 32 * c, r, scale);
      }
      fence_proxy_async_smem();
      named_bar_sync(kEpiBar, 32 * kComputeWarps);
      if (threadIdx.x == 0) {
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
          tma_store_3d(&tmdQ, kb * 64, it * BT, bh, st_dq + kb * kBoxBytes);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host
template <int D, bool CAUSAL>
static cudaError_t launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            const CUtensorMap &mdo, const CUtensorMap &mdq, const CUtensorMap &mdk,
                            const CUtensorMap &mdv, const void *Q, const void *dO,
                            const float *lse2, const float *delta, int B, int H, int H_kv, int N,
                            int N_pad, int n_blk, float scale, unsigned *status,
                            cudaStream_t stream) {
  const float scale_log2 = scale * kLog2e;
  auto kkv = attn_bwd_dkdv_kernel<D, CAUSAL>;
  auto kq = attn_bwd_dq_kernel<D, CAUSAL>;
  static std::atomic<unsigned long long> set_kv{0}, set_q{0};
  cudaError_t e = smem_limit_once(kkv, static_cast<int>(CfgKV<D>::SMEM_ALLOC), set_kv);
  if (e != cudaSuccess) return e;
  e = smem_limit_once(kq, static_cast<int>(CfgQ<D>::SMEM_ALLOC), set_q);
  if (e != cudaSuccess) return e;
  kkv<<<static_cast<unsigned>(B * H_kv * n_blk), kThreads, CfgKV<D>::SMEM_ALLOC, stream>>>(
      mq, mk, mv, mdo, mdk, mdv, lse2, delta, N, N_pad, H, H_kv, n_blk, scale_log2, scale, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kq<<<static_cast<unsigned>(B * H * n_blk), kThreads, CfgQ<D>::SMEM_ALLOC, stream>>>(
      mk, mv, mdq, static_cast<const __nv_bfloat16 *>(Q), static_cast<const __nv_bfloat16 *>(dO),
      lse2, delta, N, N_pad, H, H_kv, n_blk, scale_log2, scale, status);
  return cudaGetLastError();
}

}  // namespace bwd

size_t bwd_ws_bytes(int B, int H, int N) {
  const size_t n_pad = static_cast<size_t>((N + bwd::BT - 1) / bwd::BT) * bwd::BT;
  return 2 * static_cast<size_t>(B) * H * n_pad * 4;
}

cudaError_t launch_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                       const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int H_kv,
                       int N, int d, float scale, int causal, void *ws, unsigned *status,
                       cudaStream_t stream) {
  using namespace bwd;
  const int n_blk = (N + BT - 1) / BT;
  const int N_pad = n_blk * BT;
  const long long rows = static_cast<long long>(B) * H * N_pad;
  float *lse2 = static_cast<float *>(ws);
  float *delta = lse2 + rows;
  // Grid: one row of blocks per head, up to 1024 blocks of 2 * 256 / (d / 8)
  // rows each along a head (a block loops when the head is longer).
  const int rows_per_block = 2 * kPrepThreads / (d / 8);
  const dim3 prep_grid(static_cast<unsigned>(B * H),
                       static_cast<unsigned>(std::min(1024, (N_pad + rows_per_block - 1) / rows_per_block)));
  if (d == 128)
    attn_bwd_prep_kernel<128><<<prep_grid, kPrepThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(O), static_cast<const __nv_bfloat16 *>(dO), LSE, lse2,
        delta, N, N_pad);
  else
    attn_bwd_prep_kernel<64><<<prep_grid, kPrepThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(O), static_cast<const __nv_bfloat16 *>(dO), LSE, lse2,
        delta, N, N_pad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  if (!make_bhnd_map(&mq, Q, B * H, N, d, BT) || !make_bhnd_map(&mk, K, B * H_kv, N, d, BT) ||
      !make_bhnd_map(&mv, V, B * H_kv, N, d, BT) || !make_bhnd_map(&mdo, dO, B * H, N, d, BT) ||
      !make_bhnd_map(&mdq, dQ, B * H, N, d, BT) || !make_bhnd_map(&mdk, dK, B * H_kv, N, d, BT) ||
      !make_bhnd_map(&mdv, dV, B * H_kv, N, d, BT))
    return cudaErrorInvalidValue;
  if (d == 128)
    return causal ? launch_t<128, true>(mq, mk, mv, mdo, mdq, mdk, mdv, Q, dO, lse2, delta, B, H, H_kv, N,
                                        N_pad, n_blk, scale, status, stream)
                  : launch_t<128, false>(mq, mk, mv, mdo, mdq, mdk, mdv, Q, dO, lse2, delta, B, H, H_kv, N,
                                         N_pad, n_blk, scale, status, stream);
  return causal ? launch_t<64, true>(mq, mk, mv, mdo, mdq, mdk, mdv, Q, dO, lse2, delta, B, H, H_kv, N, N_pad,
                                     n_blk, scale, status, stream)
                : launch_t<64, false>(mq, mk, mv, mdo, mdq, mdk, mdv, Q, dO, lse2, delta, B, H, H_kv, N,
                                      N_pad, n_blk, scale, status, stream);
}

}  // namespace ea
