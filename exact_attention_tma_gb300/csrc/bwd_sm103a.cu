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
//   1. prep:  -delta_i and -L_i log2(e) per query row (negated, so that the
//             tiles' exponent and dP - delta are single packed fp32x2 FMAs /
//             adds), into a workspace padded to whole 128-row tiles (padding:
//             delta = 0, L = +inf, so padded query rows get P = 0 in every
//             tile that reads them);
//   2. dK/dV: items (K/V head, 128-key tile) on a persistent grid.  K and V
//             stay in shared memory; the query tiles of every query head of
//             the group stream through two TMA rings ((Q, -L) and
//             (dO, -delta)).  Per query tile the MMA warp computes
//             S^T = K Q^T and dP^T = V dO^T into TMEM, eight compute warps turn
//             them into P^T and dS^T (bf16, written over dP^T), and the MMA
//             warp accumulates dK += dS^T Q and dV += P^T dO in TMEM.  Summing
//             over the group's query heads in the loop gives grouped-query K/V
//             gradients without atomics.
//   3. dQ:    items (query head, 128-query tile) on a persistent grid; each
//             item's Q and dO, then its K/V tiles, stream through one ring;
//             Q and dO go into TMEM, S = Q K^T and dP = dO V^T into TMEM, dS
//             over dP, dQ += dS K in TMEM.
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
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace ea {
namespace bwd {

constexpr int BT = 128;                        // rows per tile (queries or keys)
constexpr int kThreads = 320;
constexpr int kComputeWarps = 8;
constexpr int kWarpMMA = 8;
constexpr int kWarpTMA = 9;
constexpr int kRing = 4;   // item indices in flight from the TMA warp to the others
constexpr int kDqPrefetch = 4;   // dQ kernel: K / V tiles prefetched to L2 this many key tiles ahead
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBoxBytes = 64 * BT * 2;    // one TMA box: 64 columns x 128 rows bf16
constexpr float kLog2e = 1.44269504088896340736f;

// dK/dV kernel: shared memory K | V | Q ring (Q tile + its rows' -L log2 e)
// | dO ring (dO tile + its rows' -delta); TMEM dV | dK | S^T | dP^T (then
// P^T and dS^T as bf16).  Q and dO have rings of their own so that each slot
// frees as soon as its last product (dK for Q, dV for dO) has read it.
template <int D>
struct CfgKV {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int KB = D / 64;
  static constexpr uint32_t TILE = BT * D * 2;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = TILE;
  static constexpr uint32_t SLOT = TILE + 1024;          // tile + 128 fp32 (padded)
  static constexpr uint32_t SLOT_ROWS = TILE;            // offset of the row values
  static constexpr uint32_t SLOT_TX = TILE + 512;
  static constexpr int NST = (D == 64) ? 4 : 2;          // query-tile ring depth
  static constexpr uint32_t OFF_QS = 2 * TILE;
  static constexpr uint32_t OFF_DS = OFF_QS + NST * SLOT;
  static constexpr uint32_t OFF_BAR = OFF_DS + NST * SLOT;
  // kv, kv free, q full[NST], q empty[NST], do full[NST], do empty[NST], s,
  // s read, dp, p[2], done, drain, item ring full[kRing], empty[kRing]
  static constexpr int NBAR = 2 + 4 * NST + 7 + 2 * kRing;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 4 * kRing;   // tmem slot, abort flag, item ring
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

// dQ kernel: shared memory = a ring of two-tile entries | a dQ staging tile;
// TMEM S | dP (dS) | dQ | Q | dO.  The query tile's Q and dO sit in TMEM as
// the A operands of S = Q K^T and dP = dO V^T, so those products read only
// K / V from shared memory (half the shared-memory operand traffic of two SS
// products).  The CTA is persistent; each item (query head, 128-query tile)
// sends one entry through the ring with its Q and dO, which the compute warps
// copy into TMEM, then one entry (K, V) per key tile.
template <int D>
struct CfgQ {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int KB = D / 64;
  static constexpr uint32_t TILE = BT * D * 2;
  static constexpr uint32_t OFF_STAGE = 0;
  static constexpr uint32_t ST_K = 0;                    // (Q in a Q / dO entry)
  static constexpr uint32_t ST_V = TILE;                 // (dO in a Q / dO entry)
  static constexpr uint32_t STAGE_BYTES = 2 * TILE;
  static constexpr int NST = (D == 64) ? 4 : 3;          // ring depth
  static constexpr uint32_t OFF_DQ = OFF_STAGE + NST * STAGE_BYTES;   // dQ (bf16) for its store
  static constexpr uint32_t OFF_BAR = OFF_DQ + TILE;
  // q (Q, dO in TMEM), full[NST], empty[NST], s, s read, dp[2], p[2], done,
  // drain, item ring full[kRing], empty[kRing]
  static constexpr int NBAR = 1 + 2 * NST + 8 + 2 * kRing;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 4 * kRing;   // tmem slot, abort flag, item ring
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
// -delta = -sum_k dO O (fp32) and -L log2(e) per (head, padded row).  D / 8
// threads per row, 16-byte loads, two rows per thread (both loads issued
// before either is used).
constexpr int kPrepThreads = 256;
template <int D>
__global__ void __launch_bounds__(kPrepThreads)
    attn_bwd_prep_kernel(const __nv_bfloat16 *__restrict__ O, const __nv_bfloat16 *__restrict__ dO,
                         const float *__restrict__ LSE, float *__restrict__ nl2,
                         float *__restrict__ ndl, int N, int N_pad) {
  constexpr int TPR = D / 8;                          // threads per row
  constexpr int RPB = kPrepThreads / TPR;             // rows per block and pass
  const int sub = threadIdx.x % TPR;
  const size_t bh = blockIdx.x;                       // one head per grid row
  const __nv_bfloat16 *Oh = O + bh * N * D;
  const __nv_bfloat16 *dOh = dO + bh * N * D;
  // The dK/dV kernel is a programmatic dependent of this one: it may take
  // the SMs this grid leaves and set up; it waits for this grid's rows
  // before it loads them.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
          ndl[r] = -acc;
          nl2[r] = -LSE[bh * N + ii[u]] * kLog2e;
        } else {   // padding row: P = 0 wherever it is read
          ndl[r] = 0.f;
          nl2[r] = -INFINITY;
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

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// In both kernels compute warps 4h..4h+3 own half h of the 128-wide score
// tile (query columns 0-63 / 64-127 in the dK/dV kernel, key columns in the
// dQ kernel) and hand it over on a barrier of its own; the MMA warp issues
// each half's gradient products (and, in the dQ kernel, its dP product for
// the next tile) as soon as that half is in, so one half's element work
// overlaps the other half's products.  The score product S (S^T) of the
// next tile goes out whole once every warp has read the current one.

// ------------------------------------------------------------------ dK / dV
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmdO,
                         const __grid_constant__ CUtensorMap tmdK,
                         const __grid_constant__ CUtensorMap tmdV, const float *__restrict__ nl2,
                         const float *__restrict__ ndl, int N, int N_pad, int H, int H_kv,
                         int BHkv, int n_blk, float scale_log2, float scale, unsigned *status,
                         unsigned *sched) {
  using C = CfgKV<D>;
  constexpr int NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work items are (K/V head, 128-key tile) pairs.  Causal: K/V heads vary
  // fastest and key tiles go in ascending order (the first key tiles are
  // seen by the most query tiles: longest first); non-causal: key tiles vary
  // fastest, so CTAs working at the same time share their head's Q and dO
  // through L2.  The CTA is persistent: it starts with item blockIdx and
  // claims further items from a global counter (sched[0]) once the current
  // item's loads are issued; the TMA warp passes each index on through a
  // ring in shared memory, and the last CTA to finish resets the counter.
  const int n_items = BHkv * n_blk;
  const int G = static_cast<int>(gridDim.x);
  const int group = H / H_kv;
  struct Item {
    int bkv, jt, it0, n_q, n_it;   // K/V head, key tile, first query tile, query tiles, steps
  };
  auto item_at = [&](int k, Item &it) {
    if (k >= n_items) return false;
    it.bkv = CAUSAL ? k % BHkv : k / n_blk;
    it.jt = CAUSAL ? k / BHkv : k % n_blk;
    it.it0 = CAUSAL ? it.jt : 0;
    it.n_q = n_blk - it.it0;                 // query tiles per query head
    it.n_it = group * it.n_q;                // (query head of the group, query tile) steps
    return true;
  };
  auto q_head = [&](const Item &it, int t) {
    return (it.bkv / H_kv) * H + (it.bkv % H_kv) * group + t / it.n_q;
  };
  auto q_tile = [&](const Item &it, int t) { return it.it0 + t % it.n_q; };

  // Barrier phases run on across items: the Q and dO rings count query tiles
  // over the CTA's whole sequence, S/dP/P count steps, K/V, K/V-free and done
  // complete once per item.
  const uint32_t bar0 = sb + C::OFF_BAR;
  const uint32_t B_KV = bar0;                                  // K, V of the item loaded
  const uint32_t B_KVE = bar0 + 8u;                            // K, V slots free (epilogue stored)
  auto B_QF = [&](int s) { return bar0 + 8u * (2 + s); };           // Q slot s loaded
  auto B_QE = [&](int s) { return bar0 + 8u * (2 + NST + s); };     // Q slot s free
  auto B_DF = [&](int s) { return bar0 + 8u * (2 + 2 * NST + s); };  // dO slot s loaded
  auto B_DE = [&](int s) { return bar0 + 8u * (2 + 3 * NST + s); };  // dO slot s free
  const uint32_t bar1 = bar0 + 8u * (2 + 4 * NST);
  const uint32_t B_S = bar1;                                   // S^T in TMEM
  const uint32_t B_SF = bar1 + 8;                              // S^T read: region free
  const uint32_t B_DP = bar1 + 16;                             // dP^T in TMEM
  auto B_P = [&](int h) { return bar1 + 24 + 8u * h; };     // P^T, dS^T half h written
  const uint32_t B_DONE = bar1 + 40;                           // item's last products done
  const uint32_t B_DRAIN = bar1 + 48;
  auto B_IF = [&](int s) { return bar1 + 56 + 8u * s; };       // item slot s written
  auto B_IE = [&](int s) { return bar1 + 56 + 8u * (kRing + s); };   // item slot s read by all
  static_assert(2 + 4 * NST + 7 + 2 * kRing == C::NBAR, "barrier count");
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  volatile int *item_ring = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 16);
  // The t-th item of this CTA as the TMA warp published it (warp-uniform).
  auto take_item = [&](int t, Item &it, bool &ok) {
    const int s = t % kRing;
    if (!__all_sync(0xffffffffu, mbar_wait(B_IF(s), (t / kRing) & 1, status, abort_flag))) {
      ok = false;
      return false;
    }
    const int k = item_ring[s];
    __syncwarp();
    if (lane == 0) mbar_arrive(B_IE(s));
    return item_at(k, it);
  };
  auto load_kv = [&](const Item &it) {
    mbar_arrive_expect_tx(B_KV, 2 * C::TILE);
    for (int kb = 0; kb < C::KB; ++kb) {
      tma_load_3d(sb + C::OFF_K + kb * kBoxBytes, &tmK, kb * 64, it.jt * BT, it.bkv, B_KV);
      tma_load_3d(sb + C::OFF_V + kb * kBoxBytes, &tmV, kb * 64, it.jt * BT, it.bkv, B_KV);
    }
  };

  if (threadIdx.x == kWarpTMA * 32) {
    mbar_init(B_KV, 1);
    mbar_init(B_KVE, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(B_QF(s), 1);
      mbar_init(B_QE(s), 1);
      mbar_init(B_DF(s), 1);
      mbar_init(B_DE(s), 1);
    }
    mbar_init(B_S, 1);
    mbar_init(B_SF, kComputeWarps);
    mbar_init(B_DP, 1);
    for (int h = 0; h < 2; ++h) mbar_init(B_P(h), kComputeWarps / 2);
    mbar_init(B_DONE, 1);
    mbar_init(B_DRAIN, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(B_IF(s), 1);
      mbar_init(B_IE(s), 1 + kComputeWarps);   // the MMA warp and every compute warp
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmdK);
    tma_prefetch_desc(&tmdV);
    Item it0;
    if (item_at(static_cast<int>(blockIdx.x), it0)) load_kv(it0);   // (the grid is no larger than the item count)
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The dQ kernel may launch as SMs free up; it reads nothing this grid
  // writes, and it waits for this grid (and so for the row pass) before it
  // reads L and delta.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == kWarpTMA) {
    // ------------------------------------------------------------ TMA
    const bool leader = elect_one();
    // -L log2(e) and -delta come from the row pass launched just before this
    // kernel (programmatic dependent launch): the first load of them waits
    // for it; Q, dO, K and V are inputs of the whole call and load at once.
    bool rows_ready = false;
    int g = 0;                               // stages issued so far
    int gd = 0;                              // dO loads issued so far
    int kv_items = 1;                        // items whose K/V load was issued
    bool ok = true;
    int k = static_cast<int>(blockIdx.x);
    // Query tile t of the item into slot g % NST of each ring: Q with its
    // rows' -L log2(e), then dO with their -delta, each once its slot is free.
    auto load_stage = [&](const Item &it, int t) {
      const int s = g % NST;
      const uint32_t par = ((g / NST) & 1) ^ 1u;
      const int bh = q_head(it, t);
      const int qt = q_tile(it, t);
      const size_t row0 = static_cast<size_t>(bh) * N_pad + static_cast<size_t>(qt) * BT;
      if (!__all_sync(0xffffffffu, mbar_wait(B_QE(s), par, status, abort_flag))) return false;
      if (leader) {
        const uint32_t st = sb + C::OFF_QS + s * C::SLOT;
        mbar_arrive_expect_tx(B_QF(s), C::SLOT_TX);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(st + kb * kBoxBytes, &tmQ, kb * 64, qt * BT, bh, B_QF(s));
        if (!rows_ready) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          rows_ready = true;
        }
        bulk_load_1d(st + C::SLOT_ROWS, nl2 + row0, BT * 4, B_QF(s));
      }
      ++g;
      if (!__all_sync(0xffffffffu, mbar_wait(B_DE(s), par, status, abort_flag))) return false;
      if (leader) {
        const uint32_t st = sb + C::OFF_DS + s * C::SLOT;
        mbar_arrive_expect_tx(B_DF(s), C::SLOT_TX);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(st + kb * kBoxBytes, &tmdO, kb * 64, qt * BT, bh, B_DF(s));
        bulk_load_1d(st + C::SLOT_ROWS, ndl + row0, BT * 4, B_DF(s));
      }
      ++gd;
      return true;
    };
    for (int t = 0; ok; ++t) {
      const int s = t % kRing;
      if (!(ok = __all_sync(0xffffffffu,
                            mbar_wait(B_IE(s), ((t / kRing) & 1) ^ 1u, status, abort_flag))))
        break;
      if (leader) {
        item_ring[s] = k;
        mbar_arrive(B_IF(s));
      }
      __syncwarp();
      Item it;
      if (!item_at(k, it)) break;
      // The item's first stages go out at once; its K and V once the
      // previous item's epilogue has stored dK and dV out of their slots.
      const int first = it.n_it < NST ? it.n_it : NST;
      int u = 0;
      for (; ok && u < first; ++u) ok = load_stage(it, u);
      if (ok && t > 0) {
        if (!(ok = __all_sync(0xffffffffu,
                              mbar_wait(B_KVE, (t - 1) & 1, status, abort_flag))))
          break;
        if (leader) load_kv(it);
        kv_items = t + 1;
      }
      for (; ok && u < it.n_it; ++u) ok = load_stage(it, u);
      // This item's loads are all issued: claim the next one.
      int kn = 0;
      if (lane == 0) kn = G + static_cast<int>(atomicAdd(sched, 1u));
      k = __shfl_sync(0xffffffffu, kn, 0);
    }
    if (leader && *abort_flag) {
      // Let every copy this warp started land before the CTA exits.
      mbar_wait_drain(B_KV, (kv_items - 1) & 1, 100000000ull);
      for (int j = 0; j < NST && j < g; ++j) {
        const int tt = g - 1 - j;
        mbar_wait_drain(B_QF(tt % NST), (tt / NST) & 1, 100000000ull);
      }
      for (int j = 0; j < NST && j < gd; ++j) {
        const int tt = gd - 1 - j;
        mbar_wait_drain(B_DF(tt % NST), (tt / NST) & 1, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------------ MMA
    const bool leader = elect_one();
    constexpr uint32_t kIdescS = make_idesc_bf16(BT, BT, 0, 0);
    constexpr uint32_t kIdescG = make_idesc_bf16(BT, D, 0, 1);
    // Low words of the shared-memory descriptors (one common high word):
    // K-major (head dim contiguous, 16-element k-steps inside a 64-column
    // box) and MN-major (a slot's Q / dO as B operands with the query
    // index as the reduction dimension: 16-row k-steps, 64-column boxes
    // kBoxBytes apart).
    const uint64_t dK0 = make_sdesc_sw128(sb + C::OFF_K, 16, 1024);
    const uint32_t hi = static_cast<uint32_t>(dK0 >> 32);
    const uint32_t k_lo = static_cast<uint32_t>(dK0);
    const uint32_t v_lo = static_cast<uint32_t>(make_sdesc_sw128(sb + C::OFF_V, 16, 1024));
    const uint32_t qk_lo = static_cast<uint32_t>(make_sdesc_sw128(sb + C::OFF_QS, 16, 1024));
    const uint32_t dk_lo = static_cast<uint32_t>(make_sdesc_sw128(sb + C::OFF_DS, 16, 1024));
    const uint32_t qm_lo =
        static_cast<uint32_t>(make_sdesc_sw128(sb + C::OFF_QS, kBoxBytes, 1024));
    const uint32_t dm_lo =
        static_cast<uint32_t>(make_sdesc_sw128(sb + C::OFF_DS, kBoxBytes, 1024));
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort_flag));
    };
    // S^T = K Q^T and dP^T = V dO^T over the whole query tile (N = 128:
    // SS products at N = 64 are bound by shared-memory reads).
    auto issue_st = [&](int s) {
      const uint32_t so = (s * C::SLOT) >> 4;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
        mma_bf16_ss_lo(tmem + C::TM_ST, k_lo + koff, qk_lo + so + koff, hi, kIdescS,
                       kk > 0 ? 1u : 0u);
      }
      mma_commit(B_S);
    };
    auto issue_dpt = [&](int s) {
      const uint32_t so = (s * C::SLOT) >> 4;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
        mma_bf16_ss_lo(tmem + C::TM_DPT, v_lo + koff, dk_lo + so + koff, hi, kIdescS,
                       kk > 0 ? 1u : 0u);
      }
      mma_commit(B_DP);
    };
    // Half h of dK += dS^T Q (dk) or dV += P^T dO (!dk): the 16-query steps
    // 4h..4h+3, A from TMEM, B = the slot's Q / dO, MN-major.  The compute
    // warps left query step u (16 queries) of half h as P^T in dP^T columns
    // 64h + 16u .. +7 and dS^T in 64h + 16u + 8 .. +15.
    auto issue_grad = [&](int s, int h, bool dk, bool acc) {
      const uint32_t so = (s * C::SLOT) >> 4;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int kk = 4 * h + u;
        const uint32_t boff = (kk * 16 * 128) >> 4;
        const uint32_t col = C::TM_DPT + 64 * h + 16 * u + (dk ? 8 : 0);
        mma_bf16_ts_lo(tmem + (dk ? C::TM_DK : C::TM_DV), tmem + col,
                       (dk ? qm_lo : dm_lo) + so + boff, hi, kIdescG, (acc || u > 0) ? 1u : 0u);
      }
    };
    // Issuing an MMA waits while the tensor pipe's queue is full, so this
    // warp is never far ahead of the pipe, and a barrier round trip between
    // two batches would leave the pipe idle.  Each barrier is therefore
    // tested (non-blocking, every lane) before the batch ahead of it and the
    // result read after the batch; only a phase not yet complete then takes
    // the bounded wait.
    auto ready = [&](uint32_t tst, uint32_t bar, uint32_t parity) {
      return vote_all_ordered(tst) || wait_all(bar, parity);
    };
    bool ok = true;
    int g = 0;                               // stages consumed so far (= steps before this item)
    for (int t = 0; ok; ++t) {
      Item it;
      if (!take_item(t, it, ok)) break;
      const int n_it = it.n_it;
      // The item's K and V, and its first stage.  dV and dK of the previous
      // item were read out by its epilogue before the compute warps handed
      // over this item's first P^T / dS^T, so the first gradient products
      // below may overwrite them; the epilogue also came after the last
      // reads of S^T and dP^T.
      const uint32_t par0 = (g / NST) & 1;
      ok = wait_all(B_KV, t & 1) && wait_all(B_QF(g % NST), par0) &&
           wait_all(B_DF(g % NST), par0);
      if (ok) {
        tc_fence_after();
        if (leader) {
          issue_st(g % NST);
          issue_dpt(g % NST);
        }
        __syncwarp();
      }
      // Per query tile, in the tensor pipe: S^T of the next tile (once the
      // compute warps have read this one's: P^T and dS^T go over dP^T), dK of
      // this tile (each half once the compute warps hand it over; the Q slot
      // is then free), dV of this tile (the dO slot is then free), dP^T of the
      // next tile (after the products that read the P^T / dS^T it
      // overwrites: MMAs from one thread run in issue order).  Freeing each
      // slot after its last product lets the next loads start a quarter of a
      // step earlier than a shared Q / dO stage would.
      uint32_t t_qf = 0, t_sf = 0;
      for (int u = 0; ok && u < n_it; ++u) {
        const int gs = g + u, s = gs % NST, g1 = gs + 1, s1 = g1 % NST;
        const uint32_t par1 = (g1 / NST) & 1;
        const bool more = u + 1 < n_it;
        uint32_t t_p = 0;
        if (more) {
          if (!(ok = ready(t_qf, B_QF(s1), par1) && ready(t_sf, B_SF, gs & 1))) break;
          t_p = mbar_test(B_P(0), gs & 1);
          tc_fence_after();
          if (leader) issue_st(s1);
          __syncwarp();
        }
        if (!(ok = ready(t_p, B_P(0), gs & 1))) break;
        t_p = mbar_test(B_P(1), gs & 1);
        tc_fence_after();
        if (leader) issue_grad(s, 0, true, u > 0);
        __syncwarp();
        if (!(ok = ready(t_p, B_P(1), gs & 1))) break;
        const uint32_t t_df = more ? mbar_test(B_DF(s1), par1) : 0u;
        if (u + 2 < n_it) {
          t_qf = mbar_test(B_QF((gs + 2) % NST), ((gs + 2) / NST) & 1);
          t_sf = mbar_test(B_SF, g1 & 1);
        }
        tc_fence_after();
        if (leader) {
          issue_grad(s, 1, true, true);
          mma_commit(B_QE(s));
          issue_grad(s, 0, false, u > 0);
          issue_grad(s, 1, false, true);
          mma_commit(B_DE(s));
          if (!more) mma_commit(B_DONE);
        }
        __syncwarp();
        if (more) {
          if (!(ok = ready(t_df, B_DF(s1), par1))) break;
          tc_fence_after();
          if (leader) issue_dpt(s1);
          __syncwarp();
        }
      }
      g += n_it;
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
    int g = 0;                               // steps of earlier items
    for (int t = 0; ok; ++t) {
      Item itm;
      if (!take_item(t, itm, ok)) break;
      for (int u = 0; u < itm.n_it; ++u) {
        const int gs = g + u, s = gs % NST;
        const int it = q_tile(itm, u);
        // (Usually both complete already: tested together, they cost one
        // shared-memory round trip instead of two on the warps' chain.)
        ok = mbar_wait2_all(B_QF(s), (gs / NST) & 1, B_S, gs & 1, status, abort_flag);
        if (!ok) break;
        tc_fence_after();
        // The slots' -L log2(e) and -delta, one per query column.
        const float *nl_s =
            reinterpret_cast<const float *>(smem + C::OFF_QS + s * C::SLOT + C::SLOT_ROWS);
        const float *nd_s =
            reinterpret_cast<const float *>(smem + C::OFF_DS + s * C::SLOT + C::SLOT_ROWS);
        const bool diag = CAUSAL && it == itm.jt;
        // P^T for the half's 64 queries while the dP^T product is still running.
        const float2 sc2 = make_float2(scale_log2, scale_log2);
        float p[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col0 = 64 * h + 32 * c;
          uint32_t sr[32];
          tmem_ld_32cols(tmem + lane_base + C::TM_ST + col0, sr);
          tmem_ld_wait_regs(sr);
          if (c == 1) {
            // This warp's S^T is in registers: once every warp's is, the
            // region may take the next tile's S^T.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B_SF);
          }
#pragma unroll
          for (int k = 0; k < 32; k += 4) {
            const float4 lv = *reinterpret_cast<const float4 *>(nl_s + col0 + k);
            const float2 x0 = ffma2(
                make_float2(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), sc2,
                make_float2(lv.x, lv.y));
            const float2 x1 = ffma2(
                make_float2(__uint_as_float(sr[k + 2]), __uint_as_float(sr[k + 3])), sc2,
                make_float2(lv.z, lv.w));
            p[32 * c + k] = ex2_approx(x0.x);
            p[32 * c + k + 1] = ex2_approx(x0.y);
            p[32 * c + k + 2] = ex2_approx(x1.x);
            p[32 * c + k + 3] = ex2_approx(x1.y);
          }
        }
        if (diag) {   // (warp-uniform) query before key: masked
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (64 * h + e < row) p[e] = 0.f;
        }
        if (!(ok = mbar_wait2_all(B_DF(s), (gs / NST) & 1, B_DP, gs & 1, status, abort_flag)))
          break;
        tc_fence_after();
        {
          // dS^T = P^T (dP^T - delta) in four 16-query steps, each loading the
          // next step's dP^T columns while it computes; P^T and dS^T of a step
          // (bf16 pairs, 8 columns each) go over its 16 dP^T columns.
          const uint32_t dbase = tmem + lane_base + C::TM_DPT + 64 * h;
          uint32_t da[16], db[16];
          auto dstep = [&](auto kc, const uint32_t (&dp)[16]) {
            constexpr int k = decltype(kc)::value;
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const float4 dv = *reinterpret_cast<const float4 *>(nd_s + 64 * h + 16 * k + i);
              const float2 d0 = fadd2(make_float2(__uint_as_float(dp[i]), __uint_as_float(dp[i + 1])),
                                      make_float2(dv.x, dv.y));
              const float2 d1 = fadd2(
                  make_float2(__uint_as_float(dp[i + 2]), __uint_as_float(dp[i + 3])),
                  make_float2(dv.z, dv.w));
              const float2 s0 = fmul2(make_float2(p[16 * k + i], p[16 * k + i + 1]), d0);
              const float2 s1 = fmul2(make_float2(p[16 * k + i + 2], p[16 * k + i + 3]), d1);
              w[i / 2] = pack_bf16x2(p[16 * k + i], p[16 * k + i + 1]);
              w[i / 2 + 1] = pack_bf16x2(p[16 * k + i + 2], p[16 * k + i + 3]);
              w[8 + i / 2] = pack_bf16x2(s0.x, s0.y);
              w[8 + i / 2 + 1] = pack_bf16x2(s1.x, s1.y);
            }
            tmem_st_16cols(dbase + 16 * k, w);
          };
          tmem_ld_16cols(dbase, da);
          tmem_ld_wait_regs16(da);
          tmem_ld_16cols(dbase + 16, db);
          dstep(std::integral_constant<int, 0>(), da);
          tmem_ld_wait_regs16(db);
          tmem_ld_16cols(dbase + 32, da);
          dstep(std::integral_constant<int, 1>(), db);
          tmem_ld_wait_regs16(da);
          tmem_ld_16cols(dbase + 48, db);
          dstep(std::integral_constant<int, 2>(), da);
          tmem_ld_wait_regs16(db);
          dstep(std::integral_constant<int, 3>(), db);
        }
        tmem_st_wait();
        // The slots' -L / -delta were read through the generic proxy and the
        // next TMA refill writes them through the async proxy.
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B_P(h));
      }
      // Epilogue of the item: dV and dK staged as bf16 in the V and K slots
      // (free once the item's last products are done) and stored by TMA; the
      // storing thread then frees the slots for the next item's K and V.
      // The compute warps agree first, so that they all take part in the
      // barrier or all leave.
      const bool okd = ok && __all_sync(0xffffffffu, mbar_wait(B_DONE, t & 1, status, abort_flag));
      if (named_bar_any(kEpiBar, 32 * kComputeWarps, !okd)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t st_dv = sb + C::OFF_V;
      const uint32_t st_dk = sb + C::OFF_K;
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
      tc_fence_before();
      named_bar_sync(kEpiBar, 32 * kComputeWarps);
      if (threadIdx.x == 0) {
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_store_3d(&tmdV, kb * 64, itm.jt * BT, itm.bkv, st_dv + kb * kBoxBytes);
          tma_store_3d(&tmdK, kb * 64, itm.jt * BT, itm.bkv, st_dk + kb * kBoxBytes);
        }
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(B_KVE);
      }
      g += itm.n_it;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // Every claim of this CTA is behind it: the last CTA to get here resets
  // the item counter (sched[0]) and this count (sched[1]) for the next launch.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(sched, 0u);
      atomicExch(sched + 1, 0u);
    }
  }
}

// ------------------------------------------------------------------ dQ
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmdQ,
                       const float *__restrict__ nl2, const float *__restrict__ ndl,
                       int N, int N_pad, int H, int H_kv, int BH, int n_blk, float scale_log2,
                       float scale, unsigned *status, unsigned *sched) {
  using C = CfgQ<D>;
  constexpr int NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work items are (query head, 128-query tile) pairs.  Causal: heads vary
  // fastest and query tiles go in descending order (longest first);
  // non-causal: query tiles vary fastest, so the CTAs working at the same
  // time share a few heads' K/V through L2.  The CTA is persistent: it
  // starts with item blockIdx and claims each further item from a global
  // counter (sched[0]) once it has issued the current one's loads; the TMA
  // warp hands the item indices to the others through a small ring in shared
  // memory, and the last CTA to finish resets the counter.
  const int n_items = BH * n_blk;
  const int G = static_cast<int>(gridDim.x);
  const int group = H / H_kv;
  struct Item {
    int bh, kvh, it, n_j;   // query head, K/V head, query tile, key tiles
  };
  auto item_at = [&](int k, Item &w) {
    if (k >= n_items) return false;
    w.bh = CAUSAL ? k % BH : k / n_blk;
    w.it = CAUSAL ? n_blk - 1 - k / BH : k % n_blk;
    w.kvh = (w.bh / H) * H_kv + (w.bh % H) / group;
    w.n_j = CAUSAL ? w.it + 1 : n_blk;
    return true;
  };

  // Ring entries run on across items: item t's Q / dO entry, then its n_j
  // (K, V) entries, then item t + 1's.  Per-step barriers (S, S read, dP,
  // P) count key tiles over the CTA's whole sequence; Q-in-TMEM and done
  // complete once per item.
  const uint32_t bar0 = sb + C::OFF_BAR;
  const uint32_t B_Q = bar0;   // the compute warps have put the item's Q and dO into TMEM
  auto B_FULL = [&](int s) { return bar0 + 8u * (1 + s); };
  auto B_EMPTY = [&](int s) { return bar0 + 8u * (1 + NST + s); };
  const uint32_t bar1 = bar0 + 8u * (1 + 2 * NST);
  const uint32_t B_S = bar1;                                   // S in TMEM
  const uint32_t B_SF = bar1 + 8;                              // S read: region free
  auto B_DP = [&](int h) { return bar1 + 8u * (2 + h); };   // dP half h in TMEM
  auto B_P = [&](int h) { return bar1 + 8u * (4 + h); };    // dS half h written (over dP)
  const uint32_t B_DONE = bar1 + 48;                           // item's last products done
  const uint32_t B_DRAIN = bar1 + 56;
  auto B_IF = [&](int s) { return bar1 + 64 + 8u * s; };       // item slot s written
  auto B_IE = [&](int s) { return bar1 + 64 + 8u * (kRing + s); };   // item slot s read by all
  static_assert(1 + 2 * NST + 8 + 2 * kRing == C::NBAR, "barrier count");
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  volatile int *item_ring = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 16);
  // The t-th item of this CTA as the TMA warp published it (warp-uniform).
  auto take_item = [&](int t, Item &w, bool &ok) {
    const int s = t % kRing;
    if (!__all_sync(0xffffffffu, mbar_wait(B_IF(s), (t / kRing) & 1, status, abort_flag))) {
      ok = false;
      return false;
    }
    const int k = item_ring[s];
    __syncwarp();
    if (lane == 0) mbar_arrive(B_IE(s));
    return item_at(k, w);
  };

  if (threadIdx.x == kWarpTMA * 32) {
    mbar_init(B_Q, kComputeWarps);
    for (int s = 0; s < NST; ++s) {
      mbar_init(B_FULL(s), 1);
      mbar_init(B_EMPTY(s), 1);
    }
    mbar_init(B_S, 1);
    mbar_init(B_SF, kComputeWarps);
    for (int h = 0; h < 2; ++h) {
      mbar_init(B_DP(h), 1);
      mbar_init(B_P(h), kComputeWarps / 2);
    }
    mbar_init(B_DONE, 1);
    mbar_init(B_DRAIN, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(B_IF(s), 1);
      mbar_init(B_IE(s), 1 + kComputeWarps);   // the MMA warp and every compute warp
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdQ);
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
    // (Q, dO, K and V are inputs of the whole call: no wait for the kernels
    // launched before this one.)
    const bool leader = elect_one();
    int e = 0;                               // ring entries issued
    bool ok = true;
    int k = static_cast<int>(blockIdx.x);
    // The next entry's slot, once the consumers of its previous use freed it.
    auto next_slot = [&](uint32_t &st) {
      const int s = e % NST;
      st = sb + C::OFF_STAGE + s * C::STAGE_BYTES;
      return __all_sync(0xffffffffu,
                        mbar_wait(B_EMPTY(s), ((e / NST) & 1) ^ 1u, status, abort_flag));
    };
    for (int t = 0; ok; ++t) {
      const int r = t % kRing;
      if (!(ok = __all_sync(0xffffffffu,
                            mbar_wait(B_IE(r), ((t / kRing) & 1) ^ 1u, status, abort_flag))))
        break;
      if (leader) {
        item_ring[r] = k;
        mbar_arrive(B_IF(r));
      }
      __syncwarp();
      Item w;
      if (!item_at(k, w)) break;
      uint32_t st;
      if (!(ok = next_slot(st))) break;
      if (leader) {
        mbar_arrive_expect_tx(B_FULL(e % NST), 2 * C::TILE);
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_3d(st + C::ST_K + kb * kBoxBytes, &tmQ, kb * 64, w.it * BT, w.bh, B_FULL(e % NST));
          tma_load_3d(st + C::ST_V + kb * kBoxBytes, &tmdO, kb * 64, w.it * BT, w.bh, B_FULL(e % NST));
        }
      }
      ++e;
      for (int j = 0; ok && j < w.n_j; ++j) {
        // K / V tiles kDqPrefetch key tiles ahead go to L2 first, so that the
        // ring's loads (issued once a slot frees, a step or two before use)
        // find them there (causal B4 H16 N2048: 209.3 -> 207.4 us for the
        // whole backward; 6 or 8 ahead gave nothing).
        if (leader && j + kDqPrefetch < w.n_j) {
          for (int kb = 0; kb < C::KB; ++kb) {
            tma_prefetch_l2_3d(&tmK, kb * 64, (j + kDqPrefetch) * BT, w.kvh);
            tma_prefetch_l2_3d(&tmV, kb * 64, (j + kDqPrefetch) * BT, w.kvh);
          }
        }
        if (!(ok = next_slot(st))) break;
        if (leader) {
          mbar_arrive_expect_tx(B_FULL(e % NST), 2 * C::TILE);
          for (int kb = 0; kb < C::KB; ++kb) {
            tma_load_3d(st + C::ST_K + kb * kBoxBytes, &tmK, kb * 64, j * BT, w.kvh, B_FULL(e % NST));
            tma_load_3d(st + C::ST_V + kb * kBoxBytes, &tmV, kb * 64, j * BT, w.kvh, B_FULL(e % NST));
          }
        }
        ++e;
      }
      // This item's loads are all issued: claim the next one.
      int kn = 0;
      if (lane == 0) kn = G + static_cast<int>(atomicAdd(sched, 1u));
      k = __shfl_sync(0xffffffffu, kn, 0);
    }
    if (leader && *abort_flag) {
      // Let every copy this warp started land before the CTA exits.
      for (int u = 0; u < NST && u < e; ++u) {
        const int x = e - 1 - u;
        mbar_wait_drain(B_FULL(x % NST), (x / NST) & 1, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------------ MMA
    const bool leader = elect_one();
    constexpr uint32_t kIdescS = make_idesc_bf16(BT, BT / 2, 0, 0);
    constexpr uint32_t kIdescS2 = make_idesc_bf16(BT, BT, 0, 0);
    constexpr uint32_t kIdescG = make_idesc_bf16(BT, D, 0, 1);
    const uint64_t dst0 = make_sdesc_sw128(sb + C::OFF_STAGE, 16, 1024);
    const uint32_t hi = static_cast<uint32_t>(dst0 >> 32);
    const uint32_t stk_lo = static_cast<uint32_t>(dst0);
    const uint32_t stm_lo =
        static_cast<uint32_t>(make_sdesc_sw128(sb + C::OFF_STAGE, kBoxBytes, 1024));
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort_flag));
    };
    // S = Q K^T over the whole key tile (N = 128), Q from TMEM (8 columns per
    // 16-element step of the head dim).
    auto issue_s = [&](int s) {
      const uint32_t so = (s * C::STAGE_BYTES) >> 4;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
        mma_bf16_ts_lo(tmem + C::TM_S, tmem + C::TM_Q + 8 * kk,
                       stk_lo + so + (C::ST_K >> 4) + koff, hi, kIdescS2, kk > 0 ? 1u : 0u);
      }
      mma_commit(B_S);
    };
    // Half h of dP = dO V^T: keys 64h..64h+63 of the tile, dO from TMEM.
    auto issue_dp = [&](int s, int h) {
      const uint32_t so = (s * C::STAGE_BYTES + h * 64 * 128) >> 4;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
        mma_bf16_ts_lo(tmem + C::TM_DP + 64 * h, tmem + C::TM_DO + 8 * kk,
                       stk_lo + so + (C::ST_V >> 4) + koff, hi, kIdescS, kk > 0 ? 1u : 0u);
      }
      mma_commit(B_DP(h));
    };
    // Half h of dQ += dS K: key steps 4h..4h+3, dS from TMEM (columns
    // 64h..64h+31 of the dP region), K MN-major (16-key steps).
    auto issue_dq = [&](int s, int h, bool acc) {
      const uint32_t so = (s * C::STAGE_BYTES) >> 4;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int kk = 4 * h + u;
        const uint32_t boff = (kk * 16 * 128) >> 4;
        mma_bf16_ts_lo(tmem + C::TM_DQ, tmem + C::TM_DP + 64 * h + 8 * u,
                       stm_lo + so + (C::ST_K >> 4) + boff, hi, kIdescG, (acc || u > 0) ? 1u : 0u);
      }
    };
    // Issuing an MMA waits while the tensor pipe's queue is full, so this
    // warp is never far ahead of the pipe, and a barrier round trip between
    // two batches would leave the pipe idle.  Each barrier is therefore
    // tested (non-blocking, every lane) before the batch ahead of it and the
    // result read after the batch; only a phase not yet complete then takes
    // the bounded wait.
    auto ready = [&](uint32_t tst, uint32_t bar, uint32_t parity) {
      return vote_all_ordered(tst) || wait_all(bar, parity);
    };
    bool ok = true;
    int e = 0;                               // ring entries consumed
    int g = 0;                               // key tiles of earlier items
    for (int t = 0; ok; ++t) {
      Item w;
      if (!take_item(t, w, ok)) break;
      const int n_j = w.n_j;
      // The item's Q and dO are in TMEM once the compute warps have copied
      // them out of its first entry (after their last reads of the previous
      // item's S and the completion of its last dP products, the only
      // readers of the old Q and dO): that entry's slot is free.  Its S and
      // dP then overwrite regions whose previous contents the compute warps
      // have read (S) or the previous item's last dQ products, issued before
      // them, read (dS over dP).
      ok = wait_all(B_Q, t & 1);
      if (ok && leader) mbar_arrive(B_EMPTY(e % NST));
      ++e;
      ok = ok && wait_all(B_FULL(e % NST), (e / NST) & 1);
      if (ok) {
        tc_fence_after();
        if (leader) {
          issue_s(e % NST);
          issue_dp(e % NST, 0);
          issue_dp(e % NST, 1);
        }
        __syncwarp();
      }
      // Per key tile j: S of tile j + 1 goes out as soon as the compute
      // warps have read S of tile j (dS is written over dP, not over S), so
      // the next tile's exponentials overlap this tile's dQ and dP products;
      // dP half h of tile j + 1 follows dQ half h of tile j, which reads the
      // dS it overwrites (MMAs from one thread run in issue order).
      uint32_t t_full = 0, t_sf = 0;         // tests of the next tile's K/V and S-read phases
      for (int j = 0; ok && j < n_j; ++j) {
        const int gs = g + j, ej = e + j, s = ej % NST, s1 = (ej + 1) % NST;
        const bool more = j + 1 < n_j;
        uint32_t t_p = 0;
        if (more) {
          if (!(ok = ready(t_full, B_FULL(s1), ((ej + 1) / NST) & 1) &&
                     ready(t_sf, B_SF, gs & 1)))
            break;
          t_p = mbar_test(B_P(0), gs & 1);
          tc_fence_after();
          if (leader) issue_s(s1);
          __syncwarp();
        }
        if (!(ok = ready(t_p, B_P(0), gs & 1))) break;
        t_p = mbar_test(B_P(1), gs & 1);
        tc_fence_after();
        if (leader) {
          issue_dq(s, 0, j > 0);
          if (more) issue_dp(s1, 0);
        }
        __syncwarp();
        if (!(ok = ready(t_p, B_P(1), gs & 1))) break;
        if (j + 2 < n_j) {
          t_full = mbar_test(B_FULL((ej + 2) % NST), ((ej + 2) / NST) & 1);
          t_sf = mbar_test(B_SF, (gs + 1) & 1);
        }
        tc_fence_after();
        if (leader) {
          issue_dq(s, 1, true);
          mma_commit(B_EMPTY(s));
          if (more) issue_dp(s1, 1);
          else mma_commit(B_DONE);
        }
        __syncwarp();
      }
      e += n_j;
      g += n_j;
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
    const uint32_t st_dq = sb + C::OFF_DQ;
    auto row_of = [&](const Item &w) {
      return static_cast<size_t>(w.bh) * N_pad + static_cast<size_t>(w.it) * BT + row;
    };
    // Ring entry eq (an item's Q and dO) into TMEM: warps of half 0 copy the
    // Q rows, warps of half 1 the dO rows (row = lane, bf16 pairs along the
    // columns; the TMA load left rows past N zero).  A 128-byte row of a box
    // holds its 16-byte chunk v at position v ^ (row % 8) (128-byte swizzle),
    // so the 32 lanes' loads of one chunk fall in distinct banks.  Called
    // after this warp's last reads of the previous item's S (half 0) or dP
    // (half 1), so the previous item's S / dP products, the only readers of
    // the old Q / dO, have completed.
    auto copy_qdo = [&](int eq) {
      const int s = eq % NST;
      if (!__all_sync(0xffffffffu, mbar_wait(B_FULL(s), (eq / NST) & 1, status, abort_flag)))
        return false;
      const uint32_t src =
          sb + C::OFF_STAGE + s * C::STAGE_BYTES + (h == 0 ? C::ST_K : C::ST_V) + row * 128;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const uint4 y = ld_shared_v4(src + c * kBoxBytes + ((x ^ (row & 7)) << 4));
          v[4 * x] = y.x;
          v[4 * x + 1] = y.y;
          v[4 * x + 2] = y.z;
          v[4 * x + 3] = y.w;
        }
        tmem_st_32cols(tmem + lane_base + (h == 0 ? C::TM_Q : C::TM_DO) + 32 * c, v);
      }
      tmem_st_wait();
      // The TMA warp refills this slot (async proxy) after the reads above.
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B_Q);
      return true;
    };
    bool ok = true;
    int e = 0;                               // ring entry of the current item's Q / dO
    int g = 0;                               // key tiles of earlier items
    Item cur;
    bool have = take_item(0, cur, ok);
    if (have) ok = copy_qdo(e);
    // This kernel is a programmatic dependent of the dK/dV kernel, which
    // itself waited for the row pass: once that grid has finished, the row
    // pass's -L log2(e) and -delta are complete too.  Q, dO, K and V are
    // inputs: the first item's Q / dO copy above and its first products do
    // not wait.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float nl = 0.f, nd = 0.f;
    if (have) {
      nl = nl2[row_of(cur)];
      nd = ndl[row_of(cur)];
    }
    const float2 sc2 = make_float2(scale_log2, scale_log2);
    for (int t = 0;; ++t) {
      // The compute warps agree at each item (and at its epilogue below) on
      // whether to go on, so that they all take part in every named barrier
      // or all leave: every one has the item and no wait has given up.
      if (named_bar_any(kEpiBar, 32 * kComputeWarps, !(have && ok))) break;
      const int n_j = cur.n_j;
      const float2 nl2v = make_float2(nl, nl);
      const float2 nd2 = make_float2(nd, nd);
      for (int j = 0; ok && j < n_j; ++j) {
        const int gs = g + j;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(B_S, gs & 1, status, abort_flag)))) break;
        tc_fence_after();
        const bool diag = CAUSAL && j == cur.it;
        const int kmax = N - j * BT;          // keys past the sequence are masked
        float p[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col0 = 64 * h + 32 * c;
          uint32_t sr[32];
          tmem_ld_32cols(tmem + lane_base + C::TM_S + col0, sr);
          tmem_ld_wait_regs(sr);
          if (c == 1) {
            // This warp's S is in registers: once every warp's is, the
            // region may take the next tile's S.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B_SF);
          }
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float2 x =
                ffma2(make_float2(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), sc2, nl2v);
            p[32 * c + k] = ex2_approx(x.x);
            p[32 * c + k + 1] = ex2_approx(x.y);
          }
        }
        if (diag || kmax < BT) {   // (warp-uniform) key after query, or past N: masked
#pragma unroll
          for (int x = 0; x < 64; ++x) {
            const int col = 64 * h + x;
            if ((diag && col > row) || col >= kmax) p[x] = 0.f;
          }
        }
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(B_DP(h), gs & 1, status, abort_flag))))
          break;
        tc_fence_after();
        // dS as bf16 pairs over the first 32 columns of the half's dP region
        // (chunk c's 16 columns over dP columns already read).
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col0 = 64 * h + 32 * c;
          uint32_t dp[32];
          tmem_ld_32cols(tmem + lane_base + C::TM_DP + col0, dp);
          tmem_ld_wait_regs(dp);
          uint32_t dk[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float2 d =
                fadd2(make_float2(__uint_as_float(dp[k]), __uint_as_float(dp[k + 1])), nd2);
            const float2 ds = fmul2(make_float2(p[32 * c + k], p[32 * c + k + 1]), d);
            dk[k / 2] = pack_bf16x2(ds.x, ds.y);
          }
          tmem_st_16cols(tmem + lane_base + C::TM_DP + 64 * h + 16 * c, dk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B_P(h));
      }
      // The next item's Q and dO go into TMEM before this item's epilogue,
      // so that its first products overlap the epilogue.
      Item nxt;
      const bool have_next = ok && take_item(t + 1, nxt, ok);
      float nl_n = 0.f, nd_n = 0.f;
      if (have_next) {
        nl_n = nl2[row_of(nxt)];
        nd_n = ndl[row_of(nxt)];
        ok = copy_qdo(e + 1 + n_j);
      }
      // Epilogue: dQ staged as bf16 and stored by TMA.  The staging tile is
      // rewritten once the previous item's store has read it; the next
      // item's first dQ product overwrites the accumulator only after these
      // warps hand over its first dS, after the reads below.
      const bool okd = ok && __all_sync(0xffffffffu, mbar_wait(B_DONE, t & 1, status, abort_flag));
      if (threadIdx.x == 0) bulk_wait_group_read0();
      if (named_bar_any(kEpiBar, 32 * kComputeWarps, !okd)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(tmem + lane_base + C::TM_DQ + h * (D / 2) + 32 * c, r);
        tmem_ld_wait_regs(r);
        stage_row32(st_dq, row, h * (D / 2) + 32 * c, r, scale);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(kEpiBar, 32 * kComputeWarps);
      if (threadIdx.x == 0) {
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
          tma_store_3d(&tmdQ, kb * 64, cur.it * BT, cur.bh, st_dq + kb * kBoxBytes);
        bulk_commit_group();
      }
      e += 1 + n_j;
      g += n_j;
      cur = nxt;
      have = have_next;
      nl = nl_n;
      nd = nd_n;
    }
    // The last store must have read shared memory before the CTA exits.
    if (threadIdx.x == 0) bulk_wait_group_read0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // Every claim of this CTA is behind it: the last CTA to get here resets
  // the item counter (sched[0]) and this count (sched[1]) for the next launch.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(sched, 0u);
      atomicExch(sched + 1, 0u);
    }
  }
}

// ------------------------------------------------------------------ host
template <int D, bool CAUSAL>
static cudaError_t launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            const CUtensorMap &mdo, const CUtensorMap &mdq, const CUtensorMap &mdk,
                            const CUtensorMap &mdv, const float *nl2, const float *ndl, int B, int H, int H_kv, int N,
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
  // dK/dV: persistent, one CTA per SM (at most one per item).
  unsigned *sched = nullptr;
  e = sched_slot(&sched);
  if (e != cudaSuccess) return e;
  const long long kv_items = static_cast<long long>(B) * H_kv * n_blk;
  const long long kv_grid = kv_items < sm_count() ? kv_items : sm_count();
  // Both kernels are programmatic dependents of the launch before them on
  // the stream (row pass -> dK/dV -> dQ): set-up overlaps the previous
  // grid's tail, and each waits for its predecessor before using its rows.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(kv_grid));
  cfg.dynamicSmemBytes = CfgKV<D>::SMEM_ALLOC;
  e = cudaLaunchKernelEx(&cfg, kkv, mq, mk, mv, mdo, mdk, mdv, nl2, ndl, N, N_pad, H, H_kv,
                         B * H_kv, n_blk, scale_log2, scale, status, sched);
  if (e != cudaSuccess) return e;
  // dQ: persistent as well, one CTA per SM (at most one per item).
  unsigned *sched_q = nullptr;
  e = sched_slot(&sched_q);
  if (e != cudaSuccess) return e;
  const long long q_items = static_cast<long long>(B) * H * n_blk;
  cfg.gridDim = dim3(static_cast<unsigned>(q_items < sm_count() ? q_items : sm_count()));
  cfg.dynamicSmemBytes = CfgQ<D>::SMEM_ALLOC;
  return cudaLaunchKernelEx(&cfg, kq, mq, mk, mv, mdo, mdq, nl2, ndl, N, N_pad, H, H_kv, B * H,
                            n_blk, scale_log2, scale, status, sched_q);
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
  float *nl2 = static_cast<float *>(ws);    // -L log2(e) per padded row
  float *ndl = nl2 + rows;                  // -delta per padded row
  // Grid: one row of blocks per head, up to 1024 blocks of 2 * 256 / (d / 8)
  // rows each along a head (a block loops when the head is longer).
  const int rows_per_block = 2 * kPrepThreads / (d / 8);
  const dim3 prep_grid(static_cast<unsigned>(B * H),
                       static_cast<unsigned>(std::min(1024, (N_pad + rows_per_block - 1) / rows_per_block)));
  if (d == 128)
    attn_bwd_prep_kernel<128><<<prep_grid, kPrepThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(O), static_cast<const __nv_bfloat16 *>(dO), LSE, nl2,
        ndl, N, N_pad);
  else
    attn_bwd_prep_kernel<64><<<prep_grid, kPrepThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(O), static_cast<const __nv_bfloat16 *>(dO), LSE, nl2,
        ndl, N, N_pad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  if (!make_bhnd_map(&mq, Q, B * H, N, d, BT) || !make_bhnd_map(&mk, K, B * H_kv, N, d, BT) ||
      !make_bhnd_map(&mv, V, B * H_kv, N, d, BT) || !make_bhnd_map(&mdo, dO, B * H, N, d, BT) ||
      !make_bhnd_map(&mdq, dQ, B * H, N, d, BT) || !make_bhnd_map(&mdk, dK, B * H_kv, N, d, BT) ||
      !make_bhnd_map(&mdv, dV, B * H_kv, N, d, BT))
    return cudaErrorInvalidValue;
  if (d == 128)
    return causal ? launch_t<128, true>(mq, mk, mv, mdo, mdq, mdk, mdv, nl2, ndl, B, H, H_kv, N,
                                        N_pad, n_blk, scale, status, stream)
                  : launch_t<128, false>(mq, mk, mv, mdo, mdq, mdk, mdv, nl2, ndl, B, H, H_kv, N,
                                         N_pad, n_blk, scale, status, stream);
  return causal ? launch_t<64, true>(mq, mk, mv, mdo, mdq, mdk, mdv, nl2, ndl, B, H, H_kv, N, N_pad,
                                     n_blk, scale, status, stream)
                : launch_t<64, false>(mq, mk, mv, mdo, mdq, mdk, mdv, nl2, ndl, B, H, H_kv, N,
                                      N_pad, n_blk, scale, status, stream);
}

}  // namespace ea
