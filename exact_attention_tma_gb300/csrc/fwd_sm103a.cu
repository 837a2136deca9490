// fwd_sm103a.cu — fused exact-attention forward for GB300 (sm_103a).
//
// Computes O = softmax(scale * Q K^T + causal mask) V and the row log-sum-exp
// for every (batch, head), following "Why Fast GPUs Still Wait for Memory",
// sections "Attention from first principles" (the definition) and
// "FlashAttention is an IO algorithm": Q is split into blocks of B_r = 128
// rows, K/V into blocks of B_c = 128 keys that stream through shared memory,
// and a running maximum and normaliser per row rescale the output block as
// K/V blocks arrive, so S and P never reach HBM.  Causal masking follows the
// note "causal masking is not an optimisation here" on the same page: K/V
// blocks entirely above the diagonal are never loaded or multiplied.
//
// GB300 mapping: one CTA owns two 128-row query tiles of one head (256 rows)
// and streams that head's K/V tiles once for both.  16 warps:
//   warps 0-3   softmax for query tile 0   (thread = row = TMEM lane)
//   warps 4-7   softmax for query tile 1
//   warps 8-11  correction: rescales a tile's O accumulator in TMEM when its
//               running max moved by more than 2^8 (lazy rescaling: between
//               rescales the stale max is used for both P and the row sum, so
//               the final O / l is unchanged and P stays <= 256)
//   warp 12     MMA issuer (one thread): tcgen05.mma S_i = Q_i K_j^T into TMEM
//               (both operands from swizzled shared memory), then
//               O_i += P_i V_j with P_i read straight from TMEM (it overwrites
//               the first half of S_i as packed bf16)
//   warp 13     TMA producer: Q tiles once, K_j and V_j into separate rings
//               guarded by full/empty mbarriers
//   warps 14-15 idle
// The two softmax warpgroups work on different query tiles, so while one
// computes exponentials the tensor core runs the other tile's MMAs.
// Registers are re-balanced with setmaxnreg: 176 per softmax thread, 80 per
// correction thread and 80 for warps 12-15 (2*128*176 + 2*128*80 = 65536, the
// block's launch allocation of 512 threads x 128).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace ea {
namespace fwd {

constexpr int BM = 128;                  // query rows per tile (B_r)
constexpr int BN = 128;                  // keys per K/V tile (B_c)
constexpr int QT = 2;                    // query tiles per CTA
constexpr int kThreads = 512;
constexpr int kWarpMMA = 12;
constexpr int kWarpTMA = 13;
constexpr uint32_t kTmemCols = 512;      // S0 | S1 | O0 | O1
constexpr uint32_t kBoxBytes = 64 * 128 * 2;   // one TMA box: 64 columns x 128 rows bf16
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;      // log2 units: rescale when max grows > 2^8

// K/V ring depths per head dimension (shared memory: 2 query tiles + SK + SV
// tiles of 128 x d bf16 must fit in 227 KB).
#ifndef EA_FWD_SK128
#define EA_FWD_SK128 2
#endif
#ifndef EA_FWD_SV128
#define EA_FWD_SV128 2
#endif
#ifndef EA_FWD_SK64
#define EA_FWD_SK64 3
#endif
#ifndef EA_FWD_SV64
#define EA_FWD_SV64 3
#endif

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int KB = D / 64;                 // 128-byte swizzle column blocks
  static constexpr int SK = (D == 128) ? EA_FWD_SK128 : EA_FWD_SK64;   // K ring stages
  static constexpr int SV = (D == 128) ? EA_FWD_SV128 : EA_FWD_SV64;   // V ring stages
  static constexpr uint32_t Q_BYTES = BM * D * 2;   // one query tile
  static constexpr uint32_t KV_BYTES = BN * D * 2;  // one K or V tile
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + QT * Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + SK * KV_BYTES;
  static constexpr uint32_t OFF_ALPHA = OFF_V + SV * KV_BYTES;   // float[QT][BM]
  static constexpr uint32_t OFF_BAR = OFF_ALPHA + QT * BM * 4;
  // q, kf[SK], ke[SK], vf[SV], ve[SV], s[2], p[2], a[2], c[2], o[2], drain
  static constexpr int NBAR = 1 + 2 * SK + 2 * SV + 5 * QT + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;
  static constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;   // 1024-byte alignment slack
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  static constexpr uint32_t TMEM_S = 0;               // S_i at column 128 * i
  static constexpr uint32_t TMEM_O = QT * BN;         // O_i at column TMEM_O + D * i
  static_assert(TMEM_O + QT * D <= kTmemCols, "tensor memory budget");
};

// Pairs (out of every 8 pairs of a row) whose exp2 runs on the FMA pipe
// through exp2_poly2 instead of the MUFU ex2 unit, to balance the two pipes.
#ifndef EA_POLY_PAIRS_PER8
#define EA_POLY_PAIRS_PER8 0
#endif
constexpr int kPolyPairsPer8 = EA_POLY_PAIRS_PER8;

// 2^x for two lanes on the FMA pipe.  Cody-Waite range reduction: j = round(x)
// via the float32 "add 1.5 * 2^23" trick (j ends up in the low mantissa bits
// of t), f = x - j in [-1/2, 1/2]; 2^f from a degree-3 polynomial whose max
// relative error on [-1/2, 1/2] is 7.5e-5 (minimax fit by Lawson's algorithm,
// exact_attention_tma_gb300/exp2_poly.py); j is added to the exponent field.
// x is clamped at -126 so the exponent stays in range (masked -inf -> ~1e-38).
__device__ __forceinline__ float2 exp2_poly2(float2 x) {
  x.x = fmaxf(x.x, -126.f);
  x.y = fmaxf(x.y, -126.f);
  const float2 t = fadd2(x, make_float2(12582912.f, 12582912.f));
  const float2 j = fadd2(t, make_float2(-12582912.f, -12582912.f));
  const float2 f = ffma2(j, make_float2(-1.f, -1.f), x);
  float2 p = ffma2(make_float2(0.05517132207751274f, 0.05517132207751274f), f,
                   make_float2(0.24261054396629333f, 0.24261054396629333f));
  p = ffma2(p, f, make_float2(0.6932609677314758f, 0.6932609677314758f));
  p = ffma2(p, f, make_float2(0.9999281167984009f, 0.9999281167984009f));
  p.x = __uint_as_float(__float_as_uint(p.x) + (__float_as_uint(t.x) << 23));
  p.y = __uint_as_float(__float_as_uint(p.y) + (__float_as_uint(t.y) << 23));
  return p;
}

__device__ __forceinline__ void setmaxnreg_inc176() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 176;" ::: "memory");
}
__device__ __forceinline__ void setmaxnreg_dec80() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
}
__device__ __forceinline__ void setmaxnreg_dec80b() {  // warps 12-15
  asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, __nv_bfloat16 *__restrict__ O,
                    float *__restrict__ LSE, int N, int BH, int n_blk, float scale_log2,
                    unsigned *status) {
  using C = Cfg<D>;
  constexpr int SK = C::SK;
  constexpr int SV = C::SV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = warp >> 2;

  // Heads vary fastest; for causal the longest query blocks go first.
  const int bh = blockIdx.x % BH;
  const int blk = n_blk - 1 - static_cast<int>(blockIdx.x / BH);
  const int q0 = blk * (QT * BM);
  const int n_kv_total = (N + BN - 1) / BN;
  // K/V tiles each query tile needs (query tile 0 can stop one tile earlier when causal).
  const int n0 = CAUSAL ? min(QT * blk + 1, n_kv_total) : n_kv_total;
  const int n1 = CAUSAL ? min(QT * blk + 2, n_kv_total) : n_kv_total;

  const uint32_t bar0 = sb + C::OFF_BAR;
  const uint32_t B_Q = bar0;
  auto B_KF = [&](int s) { return bar0 + 8u * (1 + s); };
  auto B_KE = [&](int s) { return bar0 + 8u * (1 + SK + s); };
  auto B_VF = [&](int s) { return bar0 + 8u * (1 + 2 * SK + s); };
  auto B_VE = [&](int s) { return bar0 + 8u * (1 + 2 * SK + SV + s); };
  constexpr int kB5 = 1 + 2 * SK + 2 * SV;
  auto B_S = [&](int i) { return bar0 + 8u * (kB5 + i); };            // S_i ready (MMA)
  auto B_P = [&](int i) { return bar0 + 8u * (kB5 + QT + i); };       // P_i written (softmax)
  auto B_A = [&](int i) { return bar0 + 8u * (kB5 + 2 * QT + i); };   // alpha_i ready (softmax)
  auto B_C = [&](int i) { return bar0 + 8u * (kB5 + 3 * QT + i); };   // O_i corrected
  auto B_O = [&](int i) { return bar0 + 8u * (kB5 + 4 * QT + i); };   // P_i V_j done (MMA)
  const uint32_t B_DRAIN = bar0 + 8u * (kB5 + 5 * QT);
  float *alpha_s = reinterpret_cast<float *>(smem + C::OFF_ALPHA);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    mbar_init(B_Q, 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(B_KF(s), 1);
      mbar_init(B_KE(s), 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(B_VF(s), 1);
      mbar_init(B_VE(s), 1);
    }
    for (int i = 0; i < QT; ++i) {
      mbar_init(B_S(i), 1);
      mbar_init(B_P(i), BM);
      mbar_init(B_A(i), BM);
      mbar_init(B_C(i), BM);
      mbar_init(B_O(i), 1);
    }
    mbar_init(B_DRAIN, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTMA && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (wg < QT) {
    setmaxnreg_inc176();
    // ------------------------------------------------------------ softmax
    const int i = wg;                        // query tile
    const int r = threadIdx.x - i * BM;      // row within the tile == TMEM lane
    const int qrow = q0 + i * BM + r;
    const int n_i = (i == 0) ? n0 : n1;
    const int lim = CAUSAL ? min(qrow, N - 1) : N - 1;   // last visible key
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + C::TMEM_S + i * BN;
    float m = -INFINITY;                     // max used for the exponentials (base 2)
    float l = 0.f;                           // running sum of exp2(x - m)
    bool ok = true;
    for (int j = 0; j < n_i; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(B_S(i), j & 1, status, abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32cols(s_addr + c * 32, sr[c]);
      tmem_ld_wait();
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      const int kv0 = j * BN;
      if (kv0 + BN - 1 > lim) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (kv0 + c > lim) s[c] = -INFINITY;
      }
      // Row max: four independent chains of 3-input max.
      float mx[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        mx[q] = s[32 * q];
#pragma unroll
        for (int c = 1; c + 1 < 32; c += 2) mx[q] = fmax3(mx[q], s[32 * q + c], s[32 * q + c + 1]);
        mx[q] = fmaxf(mx[q], s[32 * q + 31]);
      }
      const float m_tile = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]) * scale_log2;
      float alpha = 1.f;
      if (m_tile - m > kRescaleThreshold) {   // true on the first tile (m = -inf)
        alpha = ex2_approx(m - m_tile);
        m = m_tile;
      }
      alpha_s[i * BM + r] = alpha;
      mbar_arrive(B_A(i));
      const float m_use = (m == -INFINITY) ? 0.f : m;
      const float2 sc2 = make_float2(scale_log2, scale_log2);
      const float2 nm2 = make_float2(-m_use, -m_use);
      float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t pk[BN / 2];
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), sc2, nm2);
        float2 p;
        if ((c & 7) < kPolyPairsPer8) {
          p = exp2_poly2(x);
        } else {
          p.x = ex2_approx(x.x);
          p.y = ex2_approx(x.y);
        }
        rs2[c & 1] = fadd2(rs2[c & 1], p);
        pk[c] = pack_bf16x2(p.x, p.y);
      }
      const float rs = (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
      l = l * alpha + rs;
      // P_i (bf16, keys packed in pairs) over the first 64 columns of S_i.
      tmem_st_32cols(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st_32cols(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(B_P(i));
    }
    // Epilogue: O_i / l -> bf16 rows, LSE.
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(B_O(i), (n_i - 1) & 1, status, abort_flag));
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      __nv_bfloat16 *orow = O + (static_cast<size_t>(bh) * N + qrow) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32cols(tmem + lane_addr + C::TMEM_O + i * D + c * 32, o);
        tmem_ld_wait();
        if (qrow < N) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[8 * v + 2 * e]) * inv_l,
                                 __uint_as_float(o[8 * v + 2 * e + 1]) * inv_l);
            st_global_v4(orow + c * 32 + v * 8, w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (qrow < N) {
        float lg;
        asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(l));
        LSE[static_cast<size_t>(bh) * N + qrow] = (m + lg) * kLn2;
      }
    }
    tc_fence_before();
  } else if (wg == QT) {
    setmaxnreg_dec80();
    // --------------------------------------------------------- correction
    const int t = threadIdx.x - QT * BM;     // row == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    for (int j = 0; ok && j < n1; ++j) {
#pragma unroll
      for (int i = 0; i < QT; ++i) {
        if (j >= (i == 0 ? n0 : n1)) continue;
        ok = __all_sync(0xffffffffu, mbar_wait(B_A(i), j & 1, status, abort_flag));
        if (!ok) break;
        const float a = alpha_s[i * BM + t];
        if (j > 0 && __any_sync(0xffffffffu, a != 1.f)) {
          // P_i V_{j-1} must have landed before O_i is scaled.
          ok = __all_sync(0xffffffffu, mbar_wait(B_O(i), (j - 1) & 1, status, abort_flag));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            const uint32_t o_addr = tmem + lane_addr + C::TMEM_O + i * D + c * 32;
            tmem_ld_32cols(o_addr, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
            tmem_st_32cols(o_addr, o);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(B_C(i));
      }
    }
    tc_fence_before();
  } else {
    setmaxnreg_dec80b();
    // Warps 12 and 13 run their schedules warp-uniformly (every lane waits on the
    // barriers) and one elected lane issues the TMA copies / MMAs, so addresses
    // and descriptors stay in the warp-uniform datapath.
    if (warp == kWarpTMA) {
      // ------------------------------------------------------ TMA producer
      const bool leader = elect_one();
      if (leader) {
        mbar_arrive_expect_tx(B_Q, QT * C::Q_BYTES);
#pragma unroll
        for (int i = 0; i < QT; ++i)
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(sb + C::OFF_Q + i * C::Q_BYTES + kb * kBoxBytes, &tmQ, kb * 64,
                        q0 + i * BM, bh, B_Q);
      }
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < n1; ++j) {
        const int sk = j % SK;
        if (!__all_sync(0xffffffffu, mbar_wait(B_KE(sk), ((j / SK) & 1) ^ 1u, status, abort_flag)))
          break;
        if (leader) {
          mbar_arrive_expect_tx(B_KF(sk), C::KV_BYTES);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(sb + C::OFF_K + sk * C::KV_BYTES + kb * kBoxBytes, &tmK, kb * 64, j * BN,
                        bh, B_KF(sk));
        }
        issued_k = j + 1;
        const int sv = j % SV;
        if (!__all_sync(0xffffffffu, mbar_wait(B_VE(sv), ((j / SV) & 1) ^ 1u, status, abort_flag)))
          break;
        if (leader) {
          mbar_arrive_expect_tx(B_VF(sv), C::KV_BYTES);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(sb + C::OFF_V + sv * C::KV_BYTES + kb * kBoxBytes, &tmV, kb * 64, j * BN,
                        bh, B_VF(sv));
        }
        issued_v = j + 1;
      }
      if (leader && *abort_flag) {
        // Let every copy this warp started land before the CTA exits.
        mbar_wait_drain(B_Q, 0, 100000000ull);
        for (int s = 0; s < SK && s < issued_k; ++s)
          mbar_wait_drain(B_KF(s), (((issued_k - 1 - s) / SK)) & 1, 100000000ull);
        for (int s = 0; s < SV && s < issued_v; ++s)
          mbar_wait_drain(B_VF(s), (((issued_v - 1 - s) / SV)) & 1, 100000000ull);
      }
      __syncwarp();
    } else if (warp == kWarpMMA) {
      // ------------------------------------------------------- MMA issuer
      const bool leader = elect_one();
      constexpr uint32_t kIdescQK = make_idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t kIdescPV = make_idesc_bf16(BM, D, 0, 1);
      // Base descriptors; a k-step or stage moves only the start-address field
      // (byte offset / 16 added to the low bits).
      const uint64_t dQ = make_sdesc_sw128(sb + C::OFF_Q, 16, 1024);
      const uint64_t dK = make_sdesc_sw128(sb + C::OFF_K, 16, 1024);
      const uint64_t dV = make_sdesc_sw128(sb + C::OFF_V, kBoxBytes, 1024);
      // S_i = Q_i K^T: both operands K-major (head dim contiguous), 128-B swizzle.
      auto issue_qk = [&](int i, int sk) {
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + C::TMEM_S + i * BN, dQ + ((i * C::Q_BYTES) >> 4) + koff,
                      dK + ((sk * C::KV_BYTES) >> 4) + koff, kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      // O_i += P_i V: P_i from TMEM (8 columns = 16 keys per step); V is MN-major
      // (head dim contiguous), 64-column blocks kBoxBytes apart, 8-key groups 1024 B apart.
      auto issue_pv = [&](int i, int sv, bool acc) {
#pragma unroll 1
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ts(tmem + C::TMEM_O + i * D, tmem + C::TMEM_S + i * BN + kk * 8,
                      dV + ((sv * C::KV_BYTES + kk * 16 * 128) >> 4), kIdescPV,
                      (acc || kk > 0) ? 1u : 0u);
      };
      auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort_flag));
      };
      bool ok = wait_all(B_Q, 0) && wait_all(B_KF(0), 0);
      if (ok) {
        tc_fence_after();
        if (leader) {
          issue_qk(0, 0);
          mma_commit(B_S(0));
          issue_qk(1, 0);
          mma_commit(B_S(1));
          if (SK < n1) mma_commit(B_KE(0));
        }
        __syncwarp();
      }
      for (int j = 0; ok && j < n1; ++j) {
        const int sv = j % SV;
        if (!(ok = wait_all(B_VF(sv), (j / SV) & 1))) break;
        if (j < n0) {
          if (!(ok = wait_all(B_P(0), j & 1) && wait_all(B_C(0), j & 1))) break;
          tc_fence_after();
          if (leader) {
            issue_pv(0, sv, j > 0);
            mma_commit(B_O(0));
          }
          __syncwarp();
        }
        const bool more = j + 1 < n1;
        const int sk1 = (j + 1) % SK;
        if (more) {
          if (!(ok = wait_all(B_KF(sk1), ((j + 1) / SK) & 1))) break;
          tc_fence_after();
          if (j + 1 < n0) {
            if (leader) {
              issue_qk(0, sk1);   // overwrites S_0/P_0 after the P_0 V_j MMA above has read it
              mma_commit(B_S(0));
            }
            __syncwarp();
          }
        }
        if (!(ok = wait_all(B_P(1), j & 1) && wait_all(B_C(1), j & 1))) break;
        tc_fence_after();
        if (leader) {
          issue_pv(1, sv, j > 0);
          mma_commit(B_O(1));
          if (j + SV < n1) mma_commit(B_VE(sv));
          if (more) {
            issue_qk(1, sk1);
            mma_commit(B_S(1));
            if (j + 1 + SK < n1) mma_commit(B_KE(sk1));
          }
        }
        __syncwarp();
      }
      // Every MMA issued so far must finish before TMEM is released.
      if (leader) {
        mma_commit(B_DRAIN);
        mbar_wait_drain(B_DRAIN, 0, 100000000ull);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// [B*H, N, d] bf16 viewed as a 3-D tensor; boxes of 64 columns x 128 rows x 1
// head with 128-byte swizzle.  Rows past N read as zeros.
static bool make_map(CUtensorMap *m, const void *base, int BH, int N, int d) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool CAUSAL>
static cudaError_t launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            void *O, float *LSE, int BH, int N, float scale_log2,
                            unsigned *status, cudaStream_t stream) {
  using C = Cfg<D>;
  auto kern = attn_fwd_kernel<D, CAUSAL>;
  static std::atomic<unsigned long long> configured{0};   // one bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::SMEM_ALLOC));
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  const int n_blk = (N + QT * BM - 1) / (QT * BM);
  const long long grid = static_cast<long long>(BH) * n_blk;
  kern<<<static_cast<unsigned>(grid), kThreads, C::SMEM_ALLOC, stream>>>(
      mq, mk, mv, static_cast<__nv_bfloat16 *>(O), LSE, N, BH, n_blk, scale_log2, status);
  return cudaGetLastError();
}

}  // namespace fwd

cudaError_t launch_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                       int H, int N, int d, float scale, int causal, unsigned *status,
                       cudaStream_t stream) {
  using namespace fwd;
  const int BH = B * H;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, Q, BH, N, d) || !make_map(&mk, K, BH, N, d) || !make_map(&mv, V, BH, N, d))
    return cudaErrorInvalidValue;
  const float scale_log2 = scale * 1.44269504088896340736f;
  if (d == 128)
    return causal ? launch_t<128, true>(mq, mk, mv, O, LSE, BH, N, scale_log2, status, stream)
                  : launch_t<128, false>(mq, mk, mv, O, LSE, BH, N, scale_log2, status, stream);
  return causal ? launch_t<64, true>(mq, mk, mv, O, LSE, BH, N, scale_log2, status, stream)
                : launch_t<64, false>(mq, mk, mv, O, LSE, BH, N, scale_log2, status, stream);
}

}  // namespace ea
