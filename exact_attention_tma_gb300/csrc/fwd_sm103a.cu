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
// GB300 mapping.  A CTA owns QT query tiles of 128 rows of one head and streams
// that head's K/V tiles once for all of them.  Tensor memory (512 columns)
// holds, per query tile, NS score buffers S (128 fp32 columns each), the O
// accumulator (d columns) and a separate P tile (64 columns of packed bf16).
// Because P does not overwrite S, the next S = Q K^T can be issued as soon as
// the softmax has *loaded* the current S into registers, so the tensor core
// never waits for a softmax to finish before starting the next score tile.
//   d = 64 : QT = 2 tiles, NS = 1  (2*128 + 2*64 + 2*64 = 512 columns)
//   d = 128: QT = 1 tile,  NS = 2  (2*128 + 128 + 64 = 448 columns)
// Warps:
//   warpgroup i < QT   softmax for query tile i (thread = row = TMEM lane)
//   warpgroup QT       (d = 64 only) correction: rescales O in TMEM when a row
//                      max grew by more than 2^8, then releases the P V MMA; with
//                      d = 128 the softmax warps do this themselves.  Lazy
//                      rescaling: between rescales the stale max is used for both
//                      P and the row sum, so O / l is unchanged and P stays <= 256
//   next warp          MMA issuer: S = Q K^T (operands in swizzled shared memory)
//                      and O += P V (P read from TMEM); one elected lane issues
//   next warp          TMA producer: Q tiles once, K and V into separate rings
//                      guarded by full/empty mbarriers
// With two softmax warpgroups, registers are re-balanced with setmaxnreg:
// 176 per softmax thread and 80 for the other warps (2*128*176 + 2*128*80 =
// 65536, the block's allocation of 512 threads x 128).
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
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBoxBytes = 64 * 128 * 2;   // one TMA box: 64 columns x 128 rows bf16
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;      // log2 units: rescale when max grows > 2^8

// K/V ring depths per head dimension (shared memory: QT query tiles + SK + SV
// tiles of 128 x d bf16 must fit in 227 KB).
#ifndef EA_FWD_SK128
#define EA_FWD_SK128 3
#endif
#ifndef EA_FWD_SV128
#define EA_FWD_SV128 3
#endif
#ifndef EA_FWD_SK64
#define EA_FWD_SK64 4
#endif
#ifndef EA_FWD_SV64
#define EA_FWD_SV64 4
#endif

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int QT = (D == 64) ? 2 : 1;      // query tiles per CTA
  static constexpr int NS = (D == 64) ? 1 : 2;      // S buffers per query tile
  static constexpr int NP = (D == 64) ? 1 : 2;      // P buffers per query tile
  // With one query tile the softmax warps also rescale O themselves; with two
  // a separate correction warpgroup does it.
  static constexpr bool SELF_CORRECT = (QT == 1);
  static constexpr int THREADS = SELF_CORRECT ? 192 : 512;
  static constexpr int WARP_MMA = SELF_CORRECT ? 4 : 4 * (QT + 1);
  static constexpr int WARP_TMA = WARP_MMA + 1;
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
  // q, kf[SK], ke[SK], vf[SV], ve[SV], s[QT*NS], sf[QT*NS], (spare)/a/c/o/ae[QT],
  // pf[QT*NP], p[QT*NP], drain
  static constexpr int NBAR = 1 + 2 * SK + 2 * SV + 2 * QT * NS + 5 * QT + 2 * QT * NP + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;
  static constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;   // 1024-byte alignment slack
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  // Tensor-memory columns.
  static constexpr uint32_t TMEM_O0 = QT * NS * BN;
  static constexpr uint32_t TMEM_P0 = TMEM_O0 + QT * D;
  static_assert(TMEM_P0 + QT * NP * (BN / 2) <= kTmemCols, "tensor memory budget");
  __host__ __device__ static constexpr uint32_t tmem_s(int i, int b) { return (i * NS + b) * BN; }
  __host__ __device__ static constexpr uint32_t tmem_o(int i) { return TMEM_O0 + i * D; }
  __host__ __device__ static constexpr uint32_t tmem_p(int i, int pb) {
    return TMEM_P0 + (i * NP + pb) * (BN / 2);
  }
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

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, __nv_bfloat16 *__restrict__ O,
                    float *__restrict__ LSE, int N, int BH, int n_blk, float scale_log2,
                    unsigned *status) {
  using C = Cfg<D>;
  constexpr int QT = C::QT;
  constexpr int NS = C::NS;
  constexpr int NP = C::NP;
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
  // K/V tiles query tile i needs; the last tile needs every tile the CTA loads.
  auto n_of = [&](int i) { return CAUSAL ? min(QT * blk + i + 1, n_kv_total) : n_kv_total; };
  const int n_last = n_of(QT - 1);

  const uint32_t bar0 = sb + C::OFF_BAR;
  const uint32_t B_Q = bar0;
  auto B_KF = [&](int s) { return bar0 + 8u * (1 + s); };
  auto B_KE = [&](int s) { return bar0 + 8u * (1 + SK + s); };
  auto B_VF = [&](int s) { return bar0 + 8u * (1 + 2 * SK + s); };
  auto B_VE = [&](int s) { return bar0 + 8u * (1 + 2 * SK + SV + s); };
  constexpr int kB5 = 1 + 2 * SK + 2 * SV;
  constexpr int kB6 = kB5 + 2 * QT * NS;
  auto B_S = [&](int i, int b) { return bar0 + 8u * (kB5 + i * NS + b); };            // S ready
  auto B_SF = [&](int i, int b) { return bar0 + 8u * (kB5 + QT * NS + i * NS + b); }; // S loaded
  auto B_P = [&](int i, int pb) {                                        // P buffer written
    return bar0 + 8u * (kB6 + 5 * QT + QT * NP + i * NP + pb);
  };
  auto B_A = [&](int i) { return bar0 + 8u * (kB6 + QT + i); };       // alpha_i ready (softmax)
  auto B_C = [&](int i) { return bar0 + 8u * (kB6 + 2 * QT + i); };   // O_i corrected
  auto B_O = [&](int i) { return bar0 + 8u * (kB6 + 3 * QT + i); };   // P_i V_j done (MMA)
  auto B_AE = [&](int i) { return bar0 + 8u * (kB6 + 4 * QT + i); };  // alpha_i consumed
  auto B_PF = [&](int i, int pb) { return bar0 + 8u * (kB6 + 5 * QT + i * NP + pb); };  // P buf read
  const uint32_t B_DRAIN = bar0 + 8u * (kB6 + 5 * QT + 2 * QT * NP);
  static_assert(kB6 + 5 * QT + 2 * QT * NP == C::NBAR - 1, "barrier layout");
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
      for (int b = 0; b < NS; ++b) {
        mbar_init(B_S(i, b), 1);
        mbar_init(B_SF(i, b), BM);
      }
      mbar_init(B_A(i), BM);
      mbar_init(B_C(i), BM);
      mbar_init(B_O(i), 1);
      mbar_init(B_AE(i), BM);
      for (int pb = 0; pb < NP; ++pb) {
        mbar_init(B_P(i, pb), BM);
        mbar_init(B_PF(i, pb), 1);
      }
    }
    mbar_init(B_DRAIN, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == C::WARP_TMA && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (wg < QT) {
    if constexpr (QT == 2) setmaxnreg_inc176();
    // ------------------------------------------------------------ softmax
    const int i = wg;                        // query tile
    const int r = threadIdx.x - i * BM;      // row within the tile == TMEM lane
    const int qrow = q0 + i * BM + r;
    const int n_i = n_of(i);
    const int lim = CAUSAL ? min(qrow, N - 1) : N - 1;   // last visible key
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;

    float m = -INFINITY;                     // max used for the exponentials (base 2)
    float l = 0.f;                           // running sum of exp2(x - m)
    bool ok = true;
    for (int j = 0; j < n_i; ++j) {
      const int b = j % NS;
      ok = __all_sync(0xffffffffu, mbar_wait(B_S(i, b), (j / NS) & 1, status, abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
      const uint32_t s_addr = tmem + lane_addr + C::tmem_s(i, b);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32cols(s_addr + c * 32, sr[c]);
      tmem_ld_wait();
      // S is in registers: the MMA warp may overwrite this buffer now.
      tc_fence_before();
      mbar_arrive(B_SF(i, b));
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
      if constexpr (C::SELF_CORRECT) {
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // P V_{j-1} (and, by commit order, every earlier MMA) must have landed
          // before this warp's O rows are scaled.  Waited on its P buffer's
          // barrier, which is never more than one phase away (B_O may be two).
          ok = __all_sync(0xffffffffu, mbar_wait(B_PF(i, (j - 1) % NP), ((j - 1) / NP) & 1,
                                                 status, abort_flag));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            const uint32_t o_addr = tmem + lane_addr + C::tmem_o(i) + c * 32;
            tmem_ld_32cols(o_addr, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_32cols(o_addr, o);
          }
          tmem_st_wait();
        }
      } else {
        // The correction warps must have read alpha_{j-1} before it is replaced
        // (this also keeps B_A at most one phase ahead of its reader).
        if (j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(B_AE(i), (j - 1) & 1, status, abort_flag));
          if (!ok) break;
        }
        alpha_s[i * BM + r] = alpha;
        mbar_arrive(B_A(i));
      }
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
      // P buffer j % NP: the P V MMA of its previous use must have read it.
      const int pb = j % NP;
      if (j >= NP) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(B_PF(i, pb), ((j / NP) - 1) & 1, status, abort_flag));
        if (!ok) break;
        tc_fence_after();
      }
      const uint32_t p_addr = tmem + lane_addr + C::tmem_p(i, pb);
      tmem_st_32cols(p_addr, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st_32cols(p_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(B_P(i, pb));
    }
    // Epilogue: O_i / l -> bf16 rows, LSE, once the last P V MMA (and so every
    // earlier one) has completed.
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(B_PF(i, (n_i - 1) % NP), ((n_i - 1) / NP) & 1,
                                             status, abort_flag));
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      __nv_bfloat16 *orow = O + (static_cast<size_t>(bh) * N + qrow) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32cols(tmem + lane_addr + C::tmem_o(i) + c * 32, o);
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
  } else if (!C::SELF_CORRECT && wg == QT) {
    if constexpr (QT == 2) setmaxnreg_dec80();
    // --------------------------------------------------------- correction
    const int t = threadIdx.x - QT * BM;     // row == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    for (int j = 0; ok && j < n_last; ++j) {
#pragma unroll
      for (int i = 0; i < QT; ++i) {
        if (j >= n_of(i)) continue;
        ok = __all_sync(0xffffffffu, mbar_wait(B_A(i), j & 1, status, abort_flag));
        if (!ok) break;
        const float a = alpha_s[i * BM + t];
        mbar_arrive(B_AE(i));
        // P_i V_{j-1} must have landed before O_i is scaled, and before P_i V_j is
        // released (so B_C never runs two phases ahead of the MMA warp).
        if (j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(B_O(i), (j - 1) & 1, status, abort_flag));
          if (!ok) break;
        }
        if (j > 0 && __any_sync(0xffffffffu, a != 1.f)) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            const uint32_t o_addr = tmem + lane_addr + C::tmem_o(i) + c * 32;
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
    if constexpr (QT == 2) setmaxnreg_dec80();
    // The MMA and TMA warps run their schedules warp-uniformly (every lane waits
    // on the barriers) and one elected lane issues, so addresses and
    // descriptors stay in the warp-uniform datapath.
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort_flag));
    };
    if (warp == C::WARP_TMA) {
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
      for (int j = 0; j < n_last; ++j) {
        const int sk = j % SK;
        if (!wait_all(B_KE(sk), ((j / SK) & 1) ^ 1u)) break;
        if (leader) {
          mbar_arrive_expect_tx(B_KF(sk), C::KV_BYTES);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(sb + C::OFF_K + sk * C::KV_BYTES + kb * kBoxBytes, &tmK, kb * 64, j * BN,
                        bh, B_KF(sk));
        }
        issued_k = j + 1;
        const int sv = j % SV;
        if (!wait_all(B_VE(sv), ((j / SV) & 1) ^ 1u)) break;
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
    } else if (warp == C::WARP_MMA) {
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
      auto issue_qk = [&](int i, int b, int sk) {
#pragma unroll(QT == 1 ? D / 16 : 1)
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + C::tmem_s(i, b), dQ + ((i * C::Q_BYTES) >> 4) + koff,
                      dK + ((sk * C::KV_BYTES) >> 4) + koff, kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      // O_i += P_i V: P_i from TMEM (8 columns = 16 keys per step); V is MN-major
      // (head dim contiguous), 64-column blocks kBoxBytes apart, 8-key groups 1024 B apart.
      auto issue_pv = [&](int i, int pb, int sv, bool acc) {
#pragma unroll(QT == 1 ? BN / 16 : 1)
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ts(tmem + C::tmem_o(i), tmem + C::tmem_p(i, pb) + kk * 8,
                      dV + ((sv * C::KV_BYTES + kk * 16 * 128) >> 4), kIdescPV,
                      (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = wait_all(B_Q, 0);
      // Prologue: the first NS score tiles of every query tile.
      for (int jj = 0; ok && jj < NS && jj < n_last; ++jj) {
        if (!(ok = wait_all(B_KF(jj % SK), (jj / SK) & 1))) break;
        tc_fence_after();
        if (leader) {
          for (int i = 0; i < QT; ++i)
            if (jj < n_of(i)) {
              issue_qk(i, jj % NS, jj % SK);
              mma_commit(B_S(i, jj % NS));
            }
          if (jj + SK < n_last) mma_commit(B_KE(jj % SK));
        }
        __syncwarp();
      }
      // Non-blocking test of every barrier step j needs (leader lane only).  A
      // wait on a completed phase still costs a shared-memory round trip
      // (~140 clk) and the tensor pipe queues only about one MMA, so the step's
      // tests are issued together (their latencies overlap) and, when all pass,
      // the step's MMAs go out back to back.
      auto test_step = [&](int j) -> uint32_t {
        if (j >= n_last) return 1u;
        const int jn = j + NS;
        uint32_t r = mbar_test(B_VF(j % SV), (j / SV) & 1);
        if (jn < n_last) {
          r &= mbar_test(B_KF(jn % SK), (jn / SK) & 1);
#pragma unroll
          for (int i = 0; i < QT; ++i)
            if (jn < n_of(i)) r &= mbar_test(B_SF(i, j % NS), (j / NS) & 1);
        }
#pragma unroll
        for (int i = 0; i < QT; ++i)
          if (j < n_of(i)) {
            r &= mbar_test(B_P(i, j % NP), (j / NP) & 1);
            if constexpr (!C::SELF_CORRECT) r &= mbar_test(B_C(i), j & 1);
          }
        return r;
      };
      for (int j = 0; ok && j < n_last; ++j) {
        const int jn = j + NS;      // score tile j + NS reuses the buffer softmax j just loaded
        const bool more = jn < n_last;
        const int sv = j % SV;
        const uint32_t r_now = leader ? test_step(j) : 0u;
        const bool ready = __ballot_sync(0xffffffffu, leader && r_now != 0) != 0;
        if (ready) {
          // Everything step j needs is in place: issue it in one go.
          tc_fence_after();
          if (leader) {
            if (more) {
              for (int i = 0; i < QT; ++i)
                if (jn < n_of(i)) {
                  issue_qk(i, jn % NS, jn % SK);
                  mma_commit(B_S(i, jn % NS));
                }
              if (jn + SK < n_last) mma_commit(B_KE(jn % SK));
            }
            for (int i = 0; i < QT; ++i)
              if (j < n_of(i)) {
                issue_pv(i, j % NP, sv, j > 0);
                mma_commit(B_O(i));
                mma_commit(B_PF(i, j % NP));
              }
            if (j + SV < n_last) mma_commit(B_VE(sv));
          }
          __syncwarp();
          continue;
        }
        // Slow path: bounded blocking waits, one barrier at a time.
        if (more) {
          if (!(ok = wait_all(B_KF(jn % SK), (jn / SK) & 1))) break;
          for (int i = 0; ok && i < QT; ++i) {
            if (jn >= n_of(i)) continue;
            if (!(ok = wait_all(B_SF(i, j % NS), (j / NS) & 1))) break;
            tc_fence_after();
            if (leader) {
              issue_qk(i, jn % NS, jn % SK);
              mma_commit(B_S(i, jn % NS));
            }
            __syncwarp();
          }
          if (!ok) break;
          if (leader && jn + SK < n_last) mma_commit(B_KE(jn % SK));
          __syncwarp();
        }
        // O_i += P_i V_j once P_i is written and O_i corrected.
        if (!(ok = wait_all(B_VF(sv), (j / SV) & 1))) break;
        for (int i = 0; ok && i < QT; ++i) {
          if (j >= n_of(i)) continue;
          if (!(ok = wait_all(B_P(i, j % NP), (j / NP) & 1) &&
                     (C::SELF_CORRECT || wait_all(B_C(i), j & 1))))
            break;
          tc_fence_after();
          if (leader) {
            issue_pv(i, j % NP, sv, j > 0);
            mma_commit(B_O(i));
            mma_commit(B_PF(i, j % NP));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (leader && j + SV < n_last) mma_commit(B_VE(sv));
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
  if (warp == C::WARP_MMA) {
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
  const int n_blk = (N + C::QT * BM - 1) / (C::QT * BM);
  const long long grid = static_cast<long long>(BH) * n_blk;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_ALLOC, stream>>>(
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
