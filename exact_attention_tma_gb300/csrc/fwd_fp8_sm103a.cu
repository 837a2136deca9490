// fwd_fp8_sm103a.cu — attention forward with FP8 (E4M3) operands on tcgen05.
//
// "Why Fast GPUs Still Wait for Memory" puts the FP8 tensor ceiling at twice
// the bf16 one (its roofline table and the compute-ceiling discussion):
// the same tiled forward with 8-bit Q, K, V and P doubles the rate of both
// products.  Inputs are E4M3 with one descale factor per tensor (the real
// values are code * descale); the scores and the softmax stay in fp32, P is
// rounded to E4M3 for the P V product, O leaves in bf16 and the LSE in fp32.
//
// Layout and launches:
//   1. a transpose pass writes V^T ([B*H, d, N_pad] bytes) into a workspace,
//      so that both products read K-major operands (V^T rows are the head
//      dimension, keys contiguous);
//   2. one CTA per (head, 128-query tile): Q in shared memory, K and V^T
//      tiles (128 keys) through TMA rings, S in TMEM (double buffered, so
//      Q K_{j+1}^T runs while the softmax works on S_j), P written as E4M3
//      over the first columns of its own S region, O += P V_j with A = P
//      from TMEM and B = the V^T tile (K-major).
// The softmax is split over key halves exactly like the bf16 kernel at
// d = 64: warps q and q + 4 own rows 32q..32q+31, warp q keys 0-63 and warp
// q + 4 keys 64-127 of every tile, each half with its own running maximum,
// sum and TMEM accumulator, merged once in the epilogue.  The maximum is
// updated lazily: a tile is redone against a new maximum only when the
// half's P sum exceeds kRescaleSum (so every P <= 64), and P is scaled by 2^2
// before the E4M3 rounding (P * 4 <= 256 < 448, and P >= 2^-8 stays a normal
// E4M3 number); the epilogue divides the 2^2 back out.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace ea {
namespace f8 {

constexpr int BM = 128;                    // queries per CTA
constexpr int BN = 128;                    // keys per tile
constexpr int D = 128;                     // head dimension (bytes per row)
constexpr int kThreads = 352;              // warps 0-7 softmax, 8 MMA, 9 TMA (Q, K), 10 TMA (V^T)
constexpr int kWarpMMA = 8;
constexpr int kWarpTMA = 9;
constexpr int kWarpTMAV = 10;
constexpr int SK = 4, SV = 4;              // K and V^T ring depths
constexpr uint32_t TILE = 128 * 128;       // one 128 x 128-byte tile
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + TILE;
constexpr uint32_t OFF_V = OFF_K + SK * TILE;
constexpr uint32_t OFF_XCH = OFF_V + SV * TILE;          // float m[2][BM], l[2][BM]
constexpr uint32_t OFF_BAR = OFF_XCH + 4 * BM * 4;
// q, kf[SK], ke[SK], vf[SV], ve[SV], s[2], p[2][2], pf[2], o, drain
constexpr int NBAR = 1 + 2 * SK + 2 * SV + 2 + 4 + 2 + 2;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
constexpr uint32_t kTmemCols = 512;        // S0 | S1 | O_0 | O_1
constexpr uint32_t TM_S = 0;
constexpr uint32_t TM_O = 2 * BN;
constexpr float kRescaleSum = 64.0f;       // half-row P sum that forces a redo
constexpr float kPScale = 4.0f;            // P is rounded to E4M3 as P * 2^2
constexpr float kLog2PScale = 2.0f;
constexpr float kMInit = -1.0e30f;
constexpr float kLn2 = 0.69314718055994530942f;

// ------------------------------------------------------------ V transpose
// V [BH, N, 128] bytes -> V^T [BH, 128, N_pad] bytes, 128 x 128 blocks
// through shared memory (row stride 132 so column reads spread over banks).
__global__ void __launch_bounds__(256)
    attn_fp8_vt_kernel(const uint8_t *__restrict__ V, uint8_t *__restrict__ VT, int N, int N_pad) {
  __shared__ uint8_t tile[128 * 132];
  const size_t bh = blockIdx.y;
  const int k0 = blockIdx.x * 128;
  const uint8_t *src = V + (bh * N + k0) * D;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int idx = threadIdx.x + u * 256;           // 1024 chunks of 16 bytes
    const int row = idx >> 3, c = idx & 7;
    uint4 x = make_uint4(0, 0, 0, 0);
    if (k0 + row < N) x = *reinterpret_cast<const uint4 *>(src + row * D + c * 16);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      *reinterpret_cast<uint32_t *>(&tile[row * 132 + c * 16 + 4 * e]) = w[e];
  }
  __syncthreads();
  uint8_t *dst = VT + bh * D * static_cast<size_t>(N_pad) + k0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int idx = threadIdx.x + u * 256;           // 1024 chunks of 16 keys
    const int d = idx >> 3, c = idx & 7;
    if (k0 + c * 16 >= N_pad) continue;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = c * 16 + 4 * e;
      w[e] = static_cast<uint32_t>(tile[k * 132 + d]) |
             (static_cast<uint32_t>(tile[(k + 1) * 132 + d]) << 8) |
             (static_cast<uint32_t>(tile[(k + 2) * 132 + d]) << 16) |
             (static_cast<uint32_t>(tile[(k + 3) * 132 + d]) << 24);
    }
    *reinterpret_cast<uint4 *>(dst + static_cast<size_t>(d) * N_pad + c * 16) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ------------------------------------------------------------ forward
template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmVT, __nv_bfloat16 *__restrict__ O,
                        float *__restrict__ LSE, int N, int BH, int n_blk, float scale_log2,
                        float out_mul, unsigned *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Causal: heads fastest, longest query tiles first; otherwise query tiles
  // fastest (CTAs running together share their head's K/V through L2).
  const int bh = CAUSAL ? static_cast<int>(blockIdx.x % BH) : static_cast<int>(blockIdx.x / n_blk);
  const int qt = CAUSAL ? n_blk - 1 - static_cast<int>(blockIdx.x / BH)
                        : static_cast<int>(blockIdx.x % n_blk);
  const int n = CAUSAL ? qt + 1 : n_blk;    // K/V tiles this query tile needs

  const uint32_t bar0 = sb + OFF_BAR;
  const uint32_t B_Q = bar0;
  auto B_KF = [&](int s) { return bar0 + 8u * (1 + s); };
  auto B_KE = [&](int s) { return bar0 + 8u * (1 + SK + s); };
  auto B_VF = [&](int s) { return bar0 + 8u * (1 + 2 * SK + s); };
  auto B_VE = [&](int s) { return bar0 + 8u * (1 + 2 * SK + SV + s); };
  constexpr int kB1 = 1 + 2 * SK + 2 * SV;
  auto B_S = [&](int b) { return bar0 + 8u * (kB1 + b); };               // S_b written
  auto B_P = [&](int b, int h) { return bar0 + 8u * (kB1 + 2 + 2 * b + h); };   // P_b half h
  auto B_PF = [&](int b) { return bar0 + 8u * (kB1 + 6 + b); };          // P V of P_b done
  const uint32_t B_O = bar0 + 8u * (kB1 + 8);
  const uint32_t B_DRAIN = bar0 + 8u * (kB1 + 9);
  static_assert(kB1 + 10 == NBAR, "barrier count");
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

  if (threadIdx.x == kWarpTMA * 32) {
    mbar_init(B_Q, 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(B_KF(s), 1);
      mbar_init(B_KE(s), 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(B_VF(s), 1);
      mbar_init(B_VE(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(B_S(b), 1);
      mbar_init(B_P(b, 0), 4);
      mbar_init(B_P(b, 1), 4);
      mbar_init(B_PF(b), 1);
    }
    mbar_init(B_O, 1);
    mbar_init(B_DRAIN, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVT);
    mbar_arrive_expect_tx(B_Q, TILE);
    tma_load_3d(sb + OFF_Q, &tmQ, 0, qt * BM, bh, B_Q);
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTMA || warp == kWarpTMAV) {
    // ------------------------------------------------ TMA (K / V^T rings)
    // One warp per ring, so that a K load never queues behind a V^T stage
    // that the (later) P V has not released yet.
    const bool is_k = (warp == kWarpTMA);
    const int S = is_k ? SK : SV;
    const uint32_t base = sb + (is_k ? OFF_K : OFF_V);
    const bool leader = elect_one();
    int issued = 0;
    for (int j = 0; j < n; ++j) {
      const int s = j % S;
      const uint32_t empty = is_k ? B_KE(s) : B_VE(s);
      const uint32_t full = is_k ? B_KF(s) : B_VF(s);
      if (!__all_sync(0xffffffffu, mbar_wait(empty, ((j / S) & 1) ^ 1u, status, abort_flag)))
        break;
      if (leader) {
        mbar_arrive_expect_tx(full, TILE);
        if (is_k)
          tma_load_3d(base + s * TILE, &tmK, 0, j * BN, bh, full);
        else
          tma_load_3d(base + s * TILE, &tmVT, j * BN, 0, bh, full);
      }
      issued = j + 1;
    }
    if (leader && *abort_flag) {
      if (is_k) mbar_wait_drain(B_Q, 0, 100000000ull);
      for (int u = 0; u < S && u < issued; ++u) {
        const int jj = issued - 1 - u;
        mbar_wait_drain(is_k ? B_KF(jj % S) : B_VF(jj % S), (jj / S) & 1, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------------ MMA
    const bool leader = elect_one();
    constexpr uint32_t kIdesc = make_idesc_e4m3(BM, BN, 0, 0);   // BN == D
    const uint64_t dq = make_sdesc_sw128(sb + OFF_Q, 16, 1024);
    const uint32_t hi = static_cast<uint32_t>(dq >> 32);
    const uint32_t q_lo = static_cast<uint32_t>(dq);
    const uint32_t k_lo = static_cast<uint32_t>(make_sdesc_sw128(sb + OFF_K, 16, 1024));
    const uint32_t v_lo = static_cast<uint32_t>(make_sdesc_sw128(sb + OFF_V, 16, 1024));
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort_flag));
    };
    // S_b = Q K_j^T: four 32-byte k-steps across the 128-byte rows.
    auto issue_qk = [&](int b, int sk) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f8_ss_lo(tmem + TM_S + b * BN, q_lo + ((kk * 32) >> 4),
                     k_lo + ((sk * TILE + kk * 32) >> 4), hi, kIdesc, kk > 0 ? 1u : 0u);
    };
    // O_h += P_b[:, keys of half h] V_j[keys of half h, :]: two 32-key steps,
    // A = P from TMEM (8 columns per step, keys 64h.. in columns 64h.. of
    // S_b), B = the V^T tile at the same keys.
    auto issue_pv = [&](int b, int sv, int h, bool acc) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int kk = 2 * h + u;
        mma_f8_ts_lo(tmem + TM_O + h * D, tmem + TM_S + b * BN + 64 * h + 8 * u,
                     v_lo + ((sv * TILE + kk * 32) >> 4), hi, kIdesc, (acc || u > 0) ? 1u : 0u);
      }
    };
    bool ok = wait_all(B_Q, 0);
    for (int j = 0; ok && j < 2 && j < n; ++j) {
      if (!(ok = wait_all(B_KF(j % SK), (j / SK) & 1))) break;
      tc_fence_after();
      if (leader) {
        issue_qk(j, j % SK);
        mma_commit(B_S(j));
        if (j + SK < n) mma_commit(B_KE(j % SK));
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < n; ++j) {
      const int b = j & 1, sv = j % SV;
      if (!(ok = wait_all(B_VF(sv), (j / SV) & 1))) break;
      for (int h = 0; h < 2; ++h) {
        if (!(ok = wait_all(B_P(b, h), (j >> 1) & 1))) break;
        tc_fence_after();
        if (leader) issue_pv(b, sv, h, j > 0);
        __syncwarp();
      }
      if (!ok) break;
      if (leader) {
        mma_commit(B_PF(b));
        if (j + SV < n) mma_commit(B_VE(sv));
        if (j + 1 == n) mma_commit(B_O);
      }
      __syncwarp();
      if (j + 2 < n) {
        // S_b (and P_b over it) is free once P_b V_j above has run (MMAs from
        // one thread execute in issue order).
        const int sk = (j + 2) % SK;
        if (!(ok = wait_all(B_KF(sk), ((j + 2) / SK) & 1))) break;
        tc_fence_after();
        if (leader) {
          issue_qk(b, sk);
          mma_commit(B_S(b));
          if (j + 2 + SK < n) mma_commit(B_KE(sk));
        }
        __syncwarp();
      }
    }
    if (leader) {
      mma_commit(B_DRAIN);
      mbar_wait_drain(B_DRAIN, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- softmax
    const int q = warp & 3;
    const int h = warp >> 2;                 // key half
    const int r = 32 * q + lane;             // query row of the tile == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    const int qrow = qt * BM + r;
    const int lim = CAUSAL ? min(qrow, N - 1) : N - 1;   // last visible key
    float m = kMInit, l = 0.f;
    bool ok = true;
    // Scores of keys k0 .. k0 + 31 past the last visible key become -inf.
    auto mask32 = [&](const uint32_t (&a)[32], int k0, float *x) {
#pragma unroll
      for (int e = 0; e < 32; ++e) x[e] = (k0 + e <= lim) ? __uint_as_float(a[e]) : -INFINITY;
    };
    // kPScale * P of 32 scores, 2^(x scale_log2 - m + log2 kPScale), as E4M3
    // packed 4 per word; returns their sum (still times kPScale).  Two scores
    // per packed FMA and add.
    const float2 sc2 = make_float2(scale_log2, scale_log2);
    auto exp32 = [&](const float *x, uint32_t *pk) {
      const float nm = kLog2PScale - m;
      const float2 nm2 = make_float2(nm, nm);
      float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float2 t0 = ffma2(make_float2(x[e], x[e + 1]), sc2, nm2);
        const float2 t1 = ffma2(make_float2(x[e + 2], x[e + 3]), sc2, nm2);
        const float2 p0 = make_float2(ex2_approx(t0.x), ex2_approx(t0.y));
        const float2 p1 = make_float2(ex2_approx(t1.x), ex2_approx(t1.y));
        acc[0] = fadd2(acc[0], p0);
        acc[1] = fadd2(acc[1], p1);
        pk[e / 4] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
      }
      return (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
    };
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(B_S(b), (j >> 1) & 1, status, abort_flag))))
        break;
      tc_fence_after();
      const int k0 = j * BN + 64 * h;
      const uint32_t s_addr = tmem + lane_addr + TM_S + b * BN + 64 * h;
      float x[64];
      uint32_t pk[16];
      float rs;
      {
        uint32_t a[32], c[32];
        tmem_ld_32cols(s_addr, a);
        tmem_ld_wait_regs(a);
        tmem_ld_32cols(s_addr + 32, c);
        mask32(a, k0, x);
        if (j == 0) {
          // First tile: the maximum of the half first.
          tmem_ld_wait_regs(c);
          mask32(c, k0 + 32, x + 32);
          float mx = -INFINITY;
#pragma unroll
          for (int e = 0; e < 64; ++e) mx = fmaxf(mx, x[e]);
          m = (mx == -INFINITY) ? kMInit : mx * scale_log2;
          rs = exp32(x, pk) + exp32(x + 32, pk + 8);
        } else {
          // Keys 32-63 are read from TMEM while keys 0-31 are exponentiated.
          rs = exp32(x, pk);
          tmem_ld_wait_regs(c);
          mask32(c, k0 + 32, x + 32);
          rs += exp32(x + 32, pk + 8);
        }
      }
      if (__any_sync(0xffffffffu, !(rs <= kRescaleSum * kPScale))) {
        // Redo the tile against the new maximum and scale O_h (and l) by
        // 2^(m_old - m_new).  O_h is written by the P V of tile j - 1: wait
        // for it first.
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < 64; ++e) mx = fmaxf(mx, x[e]);
        const float m_new = fmaxf(m, mx * scale_log2);
        const float alpha = ex2_approx(m - m_new);
        m = m_new;
        rs = exp32(x, pk) + exp32(x + 32, pk + 8);
        l *= alpha;
        if (j > 0) {
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(B_PF((j - 1) & 1), ((j - 1) >> 1) & 1,
                                                        status, abort_flag))))
            break;
          tc_fence_after();
          const uint32_t o_addr = tmem + lane_addr + TM_O + h * D;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32cols(o_addr + 32 * c, o);
            tmem_ld_wait_regs(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_32cols(o_addr + 32 * c, o);
          }
        }
      }
      l += rs * (1.0f / kPScale);
      // P (64 keys = 16 columns of E4M3 quadruples) over the first columns of
      // this half's S region, which this thread has read.
      tmem_st_16cols(s_addr, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B_P(b, h));
    }
    // Epilogue: merge the halves, O = (w_0 O_0 + w_1 O_1) / (w_0 l_0 + w_1 l_1)
    // with w_h = 2^(m_h - max m); each warp writes its half of the columns.
    float *xm = reinterpret_cast<float *>(smem + OFF_XCH);
    float *xl = xm + 2 * BM;
    xm[h * BM + r] = m;
    xl[h * BM + r] = l;
    named_bar_sync(1, 256);
    // All eight warps take part in the vote (a warp whose wait gave up votes
    // to stop), so they leave together.
    const bool w_ok = ok && mbar_wait(B_O, 0, status, abort_flag);
    const bool okw = !named_bar_any(2, 256, !__all_sync(0xffffffffu, w_ok));
    if (okw) {
      tc_fence_after();
      const float m0 = xm[r], m1 = xm[BM + r];
      const float M = fmaxf(m0, m1);
      const float w0 = ex2_approx(m0 - M), w1 = ex2_approx(m1 - M);
      const float L = w0 * xl[r] + w1 * xl[BM + r];
      const float inv = (L > 0.f) ? out_mul / L : 0.f;
      if (h == 0 && qrow < N) {
        float lg;
        asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(L));
        LSE[static_cast<size_t>(bh) * N + qrow] = (M + lg) * kLn2;
      }
      __nv_bfloat16 *orow = O + (static_cast<size_t>(bh) * N + qrow) * D + 64 * h;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t a[32], e1[32];
        tmem_ld_32cols(tmem + lane_addr + TM_O + 64 * h + 32 * c, a);
        tmem_ld_32cols(tmem + lane_addr + TM_O + D + 64 * h + 32 * c, e1);
        tmem_ld_wait_regs(a);
        reg_fence32(e1);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float o0 = (w0 * __uint_as_float(a[2 * e]) + w1 * __uint_as_float(e1[2 * e])) * inv;
          const float o1 =
              (w0 * __uint_as_float(a[2 * e + 1]) + w1 * __uint_as_float(e1[2 * e + 1])) * inv;
          pk[e] = pack_bf16x2(o0, o1);
        }
        if (qrow < N) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st_global_v4(orow + 32 * c + 8 * v, pk[4 * v], pk[4 * v + 1], pk[4 * v + 2],
                         pk[4 * v + 3]);
        }
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

// [BH, rows, cols] bytes as a 3-D tensor map: boxes of 128 x 128 bytes,
// 128-byte swizzle; rows (and columns) outside read as zeros.
static bool make_u8_map(CUtensorMap *m, const void *base, int heads, int rows, int cols,
                        int row_stride) {
  return make_bytes_map(m, base, heads, rows, cols, row_stride, 128, 128);
}

template <bool CAUSAL>
static cudaError_t launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mvt,
                            void *O, float *LSE, int N, int BH, int n_blk, float scale_log2,
                            float out_mul, unsigned *status, cudaStream_t stream) {
  auto kern = attn_fwd_fp8_kernel<CAUSAL>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = smem_limit_once(kern, static_cast<int>(SMEM_ALLOC), smem_set);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(BH) * n_blk, kThreads, SMEM_ALLOC, stream>>>(
      mq, mk, mvt, static_cast<__nv_bfloat16 *>(O), LSE, N, BH, n_blk, scale_log2, out_mul,
      status);
  return cudaGetLastError();
}

}  // namespace f8

size_t fwd_fp8_ws_bytes(int B, int H, int N) {
  const size_t n_pad = static_cast<size_t>((N + 15) / 16) * 16;
  return static_cast<size_t>(B) * H * f8::D * n_pad;
}

cudaError_t launch_fwd_fp8(const void *Q8, const void *K8, const void *V8, void *O, float *LSE,
                           int B, int H, int N, float scale, float descale_q, float descale_k,
                           float descale_v, int causal, void *ws, unsigned *status,
                           cudaStream_t stream) {
  using namespace f8;
  const int BH = B * H;
  const int N_pad = (N + 15) / 16 * 16;
  const dim3 tgrid(static_cast<unsigned>((N + 127) / 128), static_cast<unsigned>(BH));
  attn_fp8_vt_kernel<<<tgrid, 256, 0, stream>>>(static_cast<const uint8_t *>(V8),
                                                 static_cast<uint8_t *>(ws), N, N_pad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mvt;
  if (!make_u8_map(&mq, Q8, BH, N, D, D) || !make_u8_map(&mk, K8, BH, N, D, D) ||
      !make_u8_map(&mvt, ws, BH, D, N, N_pad))
    return cudaErrorInvalidValue;
  const int n_blk = (N + BM - 1) / BM;
  const float scale_log2 = scale * descale_q * descale_k * 1.44269504088896340736f;
  const float out_mul = descale_v / kPScale;
  return causal ? launch_t<true>(mq, mk, mvt, O, LSE, N, BH, n_blk, scale_log2, out_mul, status,
                                 stream)
                : launch_t<false>(mq, mk, mvt, O, LSE, N, BH, n_blk, scale_log2, out_mul, status,
                                  stream);
}

}  // namespace ea
