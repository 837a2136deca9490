// fwd_sm103a.cu — fused exact-attention forward for GB300 (sm_103a).
//
// Computes O = softmax(scale * Q K^T + causal mask) V and the row log-sum-exp
// for every (batch, head), following "Why Fast GPUs Still Wait for Memory",
// sections "Attention from first principles" (the definition) and
// "FlashAttention is an IO algorithm": Q is split into blocks of B_r = 128
// rows, K/V into blocks of B_c = 128 keys that stream through shared memory,
// and a running maximum and normaliser per row rescale the output block as
// each K/V block arrives, so S and P never reach HBM.  Causal masking follows
// the note "causal masking is not an optimisation here" on the same page:
// K/V blocks entirely above the diagonal are never loaded or multiplied.
//
// GB300 mapping (one CTA per 128-row query tile, 6 warps):
//   warp 4     TMA producer: Q tile once, then K_j / V_j into a ring of
//              STAGES shared-memory slots (128-byte swizzle), each slot
//              guarded by full/empty mbarriers.
//   warp 5     MMA issuer (one thread): tcgen05.mma S_j = Q K_j^T into one of
//              two TMEM S buffers, then O += P_j V_j into the TMEM O
//              accumulator; tcgen05.commit signals the other roles.
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r); reads its S
//              row from TMEM, masks, updates the running max m and sum l in
//              the base-2 domain (scale * log2(e) folded into one FMA before
//              ex2), rescales its O row in TMEM when m moved, and writes P as
//              bf16 into a swizzled shared-memory tile for the P V MMA.
//              The epilogue divides by l, rounds to bf16 and writes O and LSE.
// S is double-buffered in TMEM, so the tensor core computes S_{j+1} while
// the softmax warps are still working on S_j.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace ea {
namespace fwd {

constexpr int BM = 128;                  // query rows per tile (B_r)
constexpr int BN = 128;                  // keys per K/V tile (B_c)
constexpr int kSoftmaxThreads = 128;     // warps 0-3
constexpr int kWarpTMA = 4;
constexpr int kWarpMMA = 5;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;      // S0 | S1 | O
constexpr uint32_t kTmemS0 = 0;
constexpr uint32_t kTmemS1 = 128;
constexpr uint32_t kTmemO = 256;
constexpr uint32_t kBoxBytes = 64 * 128 * 2;   // one TMA box: 64 columns x 128 rows bf16
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int KB = D / 64;                 // 128-byte swizzle column blocks
  static constexpr int STAGES = (D == 128) ? 2 : 3;
  static constexpr uint32_t Q_BYTES = BM * D * 2;
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr uint32_t P_BYTES = BM * BN * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr uint32_t OFF_P = OFF_V + STAGES * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_P + P_BYTES;
  // q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], p_full, o_done, drain
  static constexpr int NBAR = 1 + 3 * STAGES + 2 + 3;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;
  static constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;   // 1024-byte alignment slack
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, __nv_bfloat16 *__restrict__ O,
                    float *__restrict__ LSE, int N, int BH, int n_qt, float scale_log2,
                    unsigned *status) {
  using C = Cfg<D>;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Heads vary fastest and, for causal, the longest query tiles go first.
  const int bh = blockIdx.x % BH;
  const int qt = n_qt - 1 - static_cast<int>(blockIdx.x / BH);
  const int q0 = qt * BM;
  const int n_kv_total = (N + BN - 1) / BN;
  const int n_kv = CAUSAL ? min(qt + 1, n_kv_total) : n_kv_total;

  const uint32_t bar0 = sb + C::OFF_BAR;
  const uint32_t B_Q = bar0;
  auto B_K = [&](int st) { return bar0 + 8u * (1 + st); };
  auto B_V = [&](int st) { return bar0 + 8u * (1 + S + st); };
  auto B_E = [&](int st) { return bar0 + 8u * (1 + 2 * S + st); };
  auto B_S = [&](int b) { return bar0 + 8u * (1 + 3 * S + b); };
  const uint32_t B_P = bar0 + 8u * (3 + 3 * S);
  const uint32_t B_O = bar0 + 8u * (4 + 3 * S);
  const uint32_t B_DRAIN = bar0 + 8u * (5 + 3 * S);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    mbar_init(B_Q, 1);
    for (int st = 0; st < S; ++st) {
      mbar_init(B_K(st), 1);
      mbar_init(B_V(st), 1);
      mbar_init(B_E(st), 1);
    }
    mbar_init(B_S(0), 1);
    mbar_init(B_S(1), 1);
    mbar_init(B_P, kSoftmaxThreads);
    mbar_init(B_O, 1);
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

  if (warp == kWarpTMA) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(B_Q, C::Q_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_3d(sb + C::OFF_Q + kb * kBoxBytes, &tmQ, kb * 64, q0, bh, B_Q);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % S;
        const uint32_t ph = (j / S) & 1;
        if (!mbar_wait(B_E(st), ph ^ 1u, status, abort_flag)) break;
        mbar_arrive_expect_tx(B_K(st), C::KV_BYTES);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(sb + C::OFF_K + st * C::KV_BYTES + kb * kBoxBytes, &tmK, kb * 64, j * BN,
                      bh, B_K(st));
        mbar_arrive_expect_tx(B_V(st), C::KV_BYTES);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(sb + C::OFF_V + st * C::KV_BYTES + kb * kBoxBytes, &tmV, kb * 64, j * BN,
                      bh, B_V(st));
        issued = j + 1;
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        mbar_wait_drain(B_Q, 0, 100000000ull);
        for (int st = 0; st < S && st < issued; ++st) {
          const int last = st + ((issued - 1 - st) / S) * S;
          mbar_wait_drain(B_K(st), (last / S) & 1, 100000000ull);
          mbar_wait_drain(B_V(st), (last / S) & 1, 100000000ull);
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = make_idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t kIdescPV = make_idesc_bf16(BM, D, 0, 1);
      // S_j = Q K_j^T: both operands K-major (head dim contiguous).
      auto issue_qk = [&](uint32_t d_tmem, int st) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          const uint64_t a = make_sdesc_sw128(sb + C::OFF_Q + koff, 16, 1024);
          const uint64_t b = make_sdesc_sw128(sb + C::OFF_K + st * C::KV_BYTES + koff, 16, 1024);
          mma_bf16_ss(d_tmem, a, b, kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      // O += P_j V_j: P is K-major (keys contiguous); V is MN-major (head dim
      // contiguous), 64-column blocks kBoxBytes apart, 8-key groups 1024 B apart.
      auto issue_pv = [&](int st, bool acc) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t a =
              make_sdesc_sw128(sb + C::OFF_P + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t b =
              make_sdesc_sw128(sb + C::OFF_V + st * C::KV_BYTES + kk * 16 * 128, kBoxBytes, 1024);
          mma_bf16_ss(tmem + kTmemO, a, b, kIdescPV, (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(B_Q, 0, status, abort_flag) && mbar_wait(B_K(0), 0, status, abort_flag);
      if (ok) {
        tc_fence_after();
        issue_qk(tmem + kTmemS0, 0);
        mma_commit(B_S(0));
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          // S buffer (j+1)&1 was released when the softmax warps signalled P_{j-1}.
          const int st1 = (j + 1) % S;
          if (!mbar_wait(B_K(st1), ((j + 1) / S) & 1, status, abort_flag)) break;
          tc_fence_after();
          issue_qk(tmem + (((j + 1) & 1) ? kTmemS1 : kTmemS0), st1);
          mma_commit(B_S((j + 1) & 1));
        }
        const int st = j % S;
        if (!mbar_wait(B_P, j & 1, status, abort_flag)) break;
        if (!mbar_wait(B_V(st), (j / S) & 1, status, abort_flag)) break;
        tc_fence_after();
        issue_pv(st, j > 0);
        mma_commit(B_O);
        if (j + S < n_kv) mma_commit(B_E(st));   // slot refilled only if a later tile needs it
      }
      // Every MMA issued so far must finish before TMEM is released.
      mma_commit(B_DRAIN);
      mbar_wait_drain(B_DRAIN, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------- softmax warps
    const int r = threadIdx.x;               // row within the tile == TMEM lane
    const int qrow = q0 + r;
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    float m = -INFINITY;                     // running max of scale*log2(e)*s
    float l = 0.f;                           // running sum of exp2(x - m)
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(B_S(b), (j >> 1) & 1, status, abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
      const uint32_t s_addr = tmem + lane_addr + (b ? kTmemS1 : kTmemS0);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32cols(s_addr + c * 32, sr[c]);
      tmem_ld_wait();
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      if (j == n_kv - 1 && (CAUSAL || (N % BN) != 0)) {
        const int kv0 = j * BN;
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int key = kv0 + c;
          if (key >= N || (CAUSAL && key > qrow)) s[c] = -INFINITY;
        }
      }
      float mt = s[0];
#pragma unroll
      for (int c = 1; c < BN; ++c) mt = fmaxf(mt, s[c]);
      const float m_new = fmaxf(m, mt * scale_log2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m - m_use);
      float rs = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float p0 = ex2_approx(fmaf(s[2 * c], scale_log2, -m_use));
        const float p1 = ex2_approx(fmaf(s[2 * c + 1], scale_log2, -m_use));
        rs += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + rs;
      m = m_new;
      if (j > 0) {
        // P_{j-1} V_{j-1} must be done before O is rescaled and P is overwritten.
        ok = __all_sync(0xffffffffu, mbar_wait(B_O, (j - 1) & 1, status, abort_flag));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            const uint32_t o_addr = tmem + lane_addr + kTmemO + c * 32;
            tmem_ld_32cols(o_addr, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_32cols(o_addr, o);
          }
          tmem_st_wait();
        }
      }
      // P row r -> 128-byte-swizzled K-major tile: 16-byte chunk ch of a row
      // lands at chunk (ch ^ (row & 7)), as the TMA swizzle would place it.
#pragma unroll
      for (int c16 = 0; c16 < BN / 8; ++c16) {
        const uint32_t addr = sb + C::OFF_P + (c16 >> 3) * kBoxBytes + r * 128 +
                              ((static_cast<uint32_t>(c16 & 7) ^ (r & 7)) << 4);
        st_shared_v4(addr, pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(B_P);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(B_O, (n_kv - 1) & 1, status, abort_flag));
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      __nv_bfloat16 *orow = O + (static_cast<size_t>(bh) * N + qrow) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32cols(tmem + lane_addr + kTmemO + c * 32, o);
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
  const int n_qt = (N + BM - 1) / BM;
  const long long grid = static_cast<long long>(BH) * n_qt;
  kern<<<static_cast<unsigned>(grid), kThreads, C::SMEM_ALLOC, stream>>>(
      mq, mk, mv, static_cast<__nv_bfloat16 *>(O), LSE, N, BH, n_qt, scale_log2, status);
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
