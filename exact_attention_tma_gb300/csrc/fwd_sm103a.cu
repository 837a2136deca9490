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
// GB300 mapping: a work item is two 128-row query tiles of one head (256
// rows), whose K/V tiles stream once for both.  One persistent CTA per SM
// (18 warps) takes items one after another from a global counter, longest
// causal items first:
//   warps 0-7   softmax of query tile 0, warps 8-15 of query tile 1: warps
//               8i+q and 8i+q+4 share TMEM lanes 32q..32q+31, i.e. rows
//               32q..32q+31 of tile i; warp 8i+q takes keys 0-63 of every K/V
//               tile, warp 8i+q+4 keys 64-127 (thread = row)
//   warp 16     MMA issuer (one elected lane): tcgen05.mma S_i = Q_i K_j^T into
//               TMEM (both operands from swizzled shared memory), then
//               O += P_i V_j with P_i read straight from TMEM (each key half
//               overwrites the first 32 of its own 64 S columns as packed bf16)
//   warp 17     TMA producer: the item's Q tiles, K_j and V_j into separate
//               rings guarded by full/empty mbarriers; it claims the next
//               item and passes its index to the other warps
// Item boundaries overlap: the next item's first K/V tiles load while the
// current one finishes, and its Q tiles as soon as their buffers are free
// (after the last Q K^T where O has a staging buffer of its own, after the
// epilogue's store where O is staged in the Q buffer).
// Each sub-partition runs four softmax warps, two per query tile: while one
// tile's warps wait for their scores or hand P over, the other tile's warps
// keep the MUFU and FMA pipes busy, and the tensor core runs one tile's MMAs
// while the other tile's softmax works.
//
// Softmax per K/V tile, in the exp2 domain (x = s * scale * log2 e): the
// exponentials are computed against the running maximum m straight away (no
// separate max pass).  Only if a key half's P sum exceeds 2^15 (so some P
// exceeds 2^9: lazy rescaling) is the tile redone with the new maximum and the
// O accumulator scaled by 2^(m_old - m_new) in TMEM; otherwise the stale m is
// kept for both P and the row sum, so O / l is unchanged and P stays below
// 2^15.  The first tile computes its maximum first.  O is quiescent while the
// softmax of tile i runs: the MMA that wrote it last was committed before S_i
// was.  At d = 128 both key halves accumulate into one O_i, so they agree on
// every rescale through a named barrier; at d = 64 TMEM holds one accumulator
// per key half, each half keeps its own maximum and sum, and the two are
// merged once in the epilogue.
//
// FP8 instance (d = 128): Q, K and V arrive as E4M3 (V transposed, [d][keys],
// so that P V reads a K-major B as kind::f8f6f4 requires); both products run
// at the 8-bit rate with 32-byte k-steps, P is written to TMEM as E4M3
// quadruples (keys 0-63 of a half in 16 columns), scaled by 2^2 so that the
// smallest P kept (2^-8) is a normal E4M3 number, and the lazy-rescale
// threshold drops to a half-row sum of 64 (every P <= 64, so P * 4 stays
// below E4M3's 448).  Q_i holds half as many bytes, so O is staged in a
// buffer of its own; the epilogue multiplies by V's descale over 2^2.
//
// Registers: 18 warps leave 96 per thread (a sub-partition holds five warps);
// the softmax reads its 64 scores as two 32-column loads in turn so that it
// fits.
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
constexpr int kThreads = 576;
constexpr int kWarpMMA = 16;
constexpr int kWarpTMA = 17;
constexpr uint32_t kTmemCols = 512;      // S0 | S1 | O0 | O1
constexpr int kRing = 4;                 // item indices in flight from the TMA warp to the others
constexpr uint32_t kBoxBytes = 64 * 128 * 2;   // one TMA box: 64 columns x 128 rows bf16
constexpr float kLn2 = 0.69314718055994530942f;
// A half row (64 keys) whose P sum exceeds 2^15 has some P above 2^9: its
// maximum has grown and the tile is redone against the new maximum.  Below
// that P <= 2^15, harmless for bf16 P and the fp32 accumulators.
constexpr float kRescaleSum = 32768.0f;
// Running maximum of a key half that has seen no visible key yet: any visible
// score then overflows the half's P sum to +inf, which takes the rescale path.
constexpr float kMInit = -1.0e30f;
// First tile started from m = 0 (bf16, d = 128): a half row whose P sum is
// below 2^-50 has every score below about -44 (base 2); the tile is then
// redone against its true maximum, so that no P falls near fp32's normal
// range.
constexpr float kTinySum = 8.8817841970012523e-16f;   // 2^-50

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

// F8: Q, K and V are E4M3 (one byte per element) and V arrives transposed
// (V^T tiles [d][keys], so P V reads a K-major B); P is E4M3 in TMEM.
template <int D, bool F8 = false>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dimension");
  static_assert(!F8 || D == 128, "FP8 forward: d = 128");
  static constexpr int ESZ = F8 ? 1 : 2;            // bytes per element
  static constexpr int KB = D * ESZ / 128;          // 128-byte swizzle column blocks
  static constexpr int BOX_COLS = 128 / ESZ;        // elements per 128-byte box row
  static constexpr int KSTEPS = D * ESZ / 32;       // 32-byte k-steps of Q K^T
  static constexpr int PSTEPS = BN * ESZ / 32;      // 32-byte k-steps of P V (keys)
  static constexpr int SK = F8 ? 3 : (D == 128) ? EA_FWD_SK128 : EA_FWD_SK64;   // K ring stages
  static constexpr int SV = F8 ? 3 : (D == 128) ? EA_FWD_SV128 : EA_FWD_SV64;   // V ring stages
  static constexpr uint32_t Q_BYTES = BM * D * ESZ;   // one query tile
  static constexpr uint32_t KV_BYTES = BN * D * ESZ;  // one K or V tile
  // Q buffers hold the query tiles of QD items (QD = 2 where shared memory
  // allows: the next item's tiles then load while the current item runs).
  static constexpr int QD = (D == 64 && !F8) ? 2 : 1;
  static constexpr int NQB = QT * QD;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + NQB * Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + SK * KV_BYTES;
  // d = 64: the two key halves of a row keep separate maxima, sums and O
  // accumulators (merged once at the end); d = 128 (no room in TMEM for that):
  // the halves agree on every rescale and share one O accumulator.
  static constexpr bool kIndep = (D == 64);
  static constexpr int NPB = kIndep ? 2 : 1;        // P hand-off barriers per query tile
  // Pair exchange between the two key-half warps of a row: with independent
  // halves the maxima and the sums side by side, float[2][QT][2][BM]; with a
  // shared accumulator one float[QT][2][BM] that carries the maxima during
  // the K/V steps and the sums in the epilogue.
  static constexpr uint32_t XCH_BYTES = (kIndep ? 2 : 1) * QT * 2 * BM * 4;
  static constexpr uint32_t OFF_XCH = OFF_V + SV * KV_BYTES;
  // The epilogue stages O (bf16) for its TMA store in buffers of its own, so
  // a Q buffer is free as soon as the item's last Q K^T has read it.  At
  // d = 128 bf16 (shared memory is full) both query tiles use one staging
  // buffer in turn; otherwise each tile has its own.
  static constexpr uint32_t O_TILE = BM * D * 2;
  static constexpr int NSTG = (D == 128 && !F8) ? 1 : QT;
  static constexpr uint32_t OFF_OST = OFF_XCH + XCH_BYTES;
  static_assert(OFF_OST % 1024 == 0, "128-byte-swizzled staging needs 1024-byte alignment");
  static constexpr uint32_t OFF_BAR = OFF_OST + NSTG * O_TILE;
  // q[NQB], qe[NQB], kf[SK], ke[SK], vf[SV], ve[SV], s[QT], p[QT][NPB], o[QT],
  // drain, ostg, item ring full[kRing], empty[kRing]
  static constexpr int NBAR = 2 * NQB + 2 * SK + 2 * SV + QT + QT * NPB + QT + 2 + 2 * kRing;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  // tmem slot, abort flag, pair_abort[8], item ring
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 48 + 4 * kRing;
  static constexpr uint32_t kSmemMax = 232448;        // 227 KB per CTA
  // Slack to align the dynamic shared memory to 1024 bytes where it fits;
  // without it the kernel checks the alignment it was given (and reports a
  // set-up error instead of running if it is not 1024-byte aligned).
  static constexpr uint32_t SMEM_ALLOC =
      SMEM_BYTES + 1024 <= kSmemMax ? SMEM_BYTES + 1024 : SMEM_BYTES;
  static_assert(SMEM_ALLOC <= kSmemMax, "shared memory budget");
  static constexpr uint32_t TMEM_S = 0;               // S_i at column 128 * i
  // O accumulators at TMEM_O + D * b: b = i (shared by both halves) or
  // b = 2 i + h (one per key half h).
  static constexpr uint32_t TMEM_O = QT * BN;
  static_assert(TMEM_O + QT * NPB * D <= kTmemCols, "tensor memory budget");
};


// exp2 of W consecutive scores of one row against the maximum m (-nm = m):
// p = 2^(s * scale_log2 - m), packed as bf16 pairs into pk (W / 2 words);
// adds the p to the two fp32x2 partial sums rs2.
template <int W>
__device__ __forceinline__ void exp_chunk(const uint32_t (&sr)[W], float2 sc2, float2 nm2,
                                          uint32_t *pk, float2 (&rs2)[2]) {
#pragma unroll
  for (int c = 0; c < W / 2; ++c) {
    const float2 x = ffma2(make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])),
                           sc2, nm2);
    const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    rs2[c & 1] = fadd2(rs2[c & 1], p);
    pk[c] = pack_bf16x2(p.x, p.y);
  }
}

// FP8 variant: P is rounded to E4M3 as P * 2^2 (nm2 = 2 - m); the lazy
// rescale keeps every P <= 64 (a 64-key half's sum <= 64), so P * 4 <= 256
// stays below E4M3's 448 and P >= 2^-8 stays a normal number.  Packs four
// scores per word (key order, low byte first; W / 4 words); adds the P * 4 to rs2.
constexpr float kPScale8 = 4.0f;
constexpr float kLog2PScale8 = 2.0f;
constexpr float kRescaleSum8 = 64.0f;
template <int W>
__device__ __forceinline__ void exp_chunk_f8(const uint32_t (&sr)[W], float2 sc2, float2 nm2,
                                             uint32_t *pk, float2 (&rs2)[2]) {
#pragma unroll
  for (int c = 0; c < W / 4; ++c) {
    const float2 x0 = ffma2(make_float2(__uint_as_float(sr[4 * c]), __uint_as_float(sr[4 * c + 1])),
                            sc2, nm2);
    const float2 x1 = ffma2(
        make_float2(__uint_as_float(sr[4 * c + 2]), __uint_as_float(sr[4 * c + 3])), sc2, nm2);
    const float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
    const float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
    rs2[0] = fadd2(rs2[0], p0);
    rs2[1] = fadd2(rs2[1], p1);
    pk[c] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
  }
}

// Scores of keys first_key .. first_key + W - 1 that lie past the last
// visible key lim become -inf (so p = 0).
template <int W>
__device__ __forceinline__ void mask_chunk(uint32_t (&sr)[W], int first_key, int lim) {
  if (first_key + W - 1 > lim) {
#pragma unroll
    for (int c = 0; c < W; ++c)
      if (first_key + c > lim) sr[c] = __float_as_uint(-INFINITY);
  }
}

template <int D, bool CAUSAL, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    float *__restrict__ LSE, int N, int BH, int n_blk, int H, int group,
                    float scale_log2, float out_mul, unsigned *status, unsigned *sched) {
  using C = Cfg<D, F8>;
  constexpr int SK = C::SK;
  constexpr int SV = C::SV;
  constexpr int QD = C::QD;
  constexpr int NQB = C::NQB;
  extern __shared__ uint8_t smem_raw[];
  if constexpr (C::SMEM_ALLOC == C::SMEM_BYTES) {
    // No room for alignment slack: the 128-byte-swizzled buffers need the
    // dynamic shared memory 1024-byte aligned as given (the same for every
    // CTA, so the whole grid takes this exit together, before any barrier).
    if ((smem_u32(smem_raw) & 1023u) != 0) {
      if (threadIdx.x == 0) atomicOr(status, kStatusSetupBit);
      return;
    }
  }
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = warp >> 2;

  // Work items are (head, 256-row query block) pairs.  Causal: heads vary
  // fastest and the longest query blocks come first; non-causal: query blocks
  // vary fastest, so the CTAs working at the same time share a few heads' K/V
  // through L2.  The CTA is persistent: it starts with item blockIdx and
  // claims each further item from a global counter (sched[0]) once it has
  // issued the loads of the current one, so the items go out in order to
  // whichever CTA frees up first.  The TMA warp claims them and hands each
  // item index to the MMA and softmax warps through a small ring in shared
  // memory; the last CTA to finish resets the counter for the next launch.
  const int n_items = BH * n_blk;
  const int G = static_cast<int>(gridDim.x);
  const int n_kv_total = (N + BN - 1) / BN;
  struct Item {
    int bh, kvh, q0, n0, n1;   // head, K/V head, first query row, K/V tiles of query tiles 0, 1
  };
  auto item_at = [&](int k, Item &it) {
    if (k >= n_items) return false;
    const int blk = CAUSAL ? n_blk - 1 - k / BH : k % n_blk;
    it.bh = CAUSAL ? k % BH : k / n_blk;
    // K/V head read by query head bh: H query heads per batch share H / group
    // K/V heads in contiguous groups ("Why Fast GPUs Still Wait for Memory",
    // Attention III: GQA with group size g; g = 1 is multi-head attention).
    it.kvh = (it.bh / H) * (H / group) + (it.bh % H) / group;
    it.q0 = blk * (QT * BM);
    // K/V tiles each query tile needs (query tile 0 can stop one tile earlier when causal).
    it.n0 = CAUSAL ? min(QT * blk + 1, n_kv_total) : n_kv_total;
    it.n1 = CAUSAL ? min(QT * blk + 2, n_kv_total) : n_kv_total;
    return true;
  };

  // Barrier phases run on across items: the K/V rings count K/V tiles over
  // the CTA's whole sequence, S_i / P_i count tile i's K/V steps, and the Q_i
  // and O_i barriers complete once per item.
  const uint32_t bar0 = sb + C::OFF_BAR;
  auto B_Q = [&](int b) { return bar0 + 8u * b; };                    // Q buffer b loaded
  auto B_QE = [&](int b) { return bar0 + 8u * (NQB + b); };           // Q buffer b free
  auto B_KF = [&](int s) { return bar0 + 8u * (2 * NQB + s); };
  auto B_KE = [&](int s) { return bar0 + 8u * (2 * NQB + SK + s); };
  auto B_VF = [&](int s) { return bar0 + 8u * (2 * NQB + 2 * SK + s); };
  auto B_VE = [&](int s) { return bar0 + 8u * (2 * NQB + 2 * SK + SV + s); };
  constexpr int kB5 = 2 * NQB + 2 * SK + 2 * SV;
  auto B_S = [&](int i) { return bar0 + 8u * (kB5 + i); };            // S_i ready (MMA)
  constexpr int NPB = C::NPB;
  // P_i written by the softmax (per key half when the halves are independent)
  auto B_P = [&](int i, int hh) { return bar0 + 8u * (kB5 + QT + i * NPB + (NPB > 1 ? hh : 0)); };
  auto B_O = [&](int i) { return bar0 + 8u * (kB5 + QT + QT * NPB + i); };   // item's last P_i V_j done
  const uint32_t B_DRAIN = bar0 + 8u * (kB5 + 2 * QT + QT * NPB);
  // The shared O staging buffer has been read by its latest TMA store (one
  // completion per epilogue; used when both query tiles share the buffer).
  const uint32_t B_OSTG = B_DRAIN + 8u;
  constexpr int kB6 = kB5 + 2 * QT + QT * NPB + 2;
  auto B_IF = [&](int s) { return bar0 + 8u * (kB6 + s); };           // item slot s written
  auto B_IE = [&](int s) { return bar0 + 8u * (kB6 + kRing + s); };   // item slot s read by all
  static_assert(kB6 + 2 * kRing == C::NBAR, "barrier count");
  // Query tile i of the CTA's t-th item uses Q buffer qbuf(t, i), for the
  // quse(t)-th time (the parity of the buffer's barrier phases).
  auto qbuf = [&](int t, int i) { return (t % QD) * QT + i; };
  auto quse = [&](int t) { return t / QD; };
  volatile int *item_ring = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 48);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  // Set by a softmax warp whose wait gave up, read by it and its partner warp
  // after their shared barrier (so both take the same exit).
  volatile int *pair_abort = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 16);
  // The t-th item of this CTA as the TMA warp published it (warp-uniform):
  // false past the last item, or when the wait gave up (then ok = false).
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
  // K_j and V_j into ring stages sk / sv: 128-byte-wide column boxes of the
  // [keys][d] tiles, or with FP8 one box of K and one box of the V^T tile
  // [d][keys] (keys contiguous).
  auto load_k = [&](int kvh, int j, int sk) {
#pragma unroll
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_3d(sb + C::OFF_K + sk * C::KV_BYTES + kb * kBoxBytes, &tmK, kb * C::BOX_COLS,
                  j * BN, kvh, B_KF(sk));
  };
  auto load_v = [&](int kvh, int j, int sv) {
    const uint32_t dst = sb + C::OFF_V + sv * C::KV_BYTES;
    if constexpr (F8) {
      tma_load_3d(dst, &tmV, j * BN, 0, kvh, B_VF(sv));
    } else {
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_3d(dst + kb * kBoxBytes, &tmV, kb * 64, j * BN, kvh, B_VF(sv));
    }
  };
  auto load_q = [&](const Item &it, int i, int qb) {
    mbar_arrive_expect_tx(B_Q(qb), C::Q_BYTES);
#pragma unroll
    for (int kb = 0; kb < C::KB; ++kb)
      tma_load_3d(sb + C::OFF_Q + qb * C::Q_BYTES + kb * kBoxBytes, &tmQ, kb * C::BOX_COLS,
                  it.q0 + i * BM, it.bh, B_Q(qb));
  };
  // One thread of the TMA warp sets up the barriers and at once starts the
  // first item's loads, in the order the first MMAs need them (Q_0 and K_0,
  // then Q_1 and V_0), while the MMA warp allocates TMEM.
  // The next kernel in the stream may launch now (it cannot share an SM with
  // this one's shared memory, and it waits for this grid before reading).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == kWarpTMA * 32) {
    for (int qb = 0; qb < NQB; ++qb) {
      mbar_init(B_Q(qb), 1);
      mbar_init(B_QE(qb), 1);
    }
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
      for (int hh = 0; hh < NPB; ++hh) mbar_init(B_P(i, hh), 2 * BM / NPB / 32);   // one arrival per warp
      mbar_init(B_O(i), 1);
    }
    mbar_init(B_DRAIN, 1);
    mbar_init(B_OSTG, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(B_IF(s), 1);
      mbar_init(B_IE(s), 1 + 8 * QT);   // the MMA warp and every softmax warp
    }
    *abort_flag = 0;
    for (int p = 0; p < 8; ++p) pair_abort[p] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
    Item it0;
    if (item_at(static_cast<int>(blockIdx.x), it0)) {   // (always true: the grid is no larger than the item count)
      // Launched as a programmatic dependent of the previous kernel in the
      // stream: its inputs may come from that kernel, so wait for it before
      // the first load (bf16; the FP8 instance's Q and K come from before the
      // V^T pass, so it waits just before its first V^T load).
      if constexpr (!F8) asm volatile("griddepcontrol.wait;" ::: "memory");
      load_q(it0, 0, 0);
      mbar_arrive_expect_tx(B_KF(0), C::KV_BYTES);
      load_k(it0.kvh, 0, 0);
      for (int i = 1; i < QT; ++i) load_q(it0, i, i);
      mbar_arrive_expect_tx(B_VF(0), C::KV_BYTES);
      // FP8: V^T comes from the transpose pass launched just before this
      // kernel, which may still be finishing (programmatic dependent launch).
      if constexpr (F8) asm volatile("griddepcontrol.wait;" ::: "memory");
      load_v(it0.kvh, 0, 0);
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

  if (warp < 8 * QT) {
    // ------------------------------------------------------------ softmax
    // Warps 8i + q and 8i + q + 4 share TMEM lanes 32q..32q+31 (rows
    // 32q..32q+31 of query tile i): the first takes keys 0-63 of every K/V
    // tile, the second keys 64-127.
    // With one O accumulator per row (d = 128) the pair agrees through its own
    // named barrier on each rescale (and on an abort); with one per key half
    // (d = 64) the halves run independently.  Either way the pair combines its
    // partial sums (and maxima) once at the end of each item.
    constexpr bool kIndep = C::kIndep;
    const int i = warp >> 3;                 // query tile of this group of 8 warps
    const int h = wg & 1;                    // key half
    const int q = warp & 3;
    const int r = q * 32 + lane;             // row within a tile == TMEM lane
    const uint32_t pair_bar = 1 + 4 * i + q;
    const uint32_t kEpiBar = 9 + i;          // named barrier of the group's 256 threads
    const int pa = 4 * i + q;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    float *xch = reinterpret_cast<float *>(smem + C::OFF_XCH);
    float *xi = xch + i * 2 * BM;            // maxima of the two halves
    // Partial sums of the two halves: beside the maxima, or (shared
    // accumulator) in the same slots once the item's K/V steps are done.
    float *xl = kIndep ? xch + (QT + i) * 2 * BM : xi;
    const float2 sc2 = make_float2(scale_log2, scale_log2);
    const uint32_t s_addr = tmem + lane_addr + C::TMEM_S + i * BN + h * 64;
    // O accumulator columns this thread rescales.
    const uint32_t o_blk =
        tmem + lane_addr + C::TMEM_O + (kIndep ? (2 * i + h) * D : i * D + h * (D / 2));
    // This thread's 64 scores of S_i: P = 2^(x - m_use) packed into pk and
    // their sum, 32 scores at a time.
    auto pass = [&](int k0, int lm, float m_use, uint32_t (&pk)[32], float &rs) {
      const float nm = (F8 ? kLog2PScale8 : 0.f) - m_use;
      const float2 nm2 = make_float2(nm, nm);
      float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      // (The two warps of a sub-partition that share this tile interleave
      // their loads and exponentials; loading the next chunk while this one
      // is exponentiated measured slower.)
      {
        uint32_t a[32];
        tmem_ld_32cols(s_addr, a);
        tmem_ld_wait_regs(a);
        mask_chunk<32>(a, k0, lm);
        if constexpr (F8) exp_chunk_f8<32>(a, sc2, nm2, &pk[0], rs2);
        else exp_chunk<32>(a, sc2, nm2, &pk[0], rs2);
      }
      __syncwarp();
      {
        uint32_t b[32];
        tmem_ld_32cols(s_addr + 32, b);
        tmem_ld_wait_regs(b);
        mask_chunk<32>(b, k0 + 32, lm);
        if constexpr (F8) exp_chunk_f8<32>(b, sc2, nm2, &pk[8], rs2);
        else exp_chunk<32>(b, sc2, nm2, &pk[16], rs2);
      }
      rs = (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
      if constexpr (F8) rs *= 1.0f / kPScale8;
    };
    // Maximum of this thread's 64 (masked) raw scores of S_i.
    auto half_max = [&](int k0, int lm) {
      float mx = -INFINITY;
#pragma unroll 1
      for (int u = 0; u < 2; ++u) {
        uint32_t a[32];
        tmem_ld_32cols(s_addr + 32 * u, a);
        tmem_ld_wait_regs(a);
        mask_chunk<32>(a, k0 + 32 * u, lm);
#pragma unroll
        for (int c = 0; c + 1 < 32; c += 2)
          mx = fmax3(mx, __uint_as_float(a[c]), __uint_as_float(a[c + 1]));
      }
      __syncwarp();
      return mx;
    };
    bool ok = true;
    int base = 0;                            // steps of tile i in earlier items
    for (int t = 0; ok; ++t) {
      Item it;
      if (!take_item(t, it, ok)) break;
      const int n_i = (i == 0) ? it.n0 : it.n1;
      const int lim = CAUSAL ? min(it.q0 + i * BM + r, N - 1) : N - 1;   // last visible key of the row
      float m_i = kIndep ? kMInit : 0.f;     // max used for P (base 2)
      float l_i = 0.f;                       // partial row sum
      for (int j = 0; j < n_i; ++j) {
        // With a shared accumulator, a warp whose wait gave up still takes
        // part in the pair's barriers below; the vote after the pass then
        // ends the loop for both.
        const bool okw =
            __all_sync(0xffffffffu, mbar_wait(B_S(i), (base + j) & 1, status, abort_flag));
        if (kIndep && !okw) {
          ok = false;
          break;
        }
        if (okw) tc_fence_after();
        const int k0 = j * BN + h * 64;
        // bf16 at d = 128 starts the item's first tile from m = 0 instead of
        // a separate maximum pass (redone below against the true maximum if a
        // half's P sum is then too large or too small).
        if (j == 0 && (kIndep || F8)) {
          // First tile: the maximum first (of the half, or of the whole row,
          // which always contains key 0).
          if (kIndep) {
            const float hm = half_max(k0, lim);
            m_i = (hm == -INFINITY) ? kMInit : hm * scale_log2;
          } else {
            xi[h * BM + r] = okw ? half_max(k0, lim) : 0.f;
            named_bar_sync(pair_bar, 64);
            m_i = fmaxf(xi[r], xi[BM + r]) * scale_log2;
          }
        }
        uint32_t pk[32];
        float rs = 0.f;
        if (okw) pass(k0, lim, m_i, pk, rs);
        else pair_abort[pa] = 1;
        // rs above the threshold (or not finite) means some P exceeded it:
        // the maximum grew, and the tile is redone with the new one (by both
        // halves when they share the accumulator).
        bool redo;
        constexpr float kRedo = F8 ? kRescaleSum8 : kRescaleSum;
        if (kIndep) {
          redo = __any_sync(0xffffffffu, !(rs <= kRedo));
        } else {
          redo = named_bar_any(pair_bar, 64,
                               !okw || !(rs <= kRedo) || (!F8 && j == 0 && !(rs >= kTinySum)));
          if (redo && pair_abort[pa]) {
            ok = false;
            break;
          }
        }
        float alpha = 1.f;
        if (redo) {
          float tmax;
          if (kIndep) {
            tmax = half_max(k0, lim);
          } else {
            xi[h * BM + r] = half_max(k0, lim);
            named_bar_sync(pair_bar, 64);
            tmax = fmaxf(xi[r], xi[BM + r]);
          }
          float m_new;
          if constexpr (kIndep || F8) {
            m_new = fmaxf(m_i, tmax * scale_log2);
            alpha = ex2_approx(m_i - m_new);
          } else {
            // (On the first tile nothing has accumulated yet: the factor is
            // 1, and m is the tile's maximum whatever it started from.)
            m_new = fmaxf(j == 0 ? -INFINITY : m_i, tmax * scale_log2);
            alpha = j == 0 ? 1.f : ex2_approx(m_i - m_new);
          }
          m_i = m_new;
          pass(k0, lim, m_i, pk, rs);
          if (j > 0) {
            // This thread's accumulator columns scaled by 2^(m_old - m_new).
            // O_i is quiescent: the MMA that wrote it last was committed
            // before S_i was.
#pragma unroll 1
            for (int c = 0; c < (kIndep ? D / 16 : D / 64); ++c) {
              if constexpr (kIndep) {   // (16 columns at a time: fewer live registers)
                uint32_t o[16];
                tmem_ld_16cols(o_blk + c * 16, o);
                tmem_ld_wait_regs16(o);
#pragma unroll
                for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tmem_st_16cols(o_blk + c * 16, o);
              } else {
                uint32_t o[32];
                tmem_ld_32cols(o_blk + c * 32, o);
                tmem_ld_wait_regs(o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tmem_st_32cols(o_blk + c * 32, o);
              }
            }
          }
        }
        l_i = l_i * alpha + rs;
        // P for keys 64h .. 64h+63 (bf16 pairs, or E4M3 quadruples) over the
        // first 32 (16) of this thread's own S columns, which it has already read.
        if constexpr (F8) tmem_st_16cols(s_addr, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
        else tmem_st_32cols(s_addr, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B_P(i, h));
      }
      // Epilogue of tile i: each warp stages its half of the columns of O_i
      // as bf16 in the staging buffer, in the 128-byte-swizzled box layout of
      // the O tensor map, and one thread stores the tile with TMA (rows past
      // N are dropped by the tensor map); the warp of the low half writes the
      // LSE.  Independent halves are merged with weights
      // 2^(m_h - max(m_0, m_1)).  The next item's P_i V_0 overwrites O_i only
      // after this group has written P_i, i.e. after these TMEM reads.
      const bool okw = ok && __all_sync(0xffffffffu, mbar_wait(B_O(i), t & 1, status, abort_flag));
      if (kIndep) {
        xi[h * BM + r] = m_i;
        xl[h * BM + r] = l_i;
      }
      // The staging buffer must have been read by its previous store: this
      // tile's own previous one (a buffer per tile), or the latest one of
      // either tile (one shared buffer, used by the epilogues in turn: tile
      // 0 of item t, tile 1 of item t, tile 0 of item t + 1, ...).
      bool sok = okw;
      if (threadIdx.x == i * 256) {
        if constexpr (C::NSTG == 1) {
          const int e = 2 * t + i;
          if (e > 0) sok = sok && mbar_wait(B_OSTG, (e - 1) & 1, status, abort_flag);
        } else {
          bulk_wait_group_read0();
        }
      }
      if (named_bar_any(kEpiBar, 2 * BM, !sok)) {
        ok = false;
        break;
      }
      if constexpr (!kIndep) {
        // (The partner warp read its last maximum from these slots before
        // the barrier above.)
        xl[h * BM + r] = l_i;
        named_bar_sync(kEpiBar, 2 * BM);
      }
      tc_fence_after();
      float mrow = m_i, w0 = 1.f, w1 = 1.f;
      if (kIndep) {
        mrow = fmaxf(xi[r], xi[BM + r]);
        w0 = ex2_approx(xi[r] - mrow);
        w1 = ex2_approx(xi[BM + r] - mrow);
      }
      const float lt = w0 * xl[r] + w1 * xl[BM + r];
      const float inv_l = out_mul / lt;
      const float a0 = w0 * inv_l, a1 = w1 * inv_l;
      const int qrow = it.q0 + i * BM + r;
      const uint32_t stage_base = sb + C::OFF_OST + (C::NSTG == 1 ? 0 : i) * C::O_TILE;
      const uint32_t stage = stage_base + static_cast<uint32_t>(r) * 128;
      const uint32_t o_addr = tmem + lane_addr + C::TMEM_O + (kIndep ? 2 * i * D : i * D) + h * (D / 2);
      if constexpr (kIndep) {
        // 16 columns of each half's accumulator at a time (both are live).
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[16], o1[16];
          tmem_ld_16cols(o_addr + c * 16, o);
          tmem_ld_16cols(o_addr + D + c * 16, o1);
          tmem_ld_wait_regs16(o);
          reg_fence16(o1);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            o[e] = __float_as_uint(__uint_as_float(o[e]) * a0 + __uint_as_float(o1[e]) * a1);
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[8 * v + 2 * e]), __uint_as_float(o[8 * v + 2 * e + 1]));
            const int col = h * (D / 2) + c * 16 + v * 8;   // first of these 8 columns
            const uint32_t chunk = static_cast<uint32_t>((col & 63) >> 3) ^ static_cast<uint32_t>(r & 7);
            st_shared_v4(stage + (col >> 6) * kBoxBytes + (chunk << 4), w[0], w[1], w[2], w[3]);
          }
          __syncwarp();
        }
      } else {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t o[32];
          tmem_ld_32cols(o_addr + c * 32, o);
          tmem_ld_wait_regs(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * inv_l);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[8 * v + 2 * e]), __uint_as_float(o[8 * v + 2 * e + 1]));
            const int col = h * (D / 2) + c * 32 + v * 8;   // first of these 8 columns
            const uint32_t chunk = static_cast<uint32_t>((col & 63) >> 3) ^ static_cast<uint32_t>(r & 7);
            st_shared_v4(stage + (col >> 6) * kBoxBytes + (chunk << 4), w[0], w[1], w[2], w[3]);
          }
          __syncwarp();
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(kEpiBar, 2 * BM);
      if (threadIdx.x == i * 256) {
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb)
          tma_store_3d(&tmO, kb * 64, it.q0 + i * BM, it.bh, stage_base + kb * kBoxBytes);
        bulk_commit_group();
        if constexpr (C::NSTG == 1) {
          // Hand the shared buffer to the next epilogue once the store has read it.
          bulk_wait_group_read0();
          mbar_arrive(B_OSTG);
        }
      }
      if (h == 0 && qrow < N) {
        float lg;
        asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(lt));
        LSE[static_cast<size_t>(it.bh) * N + qrow] = (mrow + lg) * kLn2;
      }
      base += n_i;
    }
    // The last stores must have finished reading shared memory before the CTA exits.
    if (threadIdx.x == i * 256) bulk_wait_group_read0();
    tc_fence_before();
  } else {
    // Warps 16 and 17 run their schedules warp-uniformly (every lane waits on the
    // barriers) and one elected lane issues the TMA copies / MMAs, so addresses
    // and descriptors stay in the warp-uniform datapath.
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, abort_flag));
    };
    if (warp == kWarpTMA) {
      // ------------------------------------------------------ TMA producer
      // (Every lane: the loads below follow the previous kernel in the stream.)
      asm volatile("griddepcontrol.wait;" ::: "memory");
      // (The first item's Q tiles and first K/V tile were issued before the
      // CTA-wide barrier.)  A Q buffer is refilled once the MMA warp has
      // released it after its previous item's last Q K^T.
      const bool leader = elect_one();
      int gk = 0, gv = 0;                    // K / V tiles issued so far
      int gq = QT;                           // Q tiles issued so far (item-major)
      bool ok = true;
      auto load_k_next = [&](int kvh, int j) {
        const int sk = gk % SK;
        if (!wait_all(B_KE(sk), ((gk / SK) & 1) ^ 1u)) return false;
        if (leader) {
          mbar_arrive_expect_tx(B_KF(sk), C::KV_BYTES);
          load_k(kvh, j, sk);
        }
        ++gk;
        return true;
      };
      auto load_v_next = [&](int kvh, int j) {
        const int sv = gv % SV;
        if (!wait_all(B_VE(sv), ((gv / SV) & 1) ^ 1u)) return false;
        if (leader) {
          mbar_arrive_expect_tx(B_VF(sv), C::KV_BYTES);
          load_v(kvh, j, sv);
        }
        ++gv;
        return true;
      };
      // Query tile i of the t-th item (t >= 1).
      auto load_q_next = [&](const Item &it, int t, int i) {
        const int qb = qbuf(t, i);
        if (t >= QD && !wait_all(B_QE(qb), (quse(t) - 1) & 1)) return false;
        if (leader) load_q(it, i, qb);
        ++gq;
        return true;
      };
      int k = static_cast<int>(blockIdx.x);
      for (int t = 0; ok; ++t) {
        // Publish item k (or the end of the sequence) to the other warps.
        const int s = t % kRing;
        if (!(ok = wait_all(B_IE(s), ((t / kRing) & 1) ^ 1u))) break;
        if (leader) {
          item_ring[s] = k;
          mbar_arrive(B_IF(s));
        }
        __syncwarp();
        Item it;
        if (!item_at(k, it)) break;
        if (t == 0) {
          gk = gv = 1;
        } else if constexpr (QD > 1) {
          // The Q buffers of this item were released an item ago: Q first.
          ok = load_q_next(it, t, 0) && load_q_next(it, t, 1) && load_k_next(it.kvh, 0) &&
               load_v_next(it.kvh, 0);
        } else {
          // In the order the buffers come free near the end of the previous
          // item (Q_0 of the next item is wanted early, see the MMA warp).
          ok = load_k_next(it.kvh, 0) && load_q_next(it, t, 0) && load_v_next(it.kvh, 0) &&
               load_q_next(it, t, 1);
        }
        for (int j = 1; ok && j < it.n1; ++j) ok = load_k_next(it.kvh, j) && load_v_next(it.kvh, j);
        // This item's loads are all issued: claim the next one.
        int kn = 0;
        if (lane == 0) kn = G + static_cast<int>(atomicAdd(sched, 1u));
        k = __shfl_sync(0xffffffffu, kn, 0);
      }
      if (leader && *abort_flag) {
        // Let every copy this warp started land before the CTA exits.
        for (int x = gq - 1; x >= 0 && x >= gq - NQB; --x)   // the last load of each buffer
          mbar_wait_drain(B_Q(qbuf(x / QT, x % QT)), quse(x / QT) & 1, 100000000ull);
        for (int s = 0; s < SK && s < gk; ++s)
          mbar_wait_drain(B_KF(s), ((gk - 1 - s) / SK) & 1, 100000000ull);
        for (int s = 0; s < SV && s < gv; ++s)
          mbar_wait_drain(B_VF(s), ((gv - 1 - s) / SV) & 1, 100000000ull);
      }
      __syncwarp();
    } else if (warp == kWarpMMA) {
      // ------------------------------------------------------- MMA issuer
      const bool leader = elect_one();
      // bf16: V is MN-major (head dim contiguous); FP8: V^T is K-major.
      constexpr uint32_t kIdescQK = F8 ? make_idesc_e4m3(BM, BN, 0, 0) : make_idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t kIdescPV = F8 ? make_idesc_e4m3(BM, D, 0, 0) : make_idesc_bf16(BM, D, 0, 1);
      // Shared-memory descriptors as low words over one common high word; a
      // k-step or stage moves only the start-address field (byte offset / 16
      // added to the low word).  The issue loops are unrolled so that each MMA
      // costs two integer adds besides the tcgen05.mma itself.
      const uint64_t dQ = make_sdesc_sw128(sb + C::OFF_Q, 16, 1024);
      const uint64_t dK = make_sdesc_sw128(sb + C::OFF_K, 16, 1024);
      const uint64_t dV = F8 ? make_sdesc_sw128(sb + C::OFF_V, 16, 1024)
                             : make_sdesc_sw128(sb + C::OFF_V, kBoxBytes, 1024);
      const uint32_t hi = static_cast<uint32_t>(dQ >> 32);   // identical for dK and dV
      const uint32_t q_lo = static_cast<uint32_t>(dQ);
      const uint32_t k_lo = static_cast<uint32_t>(dK);
      const uint32_t v_lo = static_cast<uint32_t>(dV);
      // S_i = Q K^T from Q buffer qb and K stage sk: both operands K-major
      // (head dim contiguous), 128-B swizzle.
      auto issue_qk = [&](int i, int qb, int sk) {
        const uint32_t a0 = q_lo + ((qb * C::Q_BYTES) >> 4);
        const uint32_t b0 = k_lo + ((sk * C::KV_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {   // 32-byte k-steps, 4 per 128-byte box
          const uint32_t koff = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
          if constexpr (F8)
            mma_f8_ss_lo(tmem + C::TMEM_S + i * BN, a0 + koff, b0 + koff, hi, kIdescQK,
                         kk > 0 ? 1u : 0u);
          else
            mma_bf16_ss_lo(tmem + C::TMEM_S + i * BN, a0 + koff, b0 + koff, hi, kIdescQK,
                           kk > 0 ? 1u : 0u);
        }
      };
      // O += P_i V: P_i from TMEM (8 columns = 16 keys per step; keys 0-63 in
      // columns 0-31 of S_i, keys 64-127 in columns 64-95); V is MN-major
      // (head dim contiguous), 64-column blocks kBoxBytes apart, 8-key groups 1024 B apart.
      // FP8: 32 keys per step, P_i's keys 0-63 in columns 0-15 and keys
      // 64-127 in columns 64-79 (four E4M3 per column); the V^T tile is
      // K-major, 32-byte k-steps along its 128-byte rows.
      auto issue_pv = [&](int i, int sv, bool acc, int kb, int ke, uint32_t o_col) {
        const uint32_t b0 = v_lo + ((sv * C::KV_BYTES) >> 4);
#pragma unroll
        for (int kk = kb; kk < ke; ++kk) {
          if constexpr (F8)
            mma_f8_ts_lo(tmem + o_col, tmem + C::TMEM_S + i * BN + (kk >> 1) * 64 + (kk & 1) * 8,
                         b0 + ((kk * 32) >> 4), hi, kIdescPV, (acc || kk > kb) ? 1u : 0u);
          else
            mma_bf16_ts_lo(tmem + o_col, tmem + C::TMEM_S + i * BN + (kk >> 2) * 64 + (kk & 3) * 8,
                           b0 + ((kk * 16 * 128) >> 4), hi, kIdescPV, (acc || kk > kb) ? 1u : 0u);
        }
      };
      // P_i V_j: one run over all 128 keys into O_i, or (independent halves)
      // keys 0-63 into O_i^0 as soon as that half's P is in, then keys 64-127
      // into O_i^1.  ph: parity of tile i's step.
      auto pv = [&](int i, int sv, int j, uint32_t ph) {
        if constexpr (C::kIndep) {
          if (!wait_all(B_P(i, 0), ph)) return false;
          tc_fence_after();
          if (leader) issue_pv(i, sv, j > 0, 0, C::PSTEPS / 2, C::TMEM_O + 2 * i * D);
          __syncwarp();
          if (!wait_all(B_P(i, 1), ph)) return false;
          tc_fence_after();
          if (leader) issue_pv(i, sv, j > 0, C::PSTEPS / 2, C::PSTEPS, C::TMEM_O + (2 * i + 1) * D);
          __syncwarp();
        } else {
          if (!wait_all(B_P(i, 0), ph)) return false;
          tc_fence_after();
          if (leader) issue_pv(i, sv, j > 0, 0, C::PSTEPS, C::TMEM_O + i * D);
          __syncwarp();
        }
        return true;
      };
      // S_i of the first K/V tile of the t-th item (its K_0 at ring position
      // kg); the caller has seen its operands arrive.  Tile 1 is K_0's last
      // reader; a tile with a single K/V tile releases its Q buffer at once.
      auto first_qk = [&](int i, int t, int kg, const Item &x) {
        issue_qk(i, qbuf(t, i), kg % SK);
        mma_commit(B_S(i));
        if (i == QT - 1) mma_commit(B_KE(kg % SK));
        if ((i == 0 ? x.n0 : x.n1) == 1) mma_commit(B_QE(qbuf(t, i)));
      };
      bool ok = true;
      int gk = 0, gv = 0;                    // ring positions of the current item's K_0 / V_0
      int base0 = 0, base1 = 0;              // steps of tiles 0 / 1 in earlier items
      for (int t = 0; ok; ++t) {
        Item it;
        if (!take_item(t, it, ok)) break;
        const int n0 = it.n0, n1 = it.n1;
        // S_0 = Q_0 K_0^T, then S_1 = Q_1 K_0^T.  The first P_i V_0 below
        // overwrites O_i only after tile i's softmax warps have written P_i,
        // which they do after reading O_i in the previous item's epilogue.
        ok = wait_all(B_Q(qbuf(t, 0)), quse(t) & 1) && wait_all(B_KF(gk % SK), (gk / SK) & 1);
        if (!ok) break;
        tc_fence_after();
        if (leader) first_qk(0, t, gk, it);
        __syncwarp();
        if (!(ok = wait_all(B_Q(qbuf(t, 1)), quse(t) & 1))) break;
        tc_fence_after();
        if (leader) first_qk(1, t, gk, it);
        __syncwarp();
        // Per K/V tile j but the last: the V_j and K_{j+1} stages are checked
        // first (they are normally resident long before), so that each
        // softmax hand-off is followed by one wait and an uninterrupted run of
        // MMAs: P_0 V_j, Q_0 K_{j+1}^T, then P_1 V_j, Q_1 K_{j+1}^T.
        for (int j = 0; ok && j + 1 < n1; ++j) {
          const int vp = gv + j, sv = vp % SV;
          const int kp = gk + j + 1, sk1 = kp % SK;
          if (!(ok = wait_all(B_VF(sv), (vp / SV) & 1) && wait_all(B_KF(sk1), (kp / SK) & 1))) break;
          if (j < n0) {
            if (!(ok = pv(0, sv, j, (base0 + j) & 1))) break;
            if (leader) {
              if (j + 1 == n0) mma_commit(B_O(0));
              if (j + 1 < n0) {
                issue_qk(0, qbuf(t, 0), sk1);   // overwrites S_0/P_0 after the P_0 V_j MMAs above read it
                mma_commit(B_S(0));
                if (j + 2 == n0) mma_commit(B_QE(qbuf(t, 0)));
              }
            }
            __syncwarp();
          }
          if (!(ok = pv(1, sv, j, (base1 + j) & 1))) break;
          if (leader) {
            mma_commit(B_VE(sv));
            issue_qk(1, qbuf(t, 1), sk1);
            mma_commit(B_S(1));
            mma_commit(B_KE(sk1));
            if (j + 2 == n1) mma_commit(B_QE(qbuf(t, 1)));
          }
          __syncwarp();
        }
        // The last K/V tile, kept out of the loop above so that the loop body
        // stays the short steady-state schedule (measured: a loop that also
        // handles the item's end ran every K/V step slower).
        if (ok) {
          const int j = n1 - 1;
          const int vp = gv + j, sv = vp % SV;
          ok = wait_all(B_VF(sv), (vp / SV) & 1);
          if (ok && j < n0 && (ok = pv(0, sv, j, (base0 + j) & 1))) {
            if (leader) mma_commit(B_O(0));
            __syncwarp();
          }
          if (ok && (ok = pv(1, sv, j, (base1 + j) & 1))) {
            if (leader) {
              mma_commit(B_O(1));
              mma_commit(B_VE(sv));
            }
            __syncwarp();
          }
        }
        gk += n1;
        gv += n1;
        base0 += n0;
        base1 += n1;
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
static bool make_map(CUtensorMap *m, const void *base, int BH, int N, int d, int box_rows = 128) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool CAUSAL, bool F8 = false>
static cudaError_t launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                            const CUtensorMap &mo, float *LSE, int BH, int N, int H, int group,
                            float scale_log2, float out_mul, unsigned *status,
                            cudaStream_t stream) {
  using C = Cfg<D, F8>;
  auto kern = attn_fwd_kernel<D, CAUSAL, F8>;
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
  // Persistent: one CTA per SM (at most one per work item).
  const long long n_items = static_cast<long long>(BH) * n_blk;
  const long long grid = n_items < sm_count() ? n_items : sm_count();
  unsigned *sched = nullptr;
  e = sched_slot(&sched);
  if (e != cudaSuccess) return e;
  // Launched as a programmatic dependent of the previous kernel in the stream
  // (FP8: the V^T pass, which signals once all of its blocks have started):
  // the set-up (barriers, TMEM, descriptor prefetch) overlaps that kernel's
  // end, and the loads wait for it (griddepcontrol.wait above).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, LSE, N, BH, n_blk, H, group, scale_log2,
                            out_mul, status, sched);
}

}  // namespace fwd

bool make_bhnd_map(CUtensorMap *m, const void *base, int heads, int rows, int d, int box_rows) {
  return fwd::make_map(m, base, heads, rows, d, box_rows);
}

bool make_bytes_map(CUtensorMap *m, const void *base, int heads, int rows, int cols,
                    int row_stride, int box_cols, int box_rows) {
  auto enc = fwd::encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_stride),
                           static_cast<cuuint64_t>(row_stride) * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Item counters of the persistent kernels, [slot][counter, finished CTAs];
// each launch takes the next slot and leaves it at zero when it completes, so
// launches in flight at the same time on any streams do not share one unless
// kSchedSlots launches were issued in between.  A captured CUDA graph keeps
// the slots of its capture: one graph must not be replayed on two streams at
// once (as with any workspace it holds).
constexpr int kSchedSlots = 65536;
__device__ unsigned g_sched[kSchedSlots][2];

cudaError_t sched_slot(unsigned **out) {
  static std::atomic<unsigned *> base[64] = {};
  static std::atomic<unsigned> next{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  unsigned *b = base[dev].load();
  if (!b) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_sched);
    if (e != cudaSuccess) return e;
    b = static_cast<unsigned *>(p);
    base[dev].store(b);
  }
  *out = b + 2 * (next.fetch_add(1u) % kSchedSlots);
  return cudaSuccess;
}

cudaError_t launch_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                       int H, int H_kv, int N, int d, float scale, int causal, unsigned *status,
                       cudaStream_t stream) {
  using namespace fwd;
  const int BH = B * H;
  const int group = H / H_kv;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, Q, BH, N, d) || !make_map(&mk, K, B * H_kv, N, d) ||
      !make_map(&mv, V, B * H_kv, N, d) || !make_map(&mo, O, BH, N, d))
    return cudaErrorInvalidValue;
  const float sl = scale * 1.44269504088896340736f;
  if (d == 128)
    return causal ? launch_t<128, true>(mq, mk, mv, mo, LSE, BH, N, H, group, sl, 1.f, status, stream)
                  : launch_t<128, false>(mq, mk, mv, mo, LSE, BH, N, H, group, sl, 1.f, status, stream);
  return causal ? launch_t<64, true>(mq, mk, mv, mo, LSE, BH, N, H, group, sl, 1.f, status, stream)
                : launch_t<64, false>(mq, mk, mv, mo, LSE, BH, N, H, group, sl, 1.f, status, stream);
}

cudaError_t launch_fwd_f8_tiles(const void *Q8, const void *K8, const void *VT8, int N_pad,
                                void *O, float *LSE, int B, int H, int N, float scale_log2,
                                float descale_v, int causal, unsigned *status,
                                cudaStream_t stream) {
  using namespace fwd;
  constexpr int D = 128;
  const int BH = B * H;
  CUtensorMap mq, mk, mvt, mo;
  if (!make_bytes_map(&mq, Q8, BH, N, D, D, 128, 128) ||
      !make_bytes_map(&mk, K8, BH, N, D, D, 128, 128) ||
      !make_bytes_map(&mvt, VT8, BH, D, N, N_pad, 128, 128) || !make_map(&mo, O, BH, N, D))
    return cudaErrorInvalidValue;
  // P reaches the P V product scaled by 2^2; the epilogue takes it back out
  // together with V's descale.
  const float out_mul = descale_v / kPScale8;
  return causal ? launch_t<D, true, true>(mq, mk, mvt, mo, LSE, BH, N, H, 1, scale_log2, out_mul,
                                          status, stream)
                : launch_t<D, false, true>(mq, mk, mvt, mo, LSE, BH, N, H, 1, scale_log2, out_mul,
                                           status, stream);
}

}  // namespace ea
