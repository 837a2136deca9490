// decode_gqa_mma_sm103a.cu — grouped-query split-KV decode on the tensor cores.
//
// "Why Fast GPUs Still Wait for Memory", section "Attention III · KV cache,
// GQA, MLA": when g = h / h_kv query heads share one K/V head, every K/V byte
// feeds g times the arithmetic (I = 2g / s).  At g = 8 that is eight flops per
// byte, as much as the CUDA cores can sustain next to an HBM-rate stream, so
// this kernel gives the dense part to the tensor cores: the (up to 16) query
// heads of a group that read the same K/V head form the M = 16 rows of
// mma.sync.m16n8k16 products, S = Q_g K_j^T and O += P V_j, with the online
// softmax on the accumulator fragments in between (the FlashAttention tiling of
// the same page, with a 16-row query block).  The kernel still streams every
// K/V byte once ("M4.2 GPU Execution Model for Transformer Kernels", example
// "logical GQA savings require a physical grouped path").
//
// One CTA per (batch, K/V head, chunk of up to 16 query heads, split), the
// keys cut into nsplit chunks of ceil(L / nsplit) (nsplit chosen per shape,
// at most 32; see choose_splits).  Warp 4
// streams 64-key K and V tiles through a two-stage TMA ring (128-byte
// swizzle); warps 0-3 take 16 keys of each tile.  Each warp keeps an online
// softmax state per query head (base 2) and its partial O in registers; the
// four are merged through shared memory into the split's normalised partial
// and log-sum-exp, and the combine kernel of attn_decode finishes the job.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace ea {
namespace decm {

constexpr int kTile = 64;            // keys per K/V tile
constexpr int kStages = 2;
constexpr int kComputeWarps = 4;     // 16 keys of each tile per warp
constexpr int kWarpTMA = kComputeWarps;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr int kRows = 16;            // query heads per CTA (M of the MMAs)

// Splits per (batch, K/V head, head chunk).  The split CTAs of a call run
// best as one resident wave of about 5/3 CTAs per SM at d = 128 (twice as
// many at d = 64, whose CTAs are half the size), each as long as possible.
// Measured on eight shapes (B 1..64, L 2k..64k, g 8 and 16): B16 H64 H_kv8
// L8192 86 us with 2 splits (256 CTAs) against 94 us with 8; B1 L65536 best
// at 32 splits (256 CTAs); B32 L2048 best unsplit (256 CTAs).  When the
// units alone exceed that, one split each while they fit in one wave
// (slots = SMs x resident CTAs per SM), and ~1024 keys per CTA beyond it
// (B64 H64 H_kv8 L4096: 4 splits, 2048 CTAs, 6.5 TB/s against 6.0 unsplit).
static int choose_splits(long long units, int L, int n_sm, int slots, int D) {
  const long long target = (5LL * n_sm * (128 / D)) / 3;
  int s;
  if (units < target) {
    s = static_cast<int>((target + units / 2) / units);   // nearest
  } else if (units <= slots) {
    s = 1;
  } else {
    s = (L + 1023) / 1024;
  }
  s = s < 1 ? 1 : (s > kDecodeSplits ? kDecodeSplits : s);
  while (s > 1 && L / s < kTile) --s;   // at least one whole tile of keys per split
  return s;   // 1 <= s <= kDecodeSplits: the workspace holds kDecodeSplits per head
}

template <int D>
struct Cfg {
  static constexpr int KB = D / 64;                       // 64-column swizzle boxes
  static constexpr uint32_t BOX_BYTES = kTile * 128;      // 64 keys x 64 columns bf16
  static constexpr uint32_t TILE_BYTES = KB * BOX_BYTES;  // one K or V tile
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = kStages * TILE_BYTES;
  static constexpr uint32_t OFF_BAR = 2 * kStages * TILE_BYTES;
  // full[kStages], empty[kStages]
  static constexpr uint32_t OFF_MISC = OFF_BAR + 2 * kStages * 8;   // abort flag
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;
  static constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;
  // After the loop the stages hold the per-warp partials for the merge.
  static constexpr uint32_t MERGE_BYTES = kComputeWarps * kRows * (D + 2) * 4;
  static_assert(MERGE_BYTES <= OFF_BAR, "merge buffer fits in the K/V stages");
};

// Paged caches: K/V pages [num_pages, H_kv, page_size, d] seen by the tensor
// maps as [num_pages * H_kv, page_size, d] (boxes of min(64, page_size) rows);
// key t of sequence b is row t mod page_size of page
// block_table[b][t / page_size]; seq_lens[b] keys are visible.
struct PagedArgs {
  const int *block_table;
  const int *seq_lens;
  int max_blocks, num_pages, log2_page;
};

template <int D, bool PAGED>
__global__ void __launch_bounds__(kThreads)
    attn_decode_gqa_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                               const __grid_constant__ CUtensorMap tmV,
                               const __nv_bfloat16 *__restrict__ q, float *__restrict__ ws_o,
                               float *__restrict__ ws_lse, int H, int H_kv, int L, int chunk,
                               int nsplit, float scale_log2, unsigned *status, PagedArgs pg) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The combine kernel is a programmatic dependent of this grid: it may
  // launch once every CTA has started, and waits for this grid's partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int group = H / H_kv;
  const int n_hc = (group + kRows - 1) / kRows;      // query-head chunks per K/V head
  const int split = blockIdx.x % nsplit;
  int rest = blockIdx.x / nsplit;
  const int hc = rest % n_hc;
  rest /= n_hc;
  const int hk = rest % H_kv;
  const int b = rest / H_kv;
  const int h0 = hk * group + hc * kRows;            // first query head of this CTA
  const int nh = min(kRows, group - hc * kRows);     // query heads of this CTA
  const size_t qh0 = static_cast<size_t>(b) * H + h0;
  const int kv_head = b * H_kv + hk;                 // z coordinate of the K/V maps
  int Lb = L;                                        // keys of this sequence
  if constexpr (PAGED) Lb = min(max(pg.seq_lens[b], 0), pg.max_blocks << pg.log2_page);
  const int lo = split * chunk;                      // a multiple of kTile when PAGED
  const int hi = min(Lb, lo + chunk);
  const int n_tiles = hi > lo ? (hi - lo + kTile - 1) / kTile : 0;
  // Page of key `key` (a valid id, or page 0 for keys past the sequence and
  // for ids outside [0, num_pages), which also raise the bad-input bit when
  // the key is visible).
  auto page_of = [&](int key, bool flag) {
    if (key >= Lb) return 0;
    const int p = pg.block_table[static_cast<size_t>(b) * pg.max_blocks + (key >> pg.log2_page)];
    if (p < 0 || p >= pg.num_pages) {
      if (flag) atomicOr(status, kStatusBadInputBit);
      return 0;
    }
    return p;
  };

  auto B_FULL = [&](int s) { return sb + C::OFF_BAR + 8u * s; };
  auto B_EMPTY = [&](int s) { return sb + C::OFF_BAR + 8u * (kStages + s); };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(B_FULL(s), 1);
      mbar_init(B_EMPTY(s), kComputeWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  int issued = 0;   // tiles the producer started (its copy of the count)
  if (warp == kWarpTMA) {
    // ------------------------------------------------------ TMA producer
    const bool leader = elect_one();
    if (leader) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    for (int t = 0; t < n_tiles; ++t) {
      const int s = t % kStages;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(B_EMPTY(s), ((t / kStages) & 1) ^ 1u, status, abort_flag)))
        break;
      if (leader) {
        mbar_arrive_expect_tx(B_FULL(s), 2 * C::TILE_BYTES);
        if constexpr (PAGED) {
          // 64 / rows sub-boxes of `rows` keys, each inside one page; a sub-box
          // of r rows lands r x 128 bytes into the 128-byte-swizzled box, a
          // multiple of the 1024-byte swizzle atom (rows >= 8).
          const int rows = min(kTile, 1 << pg.log2_page);
          for (int sub = 0; sub < kTile / rows; ++sub) {
            const int key = lo + t * kTile + sub * rows;
            const int z = page_of(key, false) * H_kv + hk;
            const int y = key & ((1 << pg.log2_page) - 1);
#pragma unroll
            for (int kb = 0; kb < C::KB; ++kb) {
              const uint32_t off = s * C::TILE_BYTES + kb * C::BOX_BYTES + sub * rows * 128;
              tma_load_3d(sb + C::OFF_K + off, &tmK, kb * 64, y, z, B_FULL(s));
              tma_load_3d(sb + C::OFF_V + off, &tmV, kb * 64, y, z, B_FULL(s));
            }
          }
        } else {
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb) {
            tma_load_3d(sb + C::OFF_K + s * C::TILE_BYTES + kb * C::BOX_BYTES, &tmK, kb * 64,
                        lo + t * kTile, kv_head, B_FULL(s));
            tma_load_3d(sb + C::OFF_V + s * C::TILE_BYTES + kb * C::BOX_BYTES, &tmV, kb * 64,
                        lo + t * kTile, kv_head, B_FULL(s));
          }
        }
      }
      issued = t + 1;
    }
    __syncwarp();
  }

  // Compute warps: lane l holds query rows g = l / 4 and g + 8 of the 16, and
  // key / head-dim columns 2 t, 2 t + 1 (t = l % 4) of each 8-wide fragment.
  const int g = lane >> 2;
  const int t4 = lane & 3;
  float m[2] = {-INFINITY, -INFINITY};     // running max per row (base 2)
  float l[2] = {0.f, 0.f};                 // this lane's share of the row sums
  float o[D / 8][4];                       // O rows g, g+8 x columns 8 n + 2 t, +1
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  if (warp < kComputeWarps) {
    // Query rows as A fragments, one per 16 columns of the head dimension.
    uint32_t qa[D / 16][4];
    {
      const __nv_bfloat16 *q0 = q + (qh0 + g) * D;
      const __nv_bfloat16 *q1 = q + (qh0 + g + 8) * D;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int c0 = kk * 16 + 2 * t4;
        qa[kk][0] = g < nh ? *reinterpret_cast<const uint32_t *>(q0 + c0) : 0u;
        qa[kk][1] = g + 8 < nh ? *reinterpret_cast<const uint32_t *>(q1 + c0) : 0u;
        qa[kk][2] = g < nh ? *reinterpret_cast<const uint32_t *>(q0 + c0 + 8) : 0u;
        qa[kk][3] = g + 8 < nh ? *reinterpret_cast<const uint32_t *>(q1 + c0 + 8) : 0u;
      }
    }
    const int mi = lane >> 3;              // which 8x8 matrix this lane addresses
    const int ri = lane & 7;               // which row of it
    for (int t = 0; t < n_tiles; ++t) {
      const int s = t % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(B_FULL(s), (t / kStages) & 1, status, abort_flag)))
        break;
      const uint32_t kbase = sb + C::OFF_K + s * C::TILE_BYTES;
      const uint32_t vbase = sb + C::OFF_V + s * C::TILE_BYTES;
      // S (16 rows x this warp's 16 keys) = Q K^T: matrices (key block mi / 2,
      // head-dim half mi % 2) of the K tile's rows warp * 16 + 8 (mi / 2) + ri.
      float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int krow = warp * 16 + (mi >> 1) * 8 + ri;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t chunk16 = static_cast<uint32_t>(((kk & 3) * 2 + (mi & 1)) ^ (krow & 7));
          uint32_t r[4];
          ldmatrix_x4(kbase + (kk >> 2) * C::BOX_BYTES + krow * 128 + (chunk16 << 4), r);
          mma_16816(c[0], qa[kk], r[0], r[1]);
          mma_16816(c[1], qa[kk], r[2], r[3]);
        }
      }
      // Online softmax on the fragments: keys past the split (or the cache)
      // are masked; each row's max over the quad of lanes holding it.
      const int key0 = lo + t * kTile + warp * 16;
      int lim = hi;
      if constexpr (PAGED) {
        // This warp's 16 keys share one page (page_size >= 16): skip them all
        // if its id is invalid (the producer loaded page 0 in its place).
        if (key0 < hi) {
          const int p = pg.block_table[static_cast<size_t>(b) * pg.max_blocks +
                                       (key0 >> pg.log2_page)];
          if (p < 0 || p >= pg.num_pages) {
            if (lane == 0) atomicOr(status, kStatusBadInputBit);
            lim = key0;
          }
        }
      }
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = key0 + 8 * j + 2 * t4 + (e & 1);
          c[j][e] = key < lim ? c[j][e] * scale_log2 : -INFINITY;
          mx[e >> 1] = fmaxf(mx[e >> 1], c[j][e]);
        }
      uint32_t pa[4];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
        const float m_new = fmaxf(m[rr], mx[rr]);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx(m[rr] - m_use);   // 0 while m is -inf
        l[rr] *= alpha;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          o[n][2 * rr] *= alpha;
          o[n][2 * rr + 1] *= alpha;
        }
        float p[2][2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          p[j][0] = ex2_approx(c[j][2 * rr] - m_use);
          p[j][1] = ex2_approx(c[j][2 * rr + 1] - m_use);
          l[rr] += p[j][0] + p[j][1];
        }
        // A fragment of P: rows g (rr = 0) / g + 8 (rr = 1), keys 2t.. of
        // each 8-key block.
        pa[rr] = pack_bf16x2(p[0][0], p[0][1]);
        pa[2 + rr] = pack_bf16x2(p[1][0], p[1][1]);
        m[rr] = m_new;
      }
      // O += P V: matrices (key block mi % 2, head-dim block 2 np + mi / 2) of
      // V rows warp * 16 + 8 (mi % 2) + ri, transposed into B fragments.
      {
        const int vrow = warp * 16 + (mi & 1) * 8 + ri;
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
          const int dblk = 2 * np + (mi >> 1);            // 8-column block of the head dim
          const uint32_t chunk16 = static_cast<uint32_t>((dblk & 7) ^ (vrow & 7));
          uint32_t r[4];
          ldmatrix_x4_trans(vbase + (dblk >> 3) * C::BOX_BYTES + vrow * 128 + (chunk16 << 4), r);
          mma_16816(o[2 * np], pa, r[0], r[1]);
          mma_16816(o[2 * np + 1], pa, r[2], r[3]);
        }
      }
      // The next TMA write into this stage is an async-proxy access: order
      // this warp's generic-proxy reads of it before the release.
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(B_EMPTY(s));
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 1);
      l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 2);
    }
  }
  // Every stage has been read: the stages now hold the per-warp partials.
  __syncthreads();
  if (*abort_flag) {
    // A wait gave up: let the copies the producer started land before the
    // stages are overwritten (the result is void; the status word says so).
    if (warp == kWarpTMA && lane == 0) {
      for (int j = 0; j < kStages && j < issued; ++j) {
        const int tt = issued - 1 - j;
        mbar_wait_drain(B_FULL(tt % kStages), (tt / kStages) & 1, 100000000ull);
      }
    }
    __syncthreads();
  }
  float *sm_o = reinterpret_cast<float *>(smem);                 // [warp][row][D]
  float *sm_m = sm_o + kComputeWarps * kRows * D;                // [warp][row]
  float *sm_l = sm_m + kComputeWarps * kRows;                    // [warp][row]
  if (warp < kComputeWarps) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = g + 8 * rr;
      if (t4 == 0) {
        sm_m[warp * kRows + row] = m[rr];
        sm_l[warp * kRows + row] = l[rr];
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        sm_o[(warp * kRows + row) * D + 8 * n + 2 * t4] = o[n][2 * rr];
        sm_o[(warp * kRows + row) * D + 8 * n + 2 * t4 + 1] = o[n][2 * rr + 1];
      }
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nh * D; idx += kThreads) {
    const int row = idx / D, col = idx % D;
    const size_t part = (qh0 + row) * nsplit + split;
    float mm = sm_m[row];
#pragma unroll
    for (int w = 1; w < kComputeWarps; ++w) mm = fmaxf(mm, sm_m[w * kRows + row]);
    if (mm == -INFINITY) {   // empty split
      ws_o[part * D + col] = 0.f;
      if (col == 0) ws_lse[part] = -INFINITY;
      continue;
    }
    float den = 0.f, num = 0.f;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) {
      const float wt = ex2_approx(sm_m[w * kRows + row] - mm);
      den = fmaf(sm_l[w * kRows + row], wt, den);
      num = fmaf(sm_o[(w * kRows + row) * D + col], wt, num);
    }
    ws_o[part * D + col] = num / den;
    if (col == 0) {
      float lg;
      asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(den));
      ws_lse[part] = mm + lg;   // base-2 log-sum-exp of the split
    }
  }
}

template <int D, bool PAGED>
static cudaError_t launch_t(const void *q, const void *Kc, const void *Vc, void *O, int B, int H,
                            int H_kv, int L, float scale_log2, void *ws, unsigned *status,
                            const PagedArgs &pg, cudaStream_t stream) {
  using C = Cfg<D>;
  CUtensorMap mk, mv;
  if constexpr (PAGED) {
    const int ps = 1 << pg.log2_page;
    const int rows = ps < kTile ? ps : kTile;
    if (!make_bhnd_map(&mk, Kc, pg.num_pages * H_kv, ps, D, rows) ||
        !make_bhnd_map(&mv, Vc, pg.num_pages * H_kv, ps, D, rows))
      return cudaErrorInvalidValue;
  } else {
    if (!make_bhnd_map(&mk, Kc, B * H_kv, L, D, kTile) ||
        !make_bhnd_map(&mv, Vc, B * H_kv, L, D, kTile))
      return cudaErrorInvalidValue;
  }
  auto kern = attn_decode_gqa_mma_kernel<D, PAGED>;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = smem_limit_once(kern, static_cast<int>(C::SMEM_ALLOC), smem_set);
  if (e != cudaSuccess) return e;
  const int BH = B * H;
  const int n_sm = sm_count();
  const int group = H / H_kv;
  const long long units = static_cast<long long>(B) * H_kv * ((group + kRows - 1) / kRows);
  static std::atomic<int> per_sm{0};   // resident CTAs per SM (a property of the kernel)
  int occ = per_sm.load();
  if (occ == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads,
                                                      static_cast<size_t>(C::SMEM_ALLOC));
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    per_sm.store(occ);
  }
  const int nsplit = choose_splits(units, L, n_sm, n_sm * occ, D);
  if (nsplit < 1 || nsplit > kDecodeSplits) return cudaErrorInvalidValue;
  int chunk = (L + nsplit - 1) / nsplit;
  if (PAGED) chunk = (chunk + kTile - 1) / kTile * kTile;   // tiles start on 64-key rows
  float *ws_o = static_cast<float *>(ws);
  float *ws_lse = ws_o + static_cast<size_t>(BH) * nsplit * D;
  const long long grid = units * nsplit;
  kern<<<static_cast<unsigned>(grid), kThreads, C::SMEM_ALLOC, stream>>>(
      mk, mv, static_cast<const __nv_bfloat16 *>(q), ws_o, ws_lse, H, H_kv, L, chunk, nsplit,
      scale_log2, status, pg);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_decode_combine(ws_o, ws_lse, O, BH, D, nsplit, stream);
}

}  // namespace decm

cudaError_t launch_decode_gqa_mma(const void *q, const void *Kc, const void *Vc, void *O, int B,
                                  int H, int H_kv, int L, int d, float scale, void *ws,
                                  unsigned *status, cudaStream_t stream) {
  const float scale_log2 = scale * 1.44269504088896340736f;
  const decm::PagedArgs none{};
  if (d == 128)
    return decm::launch_t<128, false>(q, Kc, Vc, O, B, H, H_kv, L, scale_log2, ws, status, none,
                                      stream);
  return decm::launch_t<64, false>(q, Kc, Vc, O, B, H, H_kv, L, scale_log2, ws, status, none,
                                   stream);
}

cudaError_t launch_decode_paged_mma(const void *q, const void *K_pages, const void *V_pages,
                                    const int *block_table, const int *seq_lens, void *O, int B,
                                    int H, int H_kv, int num_pages, int log2_page, int max_blocks,
                                    int d, float scale, void *ws, unsigned *status,
                                    cudaStream_t stream) {
  const float scale_log2 = scale * 1.44269504088896340736f;
  const decm::PagedArgs pg{block_table, seq_lens, max_blocks, num_pages, log2_page};
  const int L = max_blocks << log2_page;
  if (d == 128)
    return decm::launch_t<128, true>(q, K_pages, V_pages, O, B, H, H_kv, L, scale_log2, ws, status,
                                     pg, stream);
  return decm::launch_t<64, true>(q, K_pages, V_pages, O, B, H, H_kv, L, scale_log2, ws, status,
                                  pg, stream);
}

}  // namespace ea
