// decode_sm103a.cu — split-KV single-token decode for GB300 (sm_103a).
//
// One query row per (batch, head) against a KV cache of L keys, following
// "Why Fast GPUs Still Wait for Memory", section "Attention III · KV cache,
// GQA, MLA": W = 4Ld flops against 2*2*L*d bytes of K and V, an intensity of
// one flop per byte, so the kernel is bound by HBM bandwidth and its job is
// to stream K and V exactly once with as many bytes in flight as possible.
// Parallelism moves from the (collapsed) query axis to KV splits, as the
// prefill/decode example of "M4.2 GPU Execution Model" (operation atlas)
// describes, with the split's partial outputs reduced afterwards (schedule
// table of its section 0x08: "split-K ... partial-output reduction,
// workspace").
//
// Kernel 1 (split): one CTA per (head, split), 4 warps.  Keys are cut into 32
// chunks of ceil(L/32).  Inside a warp, d/8 consecutive lanes own one key row
// (16-byte coalesced loads, lane -> 8 consecutive head-dim elements, as in
// the K[B,H,T,d_h] lane mapping of M4.2's coalescing section); a warp-shuffle
// butterfly finishes each q.k dot product.  Each lane keeps an online-softmax
// state (running max, sum, 8 accumulators) in base 2; the 4 warps x (32 / (d/8))
// lane groups are merged through shared memory into the split's normalised
// partial O_s and its log-sum-exp, written to the fp32 workspace.
// Kernel 2 (combine): one warp per head merges its 32 partials with weights
// 2^(lse_s - max lse) and writes bf16 O.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace ea {
namespace dec {

constexpr int kWarps = 4;
constexpr int kUnroll = 8;   // 16-byte loads of K and of V in flight per lane per batch

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
    attn_decode_split_kernel(const __nv_bfloat16 *__restrict__ q,
                             const __nv_bfloat16 *__restrict__ Kc,
                             const __nv_bfloat16 *__restrict__ Vc, float *__restrict__ ws_o,
                             float *__restrict__ ws_lse, int L, int chunk, int nsplit,
                             float scale_log2) {
  constexpr int LPK = D / 8;          // lanes per key row
  constexpr int KPI = 32 / LPK;       // keys per warp-wide load
  constexpr int G = kWarps * KPI;     // lane groups per CTA
  constexpr int BATCH = kWarps * KPI * kUnroll;
  // The combine kernel is a programmatic dependent of this grid: it may
  // launch once every CTA has started, and waits for this grid's partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // This grid is itself a programmatic dependent of the previous kernel in
  // the stream: wait for it before reading q and the caches.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // 1-D grid: consecutive CTAs read consecutive chunks of one head.
  const int split = blockIdx.x % nsplit;
  const int bh = blockIdx.x / nsplit;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPK;         // which key of the warp-wide load
  const int dl = lane % LPK;          // which 8-element slice of the head dim

  const int lo = split * chunk;
  const int hi = min(L, lo + chunk);

  // q slice for this lane, in fp32.
  float qf[8];
  {
    const uint4 qv = *reinterpret_cast<const uint4 *>(q + static_cast<size_t>(bh) * D + dl * 8);
    const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qf[2 * e] = bf16lo(w[e]);
      qf[2 * e + 1] = bf16hi(w[e]);
    }
  }

  const size_t head_off = static_cast<size_t>(bh) * L * D;
  const __nv_bfloat16 *Kh = Kc + head_off + dl * 8;
  const __nv_bfloat16 *Vh = Vc + head_off + dl * 8;

  float m = -INFINITY, lsum = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;

  for (int base = lo; base < hi; base += BATCH) {
    uint4 kr[kUnroll], vr[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int key = base + (warp * kUnroll + u) * KPI + sub;
      if (key < hi) {
        kr[u] = ld_stream_v4(Kh + static_cast<size_t>(key) * D);
        vr[u] = ld_stream_v4(Vh + static_cast<size_t>(key) * D);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t w[4] = {kr[u].x, kr[u].y, kr[u].z, kr[u].w};
      float part = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        part = fmaf(qf[2 * e], bf16lo(w[e]), part);
        part = fmaf(qf[2 * e + 1], bf16hi(w[e]), part);
      }
#pragma unroll
      for (int off = LPK / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      const int key = base + (warp * kUnroll + u) * KPI + sub;
      x[u] = (key < hi) ? part * scale_log2 : -INFINITY;
    }
    float mb = x[0];
#pragma unroll
    for (int u = 1; u < kUnroll; ++u) mb = fmaxf(mb, x[u]);
    const float m_new = fmaxf(m, mb);
    if (m_new != -INFINITY) {
      const float alpha = ex2_approx(m - m_new);
      lsum *= alpha;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const float p = ex2_approx(x[u] - m_new);
        lsum += p;
        const uint32_t w[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[2 * e] = fmaf(p, bf16lo(w[e]), acc[2 * e]);
          acc[2 * e + 1] = fmaf(p, bf16hi(w[e]), acc[2 * e + 1]);
        }
      }
      m = m_new;
    }
  }

  // Merge the G lane-group states of this CTA.
  __shared__ float sm_m[G], sm_l[G];
  __shared__ float sm_acc[G][D];
  const int g = warp * KPI + sub;
  if (dl == 0) {
    sm_m[g] = m;
    sm_l[g] = lsum;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) sm_acc[g][dl * 8 + e] = acc[e];
  __syncthreads();
  const size_t part = static_cast<size_t>(bh) * nsplit + split;
  for (int t = threadIdx.x; t < D; t += blockDim.x) {
    float mx = sm_m[0];
#pragma unroll
    for (int i = 1; i < G; ++i) mx = fmaxf(mx, sm_m[i]);
    if (mx == -INFINITY) {   // empty split
      ws_o[part * D + t] = 0.f;
      if (t == 0) ws_lse[part] = -INFINITY;
      continue;
    }
    float den = 0.f, num = 0.f;
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const float w = ex2_approx(sm_m[i] - mx);
      den = fmaf(sm_l[i], w, den);
      num = fmaf(sm_acc[i][t], w, num);
    }
    ws_o[part * D + t] = num / den;
    if (t == 0) {
      float lg;
      asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(den));
      ws_lse[part] = mx + lg;   // base-2 log-sum-exp of the split
    }
  }
}

// One warp per head: lane s holds split s's log-sum-exp (nsplit <= 32).
template <int D>
__global__ void __launch_bounds__(128)
    attn_decode_combine_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_lse,
                               __nv_bfloat16 *__restrict__ O, int BH, int nsplit) {
  const int head = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  // The next kernel in the stream may launch now (it waits for this grid
  // before reading anything this grid writes).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Launched as a programmatic dependent of the split kernel: wait for its
  // partials (a no-op when the previous launch did not allow it to start early).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (head >= BH) return;
  const float lse = (lane < nsplit) ? ws_lse[static_cast<size_t>(head) * nsplit + lane] : -INFINITY;
  float mx = lse;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const float w = (lse == -INFINITY) ? 0.f : ex2_approx(lse - mx);
  float wsum = w;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  constexpr int E = D / 32;   // head-dim elements per lane
  float o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;
  const float *base = ws_o + static_cast<size_t>(head) * nsplit * D + lane * E;
  for (int s = 0; s < nsplit; ++s) {
    const float ws = __shfl_sync(0xffffffffu, w, s);
    if constexpr (E == 4) {
      const float4 v = *reinterpret_cast<const float4 *>(base + static_cast<size_t>(s) * D);
      o[0] = fmaf(ws, v.x, o[0]);
      o[1] = fmaf(ws, v.y, o[1]);
      o[2] = fmaf(ws, v.z, o[2]);
      o[3] = fmaf(ws, v.w, o[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2 *>(base + static_cast<size_t>(s) * D);
      o[0] = fmaf(ws, v.x, o[0]);
      o[1] = fmaf(ws, v.y, o[1]);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;   // a sequence with no tokens gives O = 0
  __nv_bfloat16 *out = O + static_cast<size_t>(head) * D + lane * E;
  if constexpr (E == 4) {
    const uint32_t a = pack_bf16x2(o[0] * inv, o[1] * inv);
    const uint32_t b = pack_bf16x2(o[2] * inv, o[3] * inv);
    *reinterpret_cast<uint2 *>(out) = make_uint2(a, b);
  } else {
    *reinterpret_cast<uint32_t *>(out) = pack_bf16x2(o[0] * inv, o[1] * inv);
  }
}

// Grouped-query split kernel ("Why Fast GPUs Still Wait for Memory", Attention
// III: g = h / h_kv query heads share one K/V head, so the same K/V bytes feed
// g times the arithmetic; "M4.2 GPU Execution Model", example "logical GQA
// savings require a physical grouped path": map the group's query heads to one
// shared K/V load instead of expanding the cache).  One CTA per (batch, K/V
// head, chunk of GQ query heads of its group, split): every K/V row is loaded
// once and combined in registers with the GQ query vectors (query head
// h0 + i of the CTA's chunk).  Lane mapping, online softmax and the merge are
// those of attn_decode_split_kernel, per query head; the partials go to the
// same per-query-head workspace slots, so the combine kernel is shared.
// Paged caches ("M4.2 GPU Execution Model for Transformer Kernels", pitfall 16:
// logical K/V continuity does not imply contiguous physical addresses): with
// PAGED, Kc/Vc hold pages [num_pages][H_kv][page_size][D], token t of sequence
// b lives in page block_table[b * max_blocks + t / page_size] at slot
// t % page_size, and the sequence has seq_lens[b] tokens (clamped to
// [0, max_blocks * page_size]).  A page id outside [0, num_pages) is not read:
// its tokens are skipped and kStatusBadInputBit is raised in *status.
struct Paging {
  const int *block_table;
  const int *seq_lens;
  int max_blocks, num_pages, log2_page;
  unsigned *status;
};

// Paged, one query head per K/V head (GQ = 1): 4 keys per lane group per
// batch and at most 72 registers, so that 7 CTAs fit on an SM; with 8 keys
// (94 registers, 5 CTAs) the paged cache streamed 15 % slower than the
// contiguous one although both read the same bytes (fewer warps, fewer bytes
// in flight).
template <int D, int GQ, bool PAGED>
__global__ void __launch_bounds__(kWarps * 32, (PAGED && GQ == 1) ? 7 : 1)
    attn_decode_gqa_split_kernel(const __nv_bfloat16 *__restrict__ q,
                                 const __nv_bfloat16 *__restrict__ Kc,
                                 const __nv_bfloat16 *__restrict__ Vc, float *__restrict__ ws_o,
                                 float *__restrict__ ws_lse, int H, int H_kv, int L, int chunk,
                                 int nsplit, float scale_log2, Paging pg) {
  // Keys per lane group per batch (register budget, and occupancy when paged).
  constexpr int U = (GQ >= 8) ? 4 : (PAGED && GQ == 1) ? 4 : 8;
  constexpr int LPK = D / 8;             // lanes per key row
  constexpr int KPI = 32 / LPK;          // keys per warp-wide load
  constexpr int NG = kWarps * KPI;       // lane groups per CTA
  constexpr int BATCH = NG * U;
  // The combine kernel is a programmatic dependent of this grid: it may
  // launch once every CTA has started, and waits for this grid's partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int group = H / H_kv;
  const int n_hc = group / GQ;           // query-head chunks per K/V head
  const int split = blockIdx.x % nsplit;
  int rest = blockIdx.x / nsplit;
  const int hc = rest % n_hc;
  rest /= n_hc;
  const int hk = rest % H_kv;
  const int b = rest / H_kv;
  const int h0 = hk * group + hc * GQ;   // first query head of this CTA
  const size_t qh0 = static_cast<size_t>(b) * H + h0;   // flat index of that query head
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPK;
  const int dl = lane % LPK;
  if constexpr (PAGED) {   // this sequence's length and split size
    L = min(max(pg.seq_lens[b], 0), pg.max_blocks << pg.log2_page);
    chunk = (L + nsplit - 1) / nsplit;
  }
  const int lo = split * chunk;
  const int hi = min(L, lo + chunk);

  // q slices (pairs of fp32) of the GQ query heads.
  float2 qf[GQ][4];
#pragma unroll
  for (int i = 0; i < GQ; ++i) {
    const uint4 qv = *reinterpret_cast<const uint4 *>(q + (qh0 + i) * D + dl * 8);
    const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) qf[i][e] = make_float2(bf16lo(w[e]), bf16hi(w[e]));
  }
  const size_t kv_off = PAGED ? 0 : (static_cast<size_t>(b) * H_kv + hk) * L * D;
  const __nv_bfloat16 *Kh = Kc + kv_off + dl * 8;
  const __nv_bfloat16 *Vh = Vc + kv_off + dl * 8;
  // Element offset of token `key`'s row (from Kh / Vh), or -1 for a bad page.
  auto row = [&](int key) -> long long {
    if constexpr (PAGED) {
      const int page = __ldg(pg.block_table + static_cast<size_t>(b) * pg.max_blocks +
                             (key >> pg.log2_page));
      if (page < 0 || page >= pg.num_pages) {
        atomicOr(pg.status, kStatusBadInputBit);
        return -1;
      }
      const int slot = key & ((1 << pg.log2_page) - 1);
      return ((static_cast<long long>(page) * H_kv + hk) << pg.log2_page | slot) * D;
    } else {
      return static_cast<long long>(key) * D;
    }
  };

  float m[GQ], lsum[GQ];
  float2 acc[GQ][4];
#pragma unroll
  for (int i = 0; i < GQ; ++i) {
    m[i] = -INFINITY;
    lsum[i] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[i][e] = make_float2(0.f, 0.f);
  }

  for (int base = lo; base < hi; base += BATCH) {
    uint4 kr[U], vr[U];
    bool valid[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = base + (warp * U + u) * KPI + sub;
      const long long off = (key < hi) ? row(key) : -1;
      valid[u] = off >= 0;
      if (valid[u]) {
        kr[u] = ld_stream_v4(Kh + off);
        vr[u] = ld_stream_v4(Vh + off);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int i = 0; i < GQ; ++i) {
      float x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t w[4] = {kr[u].x, kr[u].y, kr[u].z, kr[u].w};
        float2 part = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 4; ++e) part = ffma2(qf[i][e], make_float2(bf16lo(w[e]), bf16hi(w[e])), part);
        float s = part.x + part.y;
#pragma unroll
        for (int off = LPK / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        x[u] = valid[u] ? s * scale_log2 : -INFINITY;
      }
      float mb = x[0];
#pragma unroll
      for (int u = 1; u < U; ++u) mb = fmaxf(mb, x[u]);
      const float m_new = fmaxf(m[i], mb);
      if (m_new != -INFINITY) {
        const float alpha = ex2_approx(m[i] - m_new);
        lsum[i] *= alpha;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] = fmul2(acc[i][e], make_float2(alpha, alpha));
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float p = ex2_approx(x[u] - m_new);
          lsum[i] += p;
          const uint32_t w[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            acc[i][e] = ffma2(make_float2(p, p), make_float2(bf16lo(w[e]), bf16hi(w[e])), acc[i][e]);
        }
        m[i] = m_new;
      }
    }
  }

  // Merge the NG lane-group states of each query head.
  __shared__ float sm_m[GQ][NG], sm_l[GQ][NG];
  __shared__ float sm_acc[GQ][NG][D];
  const int gi = warp * KPI + sub;
#pragma unroll
  for (int i = 0; i < GQ; ++i) {
    if (dl == 0) {
      sm_m[i][gi] = m[i];
      sm_l[i][gi] = lsum[i];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sm_acc[i][gi][dl * 8 + 2 * e] = acc[i][e].x;
      sm_acc[i][gi][dl * 8 + 2 * e + 1] = acc[i][e].y;
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < GQ * D; t += blockDim.x) {
    const int i = t / D, c = t % D;
    const size_t part = (qh0 + i) * nsplit + split;
    float mx = sm_m[i][0];
#pragma unroll
    for (int k = 1; k < NG; ++k) mx = fmaxf(mx, sm_m[i][k]);
    if (mx == -INFINITY) {   // empty split
      ws_o[part * D + c] = 0.f;
      if (c == 0) ws_lse[part] = -INFINITY;
      continue;
    }
    float den = 0.f, num = 0.f;
#pragma unroll
    for (int k = 0; k < NG; ++k) {
      const float w = ex2_approx(sm_m[i][k] - mx);
      den = fmaf(sm_l[i][k], w, den);
      num = fmaf(sm_acc[i][k][c], w, num);
    }
    ws_o[part * D + c] = num / den;
    if (c == 0) {
      float lg;
      asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(den));
      ws_lse[part] = mx + lg;   // base-2 log-sum-exp of the split
    }
  }
}

// Split count for the CUDA-core split kernels: the power of two nearest (in
// ratio) to target / units CTAs per unit, at least 4 and at most
// kDecodeSplits, halved while a split would hold fewer than 64 keys.  The
// targets are measured: the contiguous multi-head kernel runs best with
// ~108 CTAs per SM in flight over the call (B16 H32 L8192: 32 splits; B64
// H32 L2048: 8 splits, 7.09 against 6.64 TB/s with 32), the paged kernel with
// ~13 (B16 H32 L8192, 64-token pages: 4 splits, 5.99 against 5.79 TB/s; B64
// L2048: 5.97 against 4.70; B4: 16 splits, 5.35 against 5.04; measured before
// the paged kernel's occupancy change, after which targets of 26 and 54 gave
// the same or slower times).
static int pow2_splits(long long units, long long target, int L) {
  int s = 1;
  while (s < kDecodeSplits && 1.41421356 * static_cast<double>(units) * s < static_cast<double>(target))
    s *= 2;
  if (s < 4) s = 4;
  while (s > 1 && L / s < 64) s /= 2;
  return s;
}

template <int D, int GQ, bool PAGED>
static cudaError_t launch_gqa_t(const void *q, const void *Kc, const void *Vc, int B, int H, int H_kv,
                                int L, float scale_log2, float *ws_o, float *ws_lse, int nsplit,
                                const Paging &pg, cudaStream_t stream) {
  const int chunk = (L + nsplit - 1) / nsplit;
  const long long grid = static_cast<long long>(B) * H_kv * (H / H_kv / GQ) * nsplit;
  attn_decode_gqa_split_kernel<D, GQ, PAGED>
      <<<static_cast<unsigned>(grid), kWarps * 32, 0, stream>>>(
          static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(Kc),
          static_cast<const __nv_bfloat16 *>(Vc), ws_o, ws_lse, H, H_kv, L, chunk, nsplit,
          scale_log2, pg);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_t(const void *q, const void *Kc, const void *Vc, void *O, int BH, int L,
                            float scale_log2, void *ws, cudaStream_t stream) {
  const int nsplit = pow2_splits(BH, 108LL * sm_count(), L);
  const int chunk = (L + nsplit - 1) / nsplit;
  float *ws_o = static_cast<float *>(ws);
  float *ws_lse = ws_o + static_cast<size_t>(BH) * nsplit * D;
  // A programmatic dependent of the previous kernel in the stream (it waits
  // for that kernel before its first read): the launch overlaps its end.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(BH) * nsplit);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_decode_split_kernel<D>,
                                     static_cast<const __nv_bfloat16 *>(q),
                                     static_cast<const __nv_bfloat16 *>(Kc),
                                     static_cast<const __nv_bfloat16 *>(Vc), ws_o, ws_lse, L, chunk,
                                     nsplit, scale_log2);
  if (e != cudaSuccess) return e;
  return launch_decode_combine(ws_o, ws_lse, O, BH, D, nsplit, stream);
}

}  // namespace dec

cudaError_t launch_decode_combine(const float *ws_o, const float *ws_lse, void *O, int BH, int d,
                                  int nsplit, cudaStream_t stream) {
  // Programmatic dependent launch: the combine grid may be resident before
  // the split grid ends; the kernel waits for it before reading.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((BH + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(O);
  if (d == 128)
    return cudaLaunchKernelEx(&cfg, dec::attn_decode_combine_kernel<128>, ws_o, ws_lse, o, BH, nsplit);
  return cudaLaunchKernelEx(&cfg, dec::attn_decode_combine_kernel<64>, ws_o, ws_lse, o, BH, nsplit);
}

size_t decode_ws_bytes(int B, int H, int d) {
  const size_t parts = static_cast<size_t>(B) * H * kDecodeSplits;
  return parts * static_cast<size_t>(d) * 4 + parts * 4;
}

cudaError_t launch_decode(const void *q, const void *Kc, const void *Vc, void *O, int B, int H,
                          int L, int d, float scale, void *ws, cudaStream_t stream) {
  const float scale_log2 = scale * 1.44269504088896340736f;
  if (d == 128) return dec::launch_t<128>(q, Kc, Vc, O, B * H, L, scale_log2, ws, stream);
  return dec::launch_t<64>(q, Kc, Vc, O, B * H, L, scale_log2, ws, stream);
}

namespace dec {
template <int D, bool PAGED>
static cudaError_t launch_gqa_d(const void *q, const void *Kc, const void *Vc, void *O, int B, int H,
                                int H_kv, int L, float scale_log2, void *ws, const Paging &pg,
                                cudaStream_t stream) {
  const int BH = B * H;
  const int group = H / H_kv;
  const int gq = group % 8 == 0 ? 8 : group % 4 == 0 ? 4 : group % 2 == 0 ? 2 : 1;
  const int nsplit =
      PAGED ? pow2_splits(static_cast<long long>(BH) / gq, 13LL * sm_count(), L) : kDecodeSplits;
  float *ws_o = static_cast<float *>(ws);
  float *ws_lse = ws_o + static_cast<size_t>(BH) * nsplit * D;
  // Query heads per CTA: the largest of 8, 4, 2 dividing the group size.
  cudaError_t e;
  if (group % 8 == 0)
    e = launch_gqa_t<D, 8, PAGED>(q, Kc, Vc, B, H, H_kv, L, scale_log2, ws_o, ws_lse, nsplit, pg,
                                  stream);
  else if (group % 4 == 0)
    e = launch_gqa_t<D, 4, PAGED>(q, Kc, Vc, B, H, H_kv, L, scale_log2, ws_o, ws_lse, nsplit, pg,
                                  stream);
  else if (group % 2 == 0)
    e = launch_gqa_t<D, 2, PAGED>(q, Kc, Vc, B, H, H_kv, L, scale_log2, ws_o, ws_lse, nsplit, pg,
                                  stream);
  else
    e = launch_gqa_t<D, 1, PAGED>(q, Kc, Vc, B, H, H_kv, L, scale_log2, ws_o, ws_lse, nsplit, pg,
                                  stream);
  if (e != cudaSuccess) return e;
  return launch_decode_combine(ws_o, ws_lse, O, BH, D, nsplit, stream);
}
}  // namespace dec

cudaError_t launch_decode_gqa(const void *q, const void *Kc, const void *Vc, void *O, int B, int H,
                              int H_kv, int L, int d, float scale, void *ws, unsigned *status,
                              cudaStream_t stream) {
  if (H_kv == H) return launch_decode(q, Kc, Vc, O, B, H, L, d, scale, ws, stream);
  // Grouped heads: the query group is the M dimension of tensor-core products.
  return launch_decode_gqa_mma(q, Kc, Vc, O, B, H, H_kv, L, d, scale, ws, status, stream);
}

cudaError_t launch_decode_paged(const void *q, const void *K_pages, const void *V_pages,
                                const int *block_table, const int *seq_lens, void *O, int B, int H,
                                int H_kv, int num_pages, int page_size, int max_blocks, int d,
                                float scale, void *ws, unsigned *status, cudaStream_t stream) {
  const float scale_log2 = scale * 1.44269504088896340736f;
  int log2_page = 0;
  while ((1 << log2_page) < page_size) ++log2_page;
  // Grouped heads on pages of at least 16 tokens: the tensor-core kernel.
  if (H_kv < H && page_size >= 16)
    return launch_decode_paged_mma(q, K_pages, V_pages, block_table, seq_lens, O, B, H, H_kv,
                                   num_pages, log2_page, max_blocks, d, scale, ws, status, stream);
  const dec::Paging pg{block_table, seq_lens, max_blocks, num_pages, log2_page, status};
  // L bounds the split size only for the host's grid; each CTA recomputes it
  // from its sequence's length.
  const int L = max_blocks * page_size;
  if (d == 128)
    return dec::launch_gqa_d<128, true>(q, K_pages, V_pages, O, B, H, H_kv, L, scale_log2, ws, pg,
                                        stream);
  return dec::launch_gqa_d<64, true>(q, K_pages, V_pages, O, B, H, H_kv, L, scale_log2, ws, pg,
                                     stream);
}

}  // namespace ea
