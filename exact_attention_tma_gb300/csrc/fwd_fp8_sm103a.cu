// fwd_fp8_sm103a.cu — attention forward with FP8 (E4M3) operands on tcgen05.
//
// "Why Fast GPUs Still Wait for Memory" puts the FP8 tensor ceiling at twice
// the bf16 one (its roofline table and the compute-ceiling discussion):
// the same tiled forward with 8-bit Q, K, V and P doubles the rate of both
// products.  Inputs are E4M3 with one descale factor per tensor (the real
// values are code * descale); the scores and the softmax stay in fp32, P is
// rounded to E4M3 for the P V product, O leaves in bf16 and the LSE in fp32.
//
// Two launches:
//   1. a transpose pass writes V^T ([B*H, d, N_pad] bytes) into a workspace,
//      so that both products read K-major operands (kind::f8f6f4 takes
//      8-bit operands K-major only; V^T rows are the head dimension with the
//      keys contiguous);
//   2. the FP8 instance of the two-query-tile forward kernel
//      (fwd_sm103a.cu): Q, K and V^T tiles of 128 x 128 bytes through TMA,
//      S in TMEM, P written as E4M3 (scaled by 2^2, with a lazy-rescale
//      threshold that keeps every P <= 64) over the first columns of its own
//      S region, O += P V with A = P from TMEM and B = the V^T tile.
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"

namespace ea {
namespace f8 {

constexpr int D = 128;                     // head dimension (bytes per row)

// ------------------------------------------------------------ V transpose
// V [BH, N, 128] bytes -> V^T [BH, 128, N_pad] bytes, one 128-key x 128-byte
// block per CTA.  The block is staged in shared memory as 32-bit words, 32
// per key row, with the word column XOR-swizzled by bits of the key (so that
// the column reads below hit 32 distinct banks); each thread then reads 4 x 4
// byte blocks (4 keys x 4 head-dim bytes) as words, transposes them with byte
// permutes, and writes 16 keys of 4 head-dim rows of V^T (8 threads cover
// one 128-byte output row, so the stores are coalesced).
__device__ __forceinline__ int vt_swz(int k) {   // word-column swizzle of key row k (bits 2-4)
  return (((k >> 5) & 3) << 2) | (((k >> 4) & 1) << 4);
}

__global__ void __launch_bounds__(256)
    attn_fp8_vt_kernel(const uint8_t *__restrict__ V, uint8_t *__restrict__ VT, int N, int N_pad) {
  __shared__ uint4 tile[128 * 8];      // [key][8 quads of 4 words], quad index swizzled
  // Every block of this pass is running: the forward kernel launched after it
  // may start (it waits for this pass's results before its first V^T load).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const size_t bh = blockIdx.y;
  const int k0 = blockIdx.x * 128;
  const uint8_t *src = V + (bh * N + k0) * D;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int idx = threadIdx.x + u * 256;           // 1024 chunks of 16 bytes
    const int row = idx >> 3, c = idx & 7;
    uint4 x = make_uint4(0, 0, 0, 0);
    if (k0 + row < N) x = *reinterpret_cast<const uint4 *>(src + row * D + c * 16);
    tile[row * 8 + (c ^ (vt_swz(row) >> 2))] = x;
  }
  __syncthreads();
  const uint32_t *words = reinterpret_cast<const uint32_t *>(tile);
  const int kg = threadIdx.x & 7;      // keys 16 kg .. 16 kg + 15
  const int dg = threadIdx.x >> 3;     // head-dim bytes 4 dg .. 4 dg + 3
  if (k0 + kg * 16 >= N_pad) return;
  uint32_t out[4][4];                  // [head-dim byte j][4-key group g]
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = kg * 16 + g * 4 + i;
      r[i] = words[k * 32 + (dg ^ vt_swz(k))];
    }
    // 4 x 4 byte transpose: out[j][g] byte i = r[i] byte j.
    const uint32_t t0 = __byte_perm(r[0], r[1], 0x5140), t1 = __byte_perm(r[0], r[1], 0x7362);
    const uint32_t t2 = __byte_perm(r[2], r[3], 0x5140), t3 = __byte_perm(r[2], r[3], 0x7362);
    out[0][g] = __byte_perm(t0, t2, 0x5410);
    out[1][g] = __byte_perm(t0, t2, 0x7632);
    out[2][g] = __byte_perm(t1, t3, 0x5410);
    out[3][g] = __byte_perm(t1, t3, 0x7632);
  }
  uint8_t *dst = VT + bh * D * static_cast<size_t>(N_pad) + k0 + kg * 16;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4 *>(dst + static_cast<size_t>(4 * dg + j) * N_pad) =
        make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]);
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
  const float scale_log2 = scale * descale_q * descale_k * 1.44269504088896340736f;
  return launch_fwd_f8_tiles(Q8, K8, ws, N_pad, O, LSE, B, H, N, scale_log2, descale_v, causal,
                             status, stream);
}

}  // namespace ea
