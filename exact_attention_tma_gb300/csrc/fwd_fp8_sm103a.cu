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
