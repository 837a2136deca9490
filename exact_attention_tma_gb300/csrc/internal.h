// internal.h — launchers shared between the C-ABI layer and the kernel files.
#pragma once
#include <atomic>
#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ea {

// Raises `kern`'s dynamic shared-memory limit to `bytes` once per device:
// `done` is the call site's static flag word, one bit per device ordinal.
template <typename Kernel>
inline cudaError_t smem_limit_once(Kernel kern, int bytes, std::atomic<unsigned long long> &done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load() & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit);
  return e;
}

// Streaming multiprocessors of the current device (looked up once per device).
inline int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int n = cache[dev].load();
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 152;
  cache[dev].store(n);
  return n;
}

// Bits of the device status word (see attn_get_device_status).
constexpr unsigned kStatusTimeoutBit = 1u;
constexpr unsigned kStatusBadInputBit = 2u;   // a kernel met an invalid index (a page id)
constexpr unsigned kStatusSetupBit = 4u;      // a kernel could not set up (shared-memory alignment)

// Forward: one launch of the fused tcgen05/TMA kernel; H query heads over
// H_kv K/V heads per batch (H % H_kv == 0; H_kv == H is multi-head).  Arguments
// are already validated by the caller.  Returns cudaSuccess or the
// launch/encode error.
cudaError_t launch_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                       int H, int H_kv, int N, int d, float scale, int causal, unsigned *status,
                       cudaStream_t stream);

// TMA map of a bf16 [heads, rows, d] tensor (d contiguous): boxes of 64
// columns x box_rows rows x 1 head, 128-byte swizzle, rows past `rows` read 0.
bool make_bhnd_map(CUtensorMap *m, const void *base, int heads, int rows, int d, int box_rows);
// TMA map of a byte tensor [heads, rows, cols] with the given row stride
// (bytes, a multiple of 16): boxes of box_cols x box_rows x 1, 128-byte
// swizzle; elements outside the tensor read 0.
bool make_bytes_map(CUtensorMap *m, const void *base, int heads, int rows, int cols,
                    int row_stride, int box_cols, int box_rows);

// FP8 (E4M3) forward, d = 128: V^T into `ws` (fwd_fp8_ws_bytes), then the
// forward kernel; O bf16, LSE fp32.
size_t fwd_fp8_ws_bytes(int B, int H, int N);
cudaError_t launch_fwd_fp8(const void *Q8, const void *K8, const void *V8, void *O, float *LSE,
                           int B, int H, int N, float scale, float descale_q, float descale_k,
                           float descale_v, int causal, void *ws, unsigned *status,
                           cudaStream_t stream);
// The FP8 instance of the two-query-tile forward kernel: E4M3 Q and K
// [B*H, N, 128], V^T [B*H, 128, N_pad] (N_pad a multiple of 16), scale_log2 =
// scale * descale_q * descale_k * log2(e); O bf16, LSE fp32.
cudaError_t launch_fwd_f8_tiles(const void *Q8, const void *K8, const void *VT8, int N_pad,
                                void *O, float *LSE, int B, int H, int N, float scale_log2,
                                float descale_v, int causal, unsigned *status,
                                cudaStream_t stream);

// A zeroed item-counter pair for one launch of a persistent kernel
// ([0] = items claimed, [1] = CTAs finished; the kernel's last CTA zeroes
// both again).  Slots rotate over 65,536 per device.
cudaError_t sched_slot(unsigned **out);

// Device address of the current device's status word (looked up once per device).
cudaError_t device_status_word(unsigned **out);

// attn_decode's host-side argument checks (null, shape, head dimension, scale,
// 16-byte alignment), in that order; returns an attn_status code, 0 if valid.
// Makes no CUDA call.
int check_decode_args(const void *q, const void *K, const void *V, const void *O, int B, int H,
                      int L, int d, float scale);

// Decode: split kernel + combine kernel on `stream`, partials in `ws`.
constexpr int kDecodeSplits = 32;
size_t decode_ws_bytes(int B, int H, int d);
cudaError_t launch_decode(const void *q, const void *Kc, const void *Vc, void *O, int B, int H,
                          int L, int d, float scale, void *ws, cudaStream_t stream);
// Grouped-query decode: H query heads over H_kv K/V heads (H % H_kv == 0);
// same workspace layout as launch_decode (per query head).  `status` is the
// device status word the grouped kernel's bounded waits report into.
cudaError_t launch_decode_gqa(const void *q, const void *Kc, const void *Vc, void *O, int B, int H,
                              int H_kv, int L, int d, float scale, void *ws, unsigned *status,
                              cudaStream_t stream);
// The combine launch of the split-KV decode (one warp per query head):
// partials [BH][nsplit][d] and log-sum-exps [BH][nsplit] (nsplit <= 32).
cudaError_t launch_decode_combine(const float *ws_o, const float *ws_lse, void *O, int BH, int d,
                                  int nsplit, cudaStream_t stream);
// Grouped-query decode on the tensor cores (mma.sync, query heads of a group
// as the M dimension); same workspace layout.
cudaError_t launch_decode_gqa_mma(const void *q, const void *Kc, const void *Vc, void *O, int B,
                                  int H, int H_kv, int L, int d, float scale, void *ws,
                                  unsigned *status, cudaStream_t stream);
// The same kernel on a paged cache (page_size = 2^log2_page >= 16).
cudaError_t launch_decode_paged_mma(const void *q, const void *K_pages, const void *V_pages,
                                    const int *block_table, const int *seq_lens, void *O, int B,
                                    int H, int H_kv, int num_pages, int log2_page, int max_blocks,
                                    int d, float scale, void *ws, unsigned *status,
                                    cudaStream_t stream);

// Backward: row statistics (2 fp32 per padded query row) in `ws`, then the
// dK/dV and dQ kernels, all on `stream`.
size_t bwd_ws_bytes(int B, int H, int N);
cudaError_t launch_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                       const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int H_kv,
                       int N, int d, float scale, int causal, void *ws, unsigned *status,
                       cudaStream_t stream);

// Paged decode (page_size a power of two): same workspace layout.
cudaError_t launch_decode_paged(const void *q, const void *K_pages, const void *V_pages,
                                const int *block_table, const int *seq_lens, void *O, int B, int H,
                                int H_kv, int num_pages, int page_size, int max_blocks, int d,
                                float scale, void *ws, unsigned *status, cudaStream_t stream);

}  // namespace ea
