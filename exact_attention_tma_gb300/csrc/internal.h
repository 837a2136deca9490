// internal.h — launchers shared between the C-ABI layer and the kernel files.
#pragma once
#include <cstddef>
#include <cuda_runtime.h>

namespace ea {

// Bits of the device status word (see attn_get_device_status).
constexpr unsigned kStatusTimeoutBit = 1u;
constexpr unsigned kStatusBadInputBit = 2u;   // a kernel met an invalid index (a page id)

// Forward: one launch of the fused tcgen05/TMA kernel; H query heads over
// H_kv K/V heads per batch (H % H_kv == 0; H_kv == H is multi-head).  Arguments
// are already validated by the caller.  Returns cudaSuccess or the
// launch/encode error.
cudaError_t launch_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                       int H, int H_kv, int N, int d, float scale, int causal, unsigned *status,
                       cudaStream_t stream);

// Device address of the current device's status word (looked up once per device).
cudaError_t device_status_word(unsigned **out);

// Decode: split kernel + combine kernel on `stream`, partials in `ws`.
constexpr int kDecodeSplits = 32;
size_t decode_ws_bytes(int B, int H, int d);
cudaError_t launch_decode(const void *q, const void *Kc, const void *Vc, void *O, int B, int H,
                          int L, int d, float scale, void *ws, cudaStream_t stream);
// Grouped-query decode: H query heads over H_kv K/V heads (H % H_kv == 0);
// same workspace layout as launch_decode (per query head).
cudaError_t launch_decode_gqa(const void *q, const void *Kc, const void *Vc, void *O, int B, int H,
                              int H_kv, int L, int d, float scale, void *ws, cudaStream_t stream);
// Paged decode (page_size a power of two): same workspace layout.
cudaError_t launch_decode_paged(const void *q, const void *K_pages, const void *V_pages,
                                const int *block_table, const int *seq_lens, void *O, int B, int H,
                                int H_kv, int num_pages, int page_size, int max_blocks, int d,
                                float scale, void *ws, unsigned *status, cudaStream_t stream);

}  // namespace ea
