// attn_api.cu — the C ABI declared in include/exact_attn.h.
//
// Host-side only: argument validation (nothing is launched for an invalid
// call), the per-device status word that bounded device waits report into,
// the library-owned decode workspace, and dispatch to the kernel launchers.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "exact_attn.h"
#include "internal.h"

namespace {

// Device status word: kernels OR in ea::kStatusTimeoutBit when a bounded wait
// gives up.  One per device (each device gets its own copy of the module).
__device__ unsigned int g_attn_status;

constexpr int kMaxDevices = 64;
constexpr int kMaxLen = 1 << 24;

std::mutex g_mu;
unsigned *g_status_ptr[kMaxDevices];
void *g_ws_ptr[kMaxDevices];
size_t g_ws_bytes[kMaxDevices];
void *g_bws_ptr[kMaxDevices];      // backward row statistics (separate from decode's)
size_t g_bws_bytes[kMaxDevices];
void *g_fws_ptr[kMaxDevices];      // FP8 forward: V^T
size_t g_fws_bytes[kMaxDevices];

// Grow-only library workspace slot of the current device.
attn_status grow_ws(void **slot, size_t *slot_bytes, size_t need, void **out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (*slot_bytes < need) {
    // cudaFree waits for work already using the old buffer.
    if (*slot) cudaFree(*slot);
    *slot = nullptr;
    *slot_bytes = 0;
    if (cudaMalloc(slot, need) != cudaSuccess) {
      *slot = nullptr;
      return ATTN_ERR_NOMEM;
    }
    *slot_bytes = need;
  }
  *out = *slot;
  return ATTN_OK;
}

attn_status current_device(int *dev) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

// Device address of this device's status word (looked up once per device).
attn_status status_ptr(unsigned **out) {
  int dev;
  attn_status st = current_device(&dev);
  if (st != ATTN_OK) return st;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_status) != cudaSuccess || !p) return ATTN_ERR_CUDA;
    g_status_ptr[dev] = static_cast<unsigned *>(p);
  }
  *out = g_status_ptr[dev];
  return ATTN_OK;
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

attn_status check_common(int B, int H, int len, int d, float scale) {
  if (B < 1 || H < 1 || len < 1 || len > kMaxLen) return ATTN_ERR_SHAPE;
  if (static_cast<long long>(B) * H > (1LL << 24)) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_HEADDIM;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_ARG;
  return ATTN_OK;
}

attn_status check_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                      const float *LSE, const void *dQ, const void *dK, const void *dV, int B,
                      int H, int H_kv, int N, int d, float scale, int causal) {
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return ATTN_ERR_NULL;
  attn_status st = check_common(B, H, N, d, scale);
  if (st != ATTN_OK) return st;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_SHAPE;
  if (causal != 0 && causal != 1) return ATTN_ERR_ARG;
  // One CTA per (head, 128-row tile) and one prep warp per padded row must
  // fit 1-D grids.
  const long long tiles = static_cast<long long>(B) * H * ((N + 127) / 128);
  if (tiles >= (1LL << 31) || tiles * 128 / 8 >= (1LL << 31)) return ATTN_ERR_SHAPE;
  if (misaligned(Q) || misaligned(K) || misaligned(V) || misaligned(O) || misaligned(dO) ||
      misaligned(dQ) || misaligned(dK) || misaligned(dV) ||
      (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0)
    return ATTN_ERR_ALIGN;
  return ATTN_OK;
}

attn_status check_decode(const void *q, const void *K, const void *V, const void *O, int B, int H,
                         int L, int d, float scale) {
  if (!q || !K || !V || !O) return ATTN_ERR_NULL;
  attn_status st = check_common(B, H, L, d, scale);
  if (st != ATTN_OK) return st;
  if (misaligned(q) || misaligned(K) || misaligned(V) || misaligned(O)) return ATTN_ERR_ALIGN;
  return ATTN_OK;
}

}  // namespace

cudaError_t ea::device_status_word(unsigned **out) {
  return status_ptr(out) == ATTN_OK ? cudaSuccess : cudaErrorUnknown;
}

int ea::check_decode_args(const void *q, const void *K, const void *V, const void *O, int B, int H,
                          int L, int d, float scale) {
  return static_cast<int>(check_decode(q, K, V, O, B, H, L, d, scale));
}

extern "C" {

attn_status attn_fwd_gqa(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                         int H, int H_kv, int N, int d, float scale, int causal,
                         cudaStream_t stream) {
  if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_NULL;
  attn_status st = check_common(B, H, N, d, scale);
  if (st != ATTN_OK) return st;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_SHAPE;
  if (causal != 0 && causal != 1) return ATTN_ERR_ARG;
  // One CTA per (head, 128-row query tile) must fit a 1-D grid.
  if (static_cast<long long>(B) * H * ((N + 127) / 128) >= (1LL << 31)) return ATTN_ERR_SHAPE;
  if (misaligned(Q) || misaligned(K) || misaligned(V) || misaligned(O) ||
      (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0)
    return ATTN_ERR_ALIGN;
  unsigned *status = nullptr;
  st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  cudaError_t e = ea::launch_fwd(Q, K, V, O, LSE, B, H, H_kv, N, d, scale, causal, status, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                     int H, int N, int d, float scale, int causal, cudaStream_t stream) {
  return attn_fwd_gqa(Q, K, V, O, LSE, B, H, H, N, d, scale, causal, stream);
}

size_t attn_decode_workspace_bytes(int B, int H, int L, int d) {
  if (check_common(B, H, L, d, 1.f) != ATTN_OK) return 0;
  return ea::decode_ws_bytes(B, H, d);
}

attn_status attn_decode_gqa_ws(const void *q, const void *Kcache, const void *Vcache, void *O,
                               int B, int H, int H_kv, int L, int d, float scale, void *ws,
                               size_t ws_bytes, cudaStream_t stream) {
  attn_status st = check_decode(q, Kcache, Vcache, O, B, H, L, d, scale);
  if (st != ATTN_OK) return st;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_SHAPE;
  if (!ws) return ATTN_ERR_NULL;
  if (misaligned(ws)) return ATTN_ERR_ALIGN;
  if (ws_bytes < ea::decode_ws_bytes(B, H, d)) return ATTN_ERR_NOMEM;
  unsigned *status = nullptr;
  st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  cudaError_t e =
      ea::launch_decode_gqa(q, Kcache, Vcache, O, B, H, H_kv, L, d, scale, ws, status, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_decode_ws(const void *q, const void *Kcache, const void *Vcache, void *O, int B,
                           int H, int L, int d, float scale, void *ws, size_t ws_bytes,
                           cudaStream_t stream) {
  return attn_decode_gqa_ws(q, Kcache, Vcache, O, B, H, H, L, d, scale, ws, ws_bytes, stream);
}

attn_status attn_decode_gqa(const void *q, const void *Kcache, const void *Vcache, void *O, int B,
                            int H, int H_kv, int L, int d, float scale, cudaStream_t stream) {
  attn_status st = check_decode(q, Kcache, Vcache, O, B, H, L, d, scale);
  if (st != ATTN_OK) return st;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_SHAPE;
  int dev;
  st = current_device(&dev);
  if (st != ATTN_OK) return st;
  unsigned *status = nullptr;
  st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  const size_t need = ea::decode_ws_bytes(B, H, d);
  void *ws = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_ws_bytes[dev] < need) {
      // Grow-only workspace; cudaFree waits for work already using the old one.
      if (g_ws_ptr[dev]) cudaFree(g_ws_ptr[dev]);
      g_ws_ptr[dev] = nullptr;
      g_ws_bytes[dev] = 0;
      if (cudaMalloc(&g_ws_ptr[dev], need) != cudaSuccess) {
        g_ws_ptr[dev] = nullptr;
        return ATTN_ERR_NOMEM;
      }
      g_ws_bytes[dev] = need;
    }
    ws = g_ws_ptr[dev];
  }
  cudaError_t e =
      ea::launch_decode_gqa(q, Kcache, Vcache, O, B, H, H_kv, L, d, scale, ws, status, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_decode(const void *q, const void *Kcache, const void *Vcache, void *O, int B,
                        int H, int L, int d, float scale, cudaStream_t stream) {
  return attn_decode_gqa(q, Kcache, Vcache, O, B, H, H, L, d, scale, stream);
}

size_t attn_fwd_fp8_workspace_bytes(int B, int H, int N, int d) {
  if (check_common(B, H, N, d, 1.f) != ATTN_OK || d != 128) return 0;
  return ea::fwd_fp8_ws_bytes(B, H, N);
}

namespace {
attn_status check_fp8(const void *Q8, const void *K8, const void *V8, const void *O,
                      const float *LSE, int B, int H, int N, int d, float scale, float descale_q,
                      float descale_k, float descale_v, int causal) {
  if (!Q8 || !K8 || !V8 || !O || !LSE) return ATTN_ERR_NULL;
  attn_status st = check_common(B, H, N, d, scale);
  if (st != ATTN_OK) return st;
  if (d != 128) return ATTN_ERR_HEADDIM;
  for (float f : {descale_q, descale_k, descale_v})
    if (!std::isfinite(f) || !(f > 0.f)) return ATTN_ERR_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_ARG;
  if (static_cast<long long>(B) * H * ((N + 127) / 128) >= (1LL << 31)) return ATTN_ERR_SHAPE;
  if (misaligned(Q8) || misaligned(K8) || misaligned(V8) || misaligned(O) ||
      (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0)
    return ATTN_ERR_ALIGN;
  return ATTN_OK;
}
}  // namespace

attn_status attn_fwd_fp8_ws(const void *Q8, const void *K8, const void *V8, void *O, float *LSE,
                            int B, int H, int N, int d, float scale, float descale_q,
                            float descale_k, float descale_v, int causal, void *ws,
                            size_t ws_bytes, cudaStream_t stream) {
  attn_status st = check_fp8(Q8, K8, V8, O, LSE, B, H, N, d, scale, descale_q, descale_k,
                             descale_v, causal);
  if (st != ATTN_OK) return st;
  if (!ws) return ATTN_ERR_NULL;
  if (misaligned(ws)) return ATTN_ERR_ALIGN;
  if (ws_bytes < ea::fwd_fp8_ws_bytes(B, H, N)) return ATTN_ERR_NOMEM;
  unsigned *status = nullptr;
  st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  cudaError_t e = ea::launch_fwd_fp8(Q8, K8, V8, O, LSE, B, H, N, scale, descale_q, descale_k,
                                     descale_v, causal, ws, status, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_fwd_fp8(const void *Q8, const void *K8, const void *V8, void *O, float *LSE,
                         int B, int H, int N, int d, float scale, float descale_q,
                         float descale_k, float descale_v, int causal, cudaStream_t stream) {
  attn_status st = check_fp8(Q8, K8, V8, O, LSE, B, H, N, d, scale, descale_q, descale_k,
                             descale_v, causal);
  if (st != ATTN_OK) return st;
  int dev;
  st = current_device(&dev);
  if (st != ATTN_OK) return st;
  const size_t need = ea::fwd_fp8_ws_bytes(B, H, N);
  void *ws = nullptr;
  st = grow_ws(&g_fws_ptr[dev], &g_fws_bytes[dev], need, &ws);
  if (st != ATTN_OK) return st;
  return attn_fwd_fp8_ws(Q8, K8, V8, O, LSE, B, H, N, d, scale, descale_q, descale_k, descale_v,
                         causal, ws, need, stream);
}

size_t attn_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_common(B, H, N, d, 1.f) != ATTN_OK) return 0;
  return ea::bwd_ws_bytes(B, H, N);
}

attn_status attn_bwd_gqa_ws(const void *Q, const void *K, const void *V, const void *O,
                            const void *dO, const float *LSE, void *dQ, void *dK, void *dV, int B,
                            int H, int H_kv, int N, int d, float scale, int causal, void *ws,
                            size_t ws_bytes, cudaStream_t stream) {
  attn_status st = check_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, H_kv, N, d, scale, causal);
  if (st != ATTN_OK) return st;
  if (!ws) return ATTN_ERR_NULL;
  if (misaligned(ws)) return ATTN_ERR_ALIGN;
  if (ws_bytes < ea::bwd_ws_bytes(B, H, N)) return ATTN_ERR_NOMEM;
  unsigned *status = nullptr;
  st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  cudaError_t e = ea::launch_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, H_kv, N, d, scale, causal,
                                 ws, status, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_bwd_gqa(const void *Q, const void *K, const void *V, const void *O,
                         const void *dO, const float *LSE, void *dQ, void *dK, void *dV, int B,
                         int H, int H_kv, int N, int d, float scale, int causal,
                         cudaStream_t stream) {
  attn_status st = check_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, H_kv, N, d, scale, causal);
  if (st != ATTN_OK) return st;
  int dev;
  st = current_device(&dev);
  if (st != ATTN_OK) return st;
  void *ws = nullptr;
  st = grow_ws(&g_bws_ptr[dev], &g_bws_bytes[dev], ea::bwd_ws_bytes(B, H, N), &ws);
  if (st != ATTN_OK) return st;
  return attn_bwd_gqa_ws(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, H_kv, N, d, scale, causal, ws,
                         ea::bwd_ws_bytes(B, H, N), stream);
}

attn_status attn_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                     const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int d,
                     float scale, int causal, cudaStream_t stream) {
  return attn_bwd_gqa(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, H, N, d, scale, causal, stream);
}

attn_status attn_decode_paged(const void *q, const void *K_pages, const void *V_pages,
                              const int *block_table, const int *seq_lens, void *O, int B, int H,
                              int H_kv, int num_pages, int page_size, int max_blocks, int d,
                              float scale, cudaStream_t stream) {
  if (!q || !K_pages || !V_pages || !block_table || !seq_lens || !O) return ATTN_ERR_NULL;
  if (num_pages < 1 || max_blocks < 1 || page_size < 1 || page_size > (1 << 16) ||
      (page_size & (page_size - 1)) != 0)
    return ATTN_ERR_SHAPE;
  if (static_cast<long long>(max_blocks) * page_size > kMaxLen) return ATTN_ERR_SHAPE;
  if (static_cast<long long>(num_pages) * (H_kv > 0 ? H_kv : 1) >= (1LL << 31))
    return ATTN_ERR_SHAPE;
  attn_status st = check_common(B, H, max_blocks * page_size, d, scale);
  if (st != ATTN_OK) return st;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_SHAPE;
  if (misaligned(q) || misaligned(K_pages) || misaligned(V_pages) || misaligned(O) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u) != 0)
    return ATTN_ERR_ALIGN;
  unsigned *status = nullptr;
  st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  int dev;
  st = current_device(&dev);
  if (st != ATTN_OK) return st;
  const size_t need = ea::decode_ws_bytes(B, H, d);
  void *ws = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_ws_bytes[dev] < need) {
      // Grow-only workspace; cudaFree waits for work already using the old one.
      if (g_ws_ptr[dev]) cudaFree(g_ws_ptr[dev]);
      g_ws_ptr[dev] = nullptr;
      g_ws_bytes[dev] = 0;
      if (cudaMalloc(&g_ws_ptr[dev], need) != cudaSuccess) {
        g_ws_ptr[dev] = nullptr;
        return ATTN_ERR_NOMEM;
      }
      g_ws_bytes[dev] = need;
    }
    ws = g_ws_ptr[dev];
  }
  cudaError_t e = ea::launch_decode_paged(q, K_pages, V_pages, block_table, seq_lens, O, B, H, H_kv,
                                          num_pages, page_size, max_blocks, d, scale, ws, status,
                                          stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_get_device_status(cudaStream_t stream) {
  unsigned *p = nullptr;
  attn_status st = status_ptr(&p);
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned v = 0;
  const unsigned zero = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (v != 0 && cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (v & ea::kStatusTimeoutBit) return ATTN_ERR_TIMEOUT;
  if (v & ea::kStatusSetupBit) return ATTN_ERR_CUDA;
  return (v & ea::kStatusBadInputBit) ? ATTN_ERR_ARG : ATTN_OK;
}

const char *attn_status_string(attn_status status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "B, H, N or L out of range";
    case ATTN_ERR_HEADDIM: return "head dimension must be 64 or 128";
    case ATTN_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case ATTN_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case ATTN_ERR_NOMEM: return "workspace allocation failed or workspace too small";
    case ATTN_ERR_TIMEOUT: return "a bounded device-side wait expired";
    case ATTN_ERR_ARG: return "invalid argument (scale must be finite and > 0, causal 0 or 1)";
  }
  return "unknown status";
}

int attn_decode_num_splits(void) { return ea::kDecodeSplits; }

}  // extern "C"
