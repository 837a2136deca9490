// decode_noalloc.cu — attn_decode_noalloc: split-KV decode whose scratch is a
// fixed device array compiled into the library, for callers that cannot
// allocate device memory.
//
// Who needs it: a process whose memory allocator already owns the GPU's
// memory (for example a serving stack that reserves almost all HBM up front
// and hands out slices itself), code that must not let a library call
// cudaMalloc/cudaFree because those can block or synchronise the device at
// the wrong moment, and host frameworks that forbid plug-ins from allocating
// device memory on their own.  attn_decode allocates its workspace on first
// use, and attn_decode_ws needs the caller to allocate one; this entry point
// needs neither.
//
// The scratch below is one file-scope __device__ array.  Every GPU that loads
// the library holds its own copy for the life of the process.  Host code only
// sees a host-side stand-in under the array's name, so the device address is
// looked up with cudaGetSymbolAddress once per device (with that device
// current) and passed to the kernels.  No call here allocates memory.
#include <mutex>

#include "exact_attn.h"
#include "internal.h"

namespace {

// 16 MiB: enough for B*H*32*(d+1)*4 bytes of partials, i.e. B*H <= 1016 heads
// at d = 128 or B*H <= 2016 at d = 64.
constexpr size_t kNoallocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices];

// Device address of this device's copy of g_decode_scratch (set up once per
// device, with that device current).
attn_status scratch_for_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_decode_noalloc(const void *q, const void *Kcache, const void *Vcache,
                                           void *O, int B, int H, int L, int d, float scale,
                                           cudaStream_t stream) {
  // attn_decode's own checks first, then the size limit, then the one-time
  // symbol lookup: an invalid call gets the same code as from attn_decode and
  // makes no CUDA call.
  const attn_status st0 =
      static_cast<attn_status>(ea::check_decode_args(q, Kcache, Vcache, O, B, H, L, d, scale));
  if (st0 != ATTN_OK) return st0;
  if (attn_decode_workspace_bytes(B, H, L, d) > kNoallocScratchBytes)
    return ATTN_ERR_NOMEM;   // shape beyond the fixed scratch
  void *scratch = nullptr;
  const attn_status st = scratch_for_current_device(&scratch);
  if (st != ATTN_OK) return st;
  // Same kernels as attn_decode_ws, with the fixed array as the workspace.
  // The partials are fully written by the split kernel before the combine
  // kernel reads them, so nothing in the array has to start at zero.
  return attn_decode_ws(q, Kcache, Vcache, O, B, H, L, d, scale, scratch, kNoallocScratchBytes,
                        stream);
}
