// selftest.cu — attn_selftest_bounded_wait: exercises the bounded mbarrier wait
// the kernels use, on a barrier phase that is never completed, so that the
// timeout path (status word + clean exit) can be tested without faulting or
// hanging the GPU.
#include "exact_attn_selftest.h"
#include "internal.h"
#include "ptx.cuh"

namespace {

__global__ void selftest_wait_kernel(unsigned *status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ea::mbar_init(ea::smem_u32(&bar), 1);
    abort_flag = 0;
    ea::fence_mbar_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: phase 0 never completes and the wait must
  // give up after limit_ns, raising the timeout bit in the status word.
  (void)ea::mbar_wait_limit(ea::smem_u32(&bar), 0, status, &abort_flag, limit_ns);
}

}  // namespace

extern "C" attn_status attn_selftest_bounded_wait(int limit_ms, cudaStream_t stream) {
  if (limit_ms < 1 || limit_ms > 10000) return ATTN_ERR_ARG;
  unsigned *status = nullptr;
  if (ea::device_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status,
                                             static_cast<unsigned long long>(limit_ms) * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
