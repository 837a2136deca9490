/*
 * exact_attn_selftest.h — on-device self-test of the library's failure
 * detection (bounded waits), part of libexact_attn.so.
 *
 * Every mbarrier wait in the attention kernels is bounded: when a wait runs
 * past its limit the kernel records ATTN_ERR_TIMEOUT in the device status word
 * (read and cleared by attn_get_device_status), raises a CTA-local abort flag
 * and exits instead of hanging the GPU.  The pages describe no such mechanism;
 * it exists so that a fault in the pipeline surfaces as an error code.
 */
#ifndef EXACT_ATTN_SELFTEST_H
#define EXACT_ATTN_SELFTEST_H

#include "exact_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_selftest_bounded_wait — launches one warp on `stream` that waits,
 * through the same bounded-wait routine the kernels use, on an mbarrier phase
 * that nothing ever completes.  After limit_ms milliseconds the wait gives up,
 * records ATTN_ERR_TIMEOUT in the device status word and the kernel returns;
 * the CUDA context stays usable.  1 <= limit_ms <= 10000, else ATTN_ERR_ARG.
 * Returns ATTN_OK once launched (asynchronously); read the outcome with
 * attn_get_device_status(stream), which should then report ATTN_ERR_TIMEOUT.
 */
attn_status attn_selftest_bounded_wait(int limit_ms, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTN_SELFTEST_H */
