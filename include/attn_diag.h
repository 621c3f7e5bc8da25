/*
 * attn_diag.h -- self-test entry points of libattn.so.
 *
 * These calls have no counterpart on the pages: they exercise the hardware
 * building blocks of the attention kernels in isolation so that a wrong
 * descriptor or a lost pipeline signal is reported as such rather than as a
 * wrong attention output.  Same conventions as attn.h (device pointers owned
 * by the caller, asynchronous on `stream`, status codes of attn_status).
 */
#ifndef ATTN_DIAG_H
#define ATTN_DIAG_H

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_diag_mma_tile -- one CTA runs the two tensor-core products of the
 * prefill kernel on a single tile, with the same shared-memory layouts,
 * descriptors and tensor-memory placement:
 *   s_out[128][128] = a[128][D] . b[128][D]^T       (fp32; both K-major)
 *   o_out[128][D]   = bf16(s_out) . v[128][D]         (fp32; P read from
 *                                                     tensor memory, V is the
 *                                                     MN-major operand)
 * a, b, v: bf16 row-major device arrays; D in {64, 128}.
 */
attn_status attn_diag_mma_tile(const void* a, const void* b, const void* v,
                               float* s_out, float* o_out, int D,
                               cudaStream_t stream);

/*
 * attn_diag_wait_timeout -- launch one CTA that waits on a pipeline barrier
 * nobody signals, with a limit of timeout_ns nanoseconds.  The wait must give
 * up, record ATTN_ERR_TIMEOUT in the device status word and return; the
 * following attn_get_device_status(stream) then reports ATTN_ERR_TIMEOUT and
 * the context stays usable.
 */
attn_status attn_diag_wait_timeout(long long timeout_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_DIAG_H */
