/*
 * attn_diag.h -- diagnostic entry points of libattn_gb300.so (test support).
 *
 * These calls exercise pieces of the backward kernel in isolation on the GPU.
 * They are not part of the attention computation and the pages describe no
 * counterpart; they exist so that a layout or descriptor mistake in the
 * tensor-core path can be located without reading compiled code, and so that
 * the device-side timeout path can be tested without hanging a GPU.
 */
#ifndef ATTN_DIAG_GB300_H
#define ATTN_DIAG_GB300_H

#include <stdint.h>

#include "attn_bwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_diag_mma -- one 128-row tile through tcgen05.mma (fp32 accumulation),
 * in one of the three operand forms of the backward kernel.  All pointers are
 * device memory, row-major, dtype fp16 or bf16, head_dim 64 or 128 (= D):
 *   mode 0: c[128][128] = a[128][D] * b[128][D]^T   (both operands K-major, TMA loaded;
 *           the S^T = K Q^T and dP^T = V dO^T form)
 *   mode 1: c[128][D]   = a[128][128] * b[128][D]   (a from tensor memory, b MN-major;
 *           the dV += P^T dO and dK += dS^T Q form)
 *   mode 2: c[128][D]   = a[128][128]^T * b[128][D] (a stored by threads with the 128-byte
 *           swizzle, MN-major; the dQ = dS K form)
 * Asynchronous on stream; check attn_check_device_status afterwards.
 */
int attn_diag_mma(int mode, int dtype, int head_dim, const void* a, const void* b, float* c,
                  attn_stream_t stream);

/*
 * attn_diag_tanh -- y[i] = tanh(x[i]) computed as the logit cap of the
 * kernels does (1 - 2 / (e^{2x} + 1) from the hardware exponential and
 * reciprocal), so its error can be checked against a reference.
 * x, y: device fp32 arrays of n elements.
 */
int attn_diag_tanh(const float* x, float* y, int n, attn_stream_t stream);

/*
 * attn_diag_wait_timeout -- launches a kernel whose only work is a bounded wait
 * on a barrier that nothing completes.  After timeout_ns (1 .. 2e9) the wait
 * gives up, so attn_check_device_status(stream) must then return
 * ATTN_ERR_DEVICE_TIMEOUT and the CUDA context stays usable.
 */
int attn_diag_wait_timeout(int64_t timeout_ns, attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_DIAG_GB300_H */
