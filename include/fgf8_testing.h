/*
 * fgf8_testing.h -- test hooks of the fgf8 library (not part of the compute
 * path).  Same conventions as fgf8.h.
 */
#ifndef FGF8_TESTING_H
#define FGF8_TESTING_H

#include <stdint.h>

#include "fgf8.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fgf8_selftest_wait_timeout -- launches one warp that allocates tensor
 * memory, waits on a shared-memory barrier that nothing ever arrives on, and
 * gives up after `budget_us` microseconds (1 .. 2,000,000): it records
 * FGF8_ERR_TIMEOUT with site id 99 in the status word of `workspace`
 * (>= 256 bytes, 256-byte aligned, zero-filled), releases its tensor memory
 * and returns.  It exercises the bounded-wait path that every kernel of the
 * library takes when a wait expires, without faulting or hanging the GPU;
 * read the result with fgf8_read_status.  The pages describe no such
 * mechanism; it exists so that failure handling can be tested.
 */
fgf8_status fgf8_selftest_wait_timeout(void *workspace, uint32_t budget_us, void *stream);

/*
 * fgf8_selftest_scaled_div -- for i < n, q_encoder[i] = the binary32 quotient
 * x[i] / s[i] exactly as the quantization kernels compute it (a correctly
 * rounded reciprocal of s and one fused correction step), and q_ieee[i] =
 * CUDA's IEEE round-to-nearest division, so that a test can check that the
 * two agree bit for bit.  Device pointers, float32, n >= 0.
 */
fgf8_status fgf8_selftest_scaled_div(const float *x, const float *s, int64_t n, float *q_encoder,
                                     float *q_ieee, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FGF8_TESTING_H */
