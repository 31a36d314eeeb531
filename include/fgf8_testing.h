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

/*
 * fgf8_testing_gemm_schedule -- host only, launches nothing: the schedule that
 * fp8_gemm_blockscaled picks for a dense M x N x K GEMM with B scales of
 * `bkind` (0 block, 1 per row), a workspace of `ws_bytes` and `num_sms` SMs:
 *   schedule[0] = 1 if the small-M kernel runs (the rest is then 0);
 *   schedule[1] = output tile width (128 or 256 columns, 128 rows);
 *   schedule[2] = tiles computed whole (a multiple of min(num_sms, 148) when
 *                 the last wave is split, else all of them);
 *   schedule[3] = K pieces per remaining tile (1 = no split).
 * `schedule` points to 4 host int32.  Lets tests check the schedule choice on
 * a CPU and confirm that a GPU case covers the path it is meant to.
 */
fgf8_status fgf8_testing_gemm_schedule(int64_t M, int64_t N, int64_t K, int32_t bkind, size_t ws_bytes,
                                       int32_t num_sms, int32_t *schedule);

#ifdef __cplusplus
}
#endif

#endif /* FGF8_TESTING_H */
