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
 *   schedule[0] = 1 if the small-M kernel runs (then only schedule[3] is
 *                 set besides);
 *   schedule[1] = output tile width (128 or 256 columns);
 *   schedule[2] = tiles computed whole (a multiple of the number of
 *                 concurrent CTAs, or CTA pairs, when the last wave is
 *                 split, else all of them); with multicast clusters a tile
 *                 is a cluster tile of two 128-row blocks;
 *   schedule[3] = K pieces per remaining tile (1 = no split); for the
 *                 small-M kernel, the CTAs (one cluster) that split the K
 *                 groups of each 128-row weight tile;
 *   schedule[4] = 1 if the CTA-pair kernel runs (256 x 128 tiles on two SMs;
 *                 num_sms / 2 pairs are assumed), 2 if 128 x 256 tiles run
 *                 in clusters of two sharing B by TMA multicast (num_sms / 2
 *                 clusters assumed), 0 for 128-row tiles on single CTAs.
 * `schedule` points to 5 host int32.  Lets tests check the schedule choice on
 * a CPU and confirm that a GPU case covers the path it is meant to.
 */
fgf8_status fgf8_testing_gemm_schedule(int64_t M, int64_t N, int64_t K, int32_t bkind, size_t ws_bytes,
                                       int32_t num_sms, int32_t *schedule);

/*
 * fgf8_testing_set_pair -- 1: from now on, in this process, dense GEMMs with
 * 128x128 block scales and more than 128 rows (and more weight tiles than the
 * small-M kernel takes) run on the CTA-pair kernel: 256 x 128 output tiles on
 * two SMs whose tensor cores work as one (tcgen05 .cta_group::2), four FP32
 * partial buffers per SM, even and odd K groups promoted by different warps.
 * 2: dense GEMMs with 128x128 block scales and more than 128 rows run the
 * 128 x 256 single-SM kernel in clusters of two CTAs on vertically adjacent
 * tiles: each CTA loads its own A panel and half of the B panel they share,
 * multicast into both (cp.async.bulk.tensor .multicast::cluster, this GPU's
 * memory only), and each MMA warp's commit frees the stage in both CTAs.
 * 0: back to the planner's choice (128-row tiles on single SMs, which are
 * faster on the B300).  Returns FGF8_ERR_INVALID_ARG for other values.  Not
 * thread-safe: set it while no other thread calls the library.
 */
fgf8_status fgf8_testing_set_pair(int32_t mode);

/*
 * fgf8_testing_set_small_splits -- 1..8: from now on, in this process, the
 * dense small-M kernel (fp8_gemm_blockscaled with M <= 128 and block scales)
 * splits the K groups of each weight tile over this many CTAs (at most K/128);
 * 0: back to the planner's choice.  Results are the same sum grouped
 * differently (within the GEMM bound).  Returns FGF8_ERR_INVALID_ARG outside
 * 0..8.  Not thread-safe: set it while no other thread calls the library.
 */
fgf8_status fgf8_testing_set_small_splits(int32_t splits);

/*
 * fgf8_testing_pair_clusters -- the number of CTA pairs of the pair GEMM
 * kernel that the current device runs at once (0 if it cannot run it).
 * Calls the CUDA runtime's occupancy query; launches nothing.  Passing twice
 * this number as `num_sms` to fgf8_testing_gemm_schedule gives the schedule
 * the device actually runs.
 */
int32_t fgf8_testing_pair_clusters(void);

/*
 * fgf8_testing_multicast_clusters -- the number of two-CTA clusters of the
 * multicast variant (fgf8_testing_set_pair(2)) that the current device runs
 * at once (0 if it cannot run it); an occupancy query, launches nothing.
 * Twice this number as `num_sms` gives fgf8_testing_gemm_schedule the
 * schedule the device runs in that mode.
 */
int32_t fgf8_testing_multicast_clusters(void);

#ifdef __cplusplus
}
#endif

#endif /* FGF8_TESTING_H */
