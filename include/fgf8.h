/*
 * fgf8.h -- C ABI of the fine-grained FP8 library for B300 (sm_103a).
 *
 * Fine-grained FP8 quantization and block-scaled FP8 GEMM, after the
 * DeepSeek-V3 FP8 training scheme as described on the pages cited below:
 *   [dssusan]  "dssusan.co.kr Q&A post 93378" -- Figure 7(a) passage (1x128
 *              activation tiles, 128x128 weight blocks), inner-dimension
 *              passage (per-group scales along K; about 14 accumulated bits
 *              on H800), Figure 7(b) passage (FP8 inputs, BF16 or FP32
 *              outputs, promotion of partial sums to FP32), E4M3 passage
 *              (E4M3 on all tensors, FP8 Wgrad, dequantization by scale
 *              multiplication on CUDA cores).
 *   [kailasan] "kailasan.com recruit post 147436" -- hardware-suggestion
 *              passage (at each promotion interval the partial results are
 *              multiplied by the scaling factors and added to FP32).
 *   [why-be]   "why-be.co.kr A/S post 36949" -- FP8-cast-with-TMA and
 *              transposed-read passages (quantization round trip through HBM;
 *              transposed copies for the backward pass).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates nothing and keeps no pointer after the call returns.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  Outputs are valid once the stream reaches
 *     that point.
 *   - Arguments are checked on the host before anything is launched; a
 *     failed check returns an error code and launches nothing.  A launch
 *     failure returns FGF8_ERR_CUDA.
 *   - Matrices are row-major with the stated leading dimension (in
 *     elements).  E4M3 tensors are one byte per element (OCP E4M3 codes).
 *   - Scale tensors are "K-group major": the scales of one K group (or token
 *     group) are contiguous, so that one aligned copy serves a whole tile.
 *     Every scale leading dimension must be a multiple of 4 (16 bytes).
 *   - Outputs must not alias inputs.  Inputs are assumed finite.
 *   - The library runs only on compute capability 10.3 (B300, sm_103a);
 *     other devices get FGF8_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef FGF8_H
#define FGF8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FGF8_OK = 0,
    FGF8_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum, bad stride */
    FGF8_ERR_MISALIGNED = 2,         /* a pointer or row stride breaks the 16-byte rule */
    FGF8_ERR_UNSUPPORTED_SHAPE = 3,  /* e.g. K % 128 != 0, N % 16 != 0 */
    FGF8_ERR_UNSUPPORTED_DEVICE = 4, /* not a compute capability 10.3 device */
    FGF8_ERR_WORKSPACE_TOO_SMALL = 5,
    FGF8_ERR_CUDA = 6,               /* a CUDA runtime/driver call failed */
    FGF8_ERR_TIMEOUT = 7             /* a device-side wait gave up (see fgf8_read_status) */
} fgf8_status;

typedef enum { FGF8_OUT_BF16 = 0, FGF8_OUT_FP32 = 1 } fgf8_out_dtype;

typedef enum {
    /* one scale per 128x128 block of B: sb[kb*ldsb + n/128] ([dssusan] Figure 7(a)) */
    FGF8_BSCALE_BLOCK128 = 0,
    /* one scale per row of B per 128-wide K group: sb[kb*ldsb + n]
     * (B quantized in 128x1 tiles along K, as for the weight-gradient GEMM) */
    FGF8_BSCALE_ROW1x128 = 1
} fgf8_bscale_kind;

/* Human-readable name of a status code (static string). */
const char *fgf8_status_string(fgf8_status st);

/* Library version string (static). */
const char *fgf8_version(void);

/*
 * fp8_quant_act_1x128 -- activation quantization in 1x128 tiles (per token per
 * 128 channels), [dssusan] Figure 7(a) passage, with the optional transposed
 * 128x1 output kept for the weight-gradient GEMM ([dssusan] E4M3 passage, FP8
 * Wgrad; [why-be] transposed-read passage).
 *
 * For each group g of 128 values: amax = max|x|; s = amax / 448 (binary32
 * division); q = E4M3(fl32(x / s)) with round-to-nearest-even and saturation
 * to +-448; an all-zero group gives s = 0 and signed zeros.
 *
 *   x   : BF16 [M][ldx], ldx >= K.  K % 128 == 0.  M >= 0; M == 0 is a no-op
 *         that reads no pointer (they may be NULL).
 *   q   : E4M3 [M][K] (row stride K), groups along K;           may be NULL
 *   s   : float [K/128][lds], s[kb*lds + m]; lds >= M, lds % 4 == 0;  NULL iff q is
 *   qT  : E4M3 [K][M] (row stride M), groups of 128 tokens along M (the last
 *         group may be partial: amax over the tokens present);       may be NULL
 *   sT  : float [ceil(M/128)][ldsT], sT[tb*ldsT + k]; ldsT >= K, ldsT % 4 == 0; NULL iff qT is
 * At least one of q, qT must be given.  x must be 16-byte aligned with
 * ldx % 8 == 0; q, s, qT, sT 16-byte aligned; with qT given, M % 16 == 0.
 */
fgf8_status fp8_quant_act_1x128(const void *x, int64_t M, int64_t K, int64_t ldx,
                                uint8_t *q, float *s, int64_t lds,
                                uint8_t *qT, float *sT, int64_t ldsT,
                                void *stream);

/*
 * fp8_quant_w_128x128 -- weight quantization in 128x128 blocks (per 128 input
 * channels per 128 output channels), [dssusan] Figure 7(a) passage.  Same rule
 * as above with amax over the block; a ragged last block row (N % 128 != 0)
 * takes amax over the rows present.  N == 0 is a no-op that reads no pointer.
 *
 *   w : BF16 [N][ldw], ldw >= K, ldw % 8 == 0, 16-byte aligned.  K % 128 == 0.
 *   q : E4M3 [N][K], 16-byte aligned.
 *   s : float [K/128][lds], s[kb*lds + nb]; lds >= ceil(N/128), lds % 4 == 0.
 */
fgf8_status fp8_quant_w_128x128(const void *w, int64_t N, int64_t K, int64_t ldw,
                                uint8_t *q, float *s, int64_t lds, void *stream);

/*
 * fp8_quant_w_128x128_grouped -- the same 128x128 block quantization for a
 * stack of expert weights (MoE), one launch for all experts, writing the
 * per-expert scale layout that fp8_grouped_gemm_blockscaled reads.
 *
 *   w : BF16 [num_experts][N][ldw] (expert stride N*ldw), ldw >= K, ldw % 8 == 0.
 *   q : E4M3 [num_experts][N][K].
 *   s : float [num_experts][K/128][lds], s[(e*(K/128) + kb)*lds + nb];
 *       lds >= ceil(N/128), lds % 4 == 0.
 *   1 <= num_experts <= 65535 (0 is a no-op).  Alignment as above.
 */
fgf8_status fp8_quant_w_128x128_grouped(const void *w, int32_t num_experts, int64_t N, int64_t K,
                                        int64_t ldw, uint8_t *q, float *s, int64_t lds, void *stream);

/*
 * fp8_quant_w_128x128_t -- the 128x128 block quantization of W written as W^T,
 * the B operand of the data-gradient GEMM dX = dY * W (whose inner dimension
 * is N), for FP8 Dgrad ([dssusan] E4M3 passage: E4M3 on the Dgrad operands;
 * [why-be] transposed-read passage: the backward pass reads transposed
 * copies).  A 128x128 block of W^T holds the elements of one block of W, so
 * its scale and codes equal fp8_quant_w_128x128's, transposed; the forward
 * layout (q, s) may be written in the same pass.
 *
 *   w  : BF16 [N][ldw], ldw >= K, ldw % 8 == 0, 16-byte aligned.
 *        N % 128 == 0 and K % 128 == 0 (the transposed operand's inner
 *        dimension is N); N == 0 is a no-op that reads no pointer.
 *   qT : E4M3 [K][N] (row k holds column k of W), 16-byte aligned.
 *   sT : float [N/128][ldsT], sT[nb*ldsT + kb] = scale of rows nb*128.. and
 *        columns kb*128.. of W; ldsT >= K/128, ldsT % 4 == 0.  This is the sb
 *        of fp8_gemm_blockscaled with B = qT (BLOCK128 kind).
 *   q, s : optional (both NULL or both set), as fp8_quant_w_128x128.
 */
fgf8_status fp8_quant_w_128x128_t(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *qT, float *sT,
                                  int64_t ldsT, uint8_t *q, float *s, int64_t lds, void *stream);

/*
 * fp8_gemm_blockscaled -- C = A_hat * B_hat^T with per-group scales along the
 * inner dimension K ([dssusan] inner-dimension and E4M3 passages).  Each
 * 128-wide K partial product P = sum_{k in group} qa*qb is formed on the
 * tensor cores, multiplied by its scale pair and added into FP32 ([kailasan]
 * hardware-suggestion passage; [dssusan] Figure 7(b) passage):
 *   C[m][n] = sum_kb P_kb[m][n] * sa[kb*ldsa + m] * sb_kb(n)
 * with sb_kb(n) = sb[kb*ldsb + n/128] (BLOCK128) or sb[kb*ldsb + n] (ROW1x128).
 *
 *   A  : E4M3 [M][K] (row stride K), 16-byte aligned.  M >= 1.
 *   sa : float [K/128][ldsa], ldsa >= M, ldsa % 4 == 0.
 *   B  : E4M3 [N][K], 16-byte aligned.  N % 16 == 0.  K % 128 == 0, K >= 128.
 *   sb : float [K/128][ldsb]; ldsb >= ceil(N/128) (BLOCK128) or >= N (ROW1x128);
 *        ldsb % 4 == 0.
 *   C  : [M][ldc] BF16 (cdt = FGF8_OUT_BF16) or FP32 (FGF8_OUT_FP32); ldc >= N,
 *        ldc * element size % 16 == 0, 16-byte aligned.
 *   workspace : device scratch of at least fgf8_gemm_workspace_min_bytes(M, N,
 *        K, 1) bytes (256), 256-byte aligned, ZERO-FILLED before its first
 *        use.  It holds the device status word.  (For small M the K groups of
 *        each 128-row weight tile are split over the CTAs of one thread-block
 *        cluster, which add their FP32 partials in split order through
 *        distributed shared memory: no workspace.)  With
 *        fgf8_gemm_workspace_bytes(M, N, K, 1)
 *        bytes it also holds the last-wave split: when the output tiles leave
 *        the last wave over the SMs partly empty, those tail tiles are cut
 *        along K into pieces that run on the idle SMs, and the last piece of
 *        each adds the FP32 partials in K order.  The result is then the same
 *        sum grouped differently (it can differ from the whole-tile schedule
 *        in the last bits, within the error bound), and it is the same on
 *        every call with the same shape and workspace size.  The kernels leave
 *        the workspace ready for the next call (counters back at zero) unless
 *        a call reports FGF8_ERR_TIMEOUT, after which it must be zero-filled
 *        again.  One workspace must not be used by two calls that can run at
 *        the same time.
 */
fgf8_status fp8_gemm_blockscaled(const uint8_t *A, const float *sa, int64_t ldsa,
                                 const uint8_t *B, const float *sb, int64_t ldsb,
                                 fgf8_bscale_kind bkind,
                                 void *C, int64_t ldc, fgf8_out_dtype cdt,
                                 int64_t M, int64_t N, int64_t K,
                                 void *workspace, size_t ws_bytes, void *stream);

/*
 * fp8_gemm_blockscaled_noalloc -- fp8_gemm_blockscaled for callers that may
 * not allocate device memory: a plugin inside a host framework that owns all
 * GPU memory and forbids allocations from plugins, or a latency-critical loop
 * where an allocation could block or fragment the memory pool.  Such a caller
 * cannot provide the workspace the other GEMM entry points need, so this one
 * uses scratch inside the library instead.  The pages have no counterpart to
 * this entry point; it exists for such callers only.
 *
 * Same arguments, layouts, checks and result as fp8_gemm_blockscaled, minus
 * the workspace.  It allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine): its scratch is a 4 KiB array in device global
 * memory that every device loading the library holds until the process exits.
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress) with the device current; make that first call
 *     before any stream capture on the device.
 *   - The scratch a call needs is that of the schedule it runs on this
 *     device: the 256-byte status header for every shape (the small-M split
 *     reduces within its thread-block cluster), so no valid shape is
 *     rejected for its size.  (FGF8_ERR_WORKSPACE_TOO_SMALL stays the answer
 *     should a schedule ever need more than the array.)  The array never holds
 *     the last-wave split of large GEMMs: whole tiles only.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents; each call clears the part that must start at zero (the device
 *     status word and the arrival counters) on `stream` before its kernel.  Calls whose work can overlap on the GPU (different streams, no
 *     ordering between them) race on the array: order them, or use
 *     fp8_gemm_blockscaled with separate workspaces.
 *   - A device-side wait that expires leaves FGF8_ERR_TIMEOUT in the array's
 *     status word: fgf8_noalloc_read_status reads it back (and clears it);
 *     otherwise the next call clears it.
 */
fgf8_status fp8_gemm_blockscaled_noalloc(const uint8_t *A, const float *sa, int64_t ldsa,
                                         const uint8_t *B, const float *sb, int64_t ldsb,
                                         fgf8_bscale_kind bkind,
                                         void *C, int64_t ldc, fgf8_out_dtype cdt,
                                         int64_t M, int64_t N, int64_t K, void *stream);

/*
 * fgf8_noalloc_read_status -- fgf8_read_status for the scratch of
 * fp8_gemm_blockscaled_noalloc on the current device: synchronizes `stream`,
 * returns the device status (FGF8_OK or FGF8_ERR_TIMEOUT; the site of the
 * first expired wait in *site when site != NULL) and clears it.  No
 * counterpart on the pages.
 */
fgf8_status fgf8_noalloc_read_status(void *stream, int32_t *site);

/*
 * fp8_gemm_bf16a_blockscaled -- the block-scaled GEMM with its token operand
 * given as BF16 and quantized 1x128 inside the GEMM, for decode-sized M:
 * the E4M3 copy of the tokens never goes through HBM ([why-be]
 * FP8-cast-with-TMA passage: the quantization round trip through memory, and
 * the wish to fuse the cast into the load).  The codes and scales are those
 * of fp8_quant_act_1x128 (same rule, same arithmetic), so for M <= 128 the
 * result equals fp8_quant_act_1x128 followed by fp8_gemm_blockscaled bit for
 * bit; for 129 <= M <= 256 fp8_gemm_blockscaled runs large tiles, whose sum is
 * grouped differently (both within the GEMM error bound).
 *
 *   x  : BF16 [M][ldx], ldx >= K, ldx % 8 == 0, 16-byte aligned.  1 <= M <= 256.
 *   B  : E4M3 [N][K] with 128x128 block scales sb [K/128][ldsb] as in
 *        fp8_gemm_blockscaled (BLOCK128 kind).  N % 16 == 0, K % 128 == 0.
 *   C  : [M][ldc] BF16 or FP32, as in fp8_gemm_blockscaled.
 *   workspace : at least fgf8_gemm_workspace_min_bytes(M, N, K, 1) bytes, as in
 *        fp8_gemm_blockscaled.  M == 0 or N == 0 is a no-op.
 */
fgf8_status fp8_gemm_bf16a_blockscaled(const void *x, int64_t ldx, const uint8_t *B, const float *sb, int64_t ldsb,
                                       void *C, int64_t ldc, fgf8_out_dtype cdt, int64_t M, int64_t N, int64_t K,
                                       void *workspace, size_t ws_bytes, void *stream);

/*
 * fp8_grouped_gemm_blockscaled -- MoE expert GEMM in the contiguous layout:
 * the rows of A are grouped by expert, each group padded to a multiple of 128
 * rows, and row m uses expert e = m_indices[m] ([dssusan] scheme applied per
 * expert; the MoE part loads one expert's parameters at a time, [kailasan]
 * micro-batch passage).
 *
 *   A         : E4M3 [M_total][K], M_total % 128 == 0.
 *   sa        : float [K/128][ldsa], ldsa >= M_total, ldsa % 4 == 0.
 *   B         : E4M3 [num_experts][N][K] (expert-major, contiguous).
 *   sb        : float [num_experts][K/128][ldsb], 128x128 block scales per
 *               expert, ldsb >= ceil(N/128), ldsb % 4 == 0.
 *   m_indices : int32 [M_total], expert id per row or -1 for a padding row.
 *               Every 128-row block belongs to one expert: its real rows
 *               come first and carry that expert's id, any padding rows at
 *               the end of the expert's group carry -1.  The expert of a
 *               block is read from its first row; a block whose first row is
 *               -1 is all padding and is skipped.  Rows marked -1 are not
 *               written.
 *   C         : [M_total][ldc], as for fp8_gemm_blockscaled.
 *   workspace : at least fgf8_gemm_workspace_bytes(M_total, N, K, num_experts).
 */
fgf8_status fp8_grouped_gemm_blockscaled(const uint8_t *A, const float *sa, int64_t ldsa,
                                         const uint8_t *B, const float *sb, int64_t ldsb,
                                         const int32_t *m_indices, int32_t num_experts,
                                         void *C, int64_t ldc, fgf8_out_dtype cdt,
                                         int64_t M_total, int64_t N, int64_t K,
                                         void *workspace, size_t ws_bytes, void *stream);

/*
 * fp8_masked_grouped_gemm_blockscaled -- the block-scaled GEMM for decode-time
 * MoE in the masked layout: expert e owns a slot of `cap` token rows of A and
 * of C and its own weight matrix B_e; only its first counts[e] tokens are real.
 * At decode a few hundred tokens at most reach one expert, so the work is
 * bound by reading the expert's weights ([kailasan] decode passage: small
 * per-expert batches, memory access the bottleneck).  For m < counts[e]:
 *   C[e][m][n] = sum_kb P_kb[m][n] * sa[e][kb][m] * sb[e][kb][n/128]
 * with P_kb the 128-wide K partial as in fp8_gemm_blockscaled.  An expert with
 * counts[e] == 0 reads none of its weights.
 *
 *   A  : E4M3 [E][cap][K] (row stride K), 16-byte aligned.  cap % 16 == 0,
 *        16 <= cap <= 256.
 *   sa : float [K/128][ldsa], ldsa >= E*cap, ldsa % 4 == 0: the scales of the
 *        stacked slots, expert e's token m in column e*cap + m -- what
 *        fp8_quant_act_1x128 writes for the [E*cap][K] buffer.
 *   B  : E4M3 [E][N][K], 16-byte aligned.  N % 16 == 0, K % 128 == 0.
 *   sb : float [E][K/128][ldsb], ldsb >= ceil(N/128), ldsb % 4 == 0.
 *   counts : DEVICE int32 [E], 4-byte aligned, read by the kernel (no host
 *        synchronisation); values are clamped to [0, cap].
 *   C  : [E][cap][ldc] BF16 or FP32, ldc >= N, ldc * element size % 16 == 0;
 *        rows m >= counts[e] are not written.
 *   num_experts : 0 .. 65535 (0 is a no-op that reads no pointer).
 *   workspace : at least fgf8_masked_gemm_workspace_bytes(E, cap, N, K) bytes
 *        (256), 256-byte aligned, zero-filled before its first use (the status
 *        word; a split of K is reduced within its thread-block cluster).
 *        Calls sharing a workspace must not overlap on the GPU.
 */
fgf8_status fp8_masked_grouped_gemm_blockscaled(const uint8_t *A, const float *sa, int64_t ldsa, const uint8_t *B,
                                                const float *sb, int64_t ldsb, const int32_t *counts,
                                                int32_t num_experts, int64_t cap, void *C, int64_t ldc,
                                                fgf8_out_dtype cdt, int64_t N, int64_t K, void *workspace,
                                                size_t ws_bytes, void *stream);

/* Workspace bytes fp8_masked_grouped_gemm_blockscaled needs for these sizes. */
size_t fgf8_masked_gemm_workspace_bytes(int32_t num_experts, int64_t cap, int64_t N, int64_t K);

/* Workspace size (bytes) with which the GEMM entry points can use every
 * schedule for this shape (for dense GEMMs, the last-wave split, about
 * 18.5 MiB), and the least they accept (FGF8_ERR_WORKSPACE_TOO_SMALL below it). */
size_t fgf8_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t num_experts);
size_t fgf8_gemm_workspace_min_bytes(int64_t M, int64_t N, int64_t K, int32_t num_experts);

/*
 * fgf8_read_status -- synchronizes `stream`, then returns the device status
 * word held in `workspace` (FGF8_OK, or FGF8_ERR_TIMEOUT if a bounded
 * device-side wait expired) and resets it to FGF8_OK.  `site` (may be NULL)
 * receives the id of the wait that expired (0 if none).
 */
fgf8_status fgf8_read_status(void *workspace, void *stream, int32_t *site);

/*
 * fgf8_mma_probe -- accumulation-precision probe for the tensor cores
 * ([dssusan] inner-dimension passage: about 14 bits kept on H800; "jp-study.kr
 * Q&A post 309256", Hopper fixed-point accumulation passage).  One CTA
 * computes D = A * B^T with E4M3 operands and no scaling, chaining K/32
 * tensor-core MMAs (K = 32 each) into one FP32 accumulator in tensor memory,
 * and writes D without any promotion, so that the caller can compare it with
 * the exact sum.
 *
 *   A : E4M3 [128][K]; B : E4M3 [N][K]; K % 128 == 0, 128 <= K <= 16384;
 *   N % 16 == 0, 16 <= N <= 256.  D : float [128][N].  16-byte aligned.
 *   workspace : >= 256 bytes, zero-filled (status word, as above).
 */
fgf8_status fgf8_mma_probe(const uint8_t *A, const uint8_t *B, float *D,
                           int32_t N, int32_t K, void *workspace, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FGF8_H */
