// quant.cu -- fine-grained E4M3 quantization kernels for sm_103a.
//
// Rule ("dssusan.co.kr Q&A post 93378", Figure 7(a) passage: 1x128 tiles for
// activations, 128x128 blocks for weights, each scaled by its own max-abs):
//   amax = max |x| over the group,  s = amax / 448 (binary32 division),
//   q = E4M3_rn_satfinite(fl32(x / s)),  s == 0 -> q = signed zero.
// Every kernel here is HBM-bound: it reads 2 bytes and writes 1 byte (plus
// 4/128 or 4/16384 bytes of scale) per element, once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "e4m3_rule.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace fgf8 {
namespace {

__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ------------------------------------------------------------------------
// 1x128 tiles along K.  Eight lanes cover one tile (16 BF16 = 32 bytes each),
// so a warp covers four consecutive tiles (1 KB) per load round; kActRounds
// rounds are loaded before any arithmetic so that enough bytes are in flight.
// ------------------------------------------------------------------------
constexpr int kActRounds = 2;
constexpr int kActWarps = 8;

__global__ void __launch_bounds__(kActWarps * 32)
    quant_act_rows_kernel(const __nv_bfloat16 *__restrict__ x, uint32_t M, uint32_t KB, int64_t ldx,
                          uint8_t *__restrict__ q, float *__restrict__ s, int64_t lds)
{
    const uint32_t total = M * KB;               // tiles; < 2^31, checked by the launcher
    const int lane = threadIdx.x & 31;
    const int quad = lane >> 3;                  // which of the warp's four tiles
    const int sub = lane & 7;                    // 16-element slice of the tile
    const uint32_t warp_global = blockIdx.x * kActWarps + (threadIdx.x >> 5);
    const int64_t K = (int64_t)KB * 128;

    uint4 raw[kActRounds][2];
    uint32_t mrow[kActRounds], kblk[kActRounds];
#pragma unroll
    for (int r = 0; r < kActRounds; ++r) {
        const uint32_t t = (warp_global * kActRounds + r) * 4 + quad;
        raw[r][0] = raw[r][1] = make_uint4(0, 0, 0, 0);
        mrow[r] = 0xFFFFFFFFu;
        if (t < total) {
            const uint32_t m = t / KB;
            mrow[r] = m;
            kblk[r] = t - m * KB;
            const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)m * ldx + (int64_t)kblk[r] * 128 + sub * 16);
            raw[r][0] = __ldcs(src);
            raw[r][1] = __ldcs(src + 1);
        }
    }
#pragma unroll
    for (int r = 0; r < kActRounds; ++r) {
        float f[2][8];
        bf16x8_to_f32(raw[r][0], f[0]);
        bf16x8_to_f32(raw[r][1], f[1]);
        float a = fmaxf(amax8(f[0]), amax8(f[1]));
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (mrow[r] != 0xFFFFFFFFu) {
            const float sc = __fdiv_rn(a, kE4M3Max);
            const Divisor dv = make_divisor(sc);
            const uint2 lo = encode8(f[0], dv), hi = encode8(f[1], dv);
            *reinterpret_cast<uint4 *>(q + (int64_t)mrow[r] * K + (int64_t)kblk[r] * 128 + sub * 16) =
                make_uint4(lo.x, lo.y, hi.x, hi.y);
            if (sub == 0) s[(int64_t)kblk[r] * lds + mrow[r]] = sc;
        }
    }
}

// ------------------------------------------------------------------------
// 128 tokens x 128 channels per CTA, held in registers: thread t owns the 8
// channels of 16-byte column chunk c = t % 16 for the 8 consecutive tokens
// 8g .. 8g+7, g = t / 16.  Column (token-direction, 128x1) max-abs: over the
// thread's 8 tokens, across the two half-warps (one shuffle) and across the
// eight warps (shared memory).  Row (1x128) max-abs, when q/s are wanted too:
// over the thread's 8 channels and across its half-warp (four shuffles).  The
// transposed output qT[channel][token] is written as 8-byte token runs.
// M % 16 == 0 when qT is written, so a thread's 8 tokens are all present or
// all absent.
// ------------------------------------------------------------------------
constexpr int kTileThreads = 256;

__global__ void __launch_bounds__(kTileThreads, 4)
    quant_act_tile_kernel(const __nv_bfloat16 *__restrict__ x, int64_t M, int64_t K, int64_t ldx,
                          uint8_t *__restrict__ q, float *__restrict__ s, int64_t lds,
                          uint8_t *__restrict__ qT, float *__restrict__ sT, int64_t ldsT)
{
    // Thread (c16, g) owns channels 8*c16 .. +7 and tokens 8*g .. +7 of the
    // 128 x 128 tile.  A warp covers 8 channel octets x 4 token octets, so a
    // transposed store writes 8 channel rows x 32 contiguous bytes (whole
    // sectors) and a load reads 4 token rows x 128 bytes.
    __shared__ float colmax[4][8 * 16];     // [token block][j * 16 + c16]
    __shared__ float rowmax[2][128];        // [channel half][token]
    const int64_t kb = blockIdx.x;          // channel group
    const int64_t tb = blockIdx.y;          // token group
    const int64_t m0 = tb * 128;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int cb = warp & 1, gb = warp >> 1;
    const int c16 = cb * 8 + (lane & 7);
    const int g = gb * 4 + (lane >> 3);
    const int64_t tok0 = m0 + 8 * g;
    const bool present = tok0 < M;          // all 8 or none (M % 16 == 0)

    uint4 raw[8];                           // [token]: 8 packed BF16 channels
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        raw[i] = make_uint4(0, 0, 0, 0);
        if (present) raw[i] = __ldcs(reinterpret_cast<const uint4 *>(x + (tok0 + i) * ldx + kb * 128 + c16 * 8));
    }

    // --- column groups (128x1): the transposed output
    if (qT != nullptr) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(bf16_lane(raw[i], j)));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
            if (lane < 8) colmax[gb][j * 16 + c16] = a;
        }
    }
    // --- row groups (1x128): this warp's 64 channels, then the partner warp's
    float rmax[8];
    if (q != nullptr) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float f[8];
            bf16x8_to_f32(raw[i], f);
            float a = amax8(f);
#pragma unroll
            for (int o = 4; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            rmax[i] = a;
            if ((lane & 7) == 0) rowmax[cb][8 * g + i] = a;
        }
    }
    __syncthreads();
    if (qT != nullptr) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float a = colmax[0][j * 16 + c16];
#pragma unroll
            for (int w = 1; w < 4; ++w) a = fmaxf(a, colmax[w][j * 16 + c16]);
            const float sc = __fdiv_rn(a, kE4M3Max);
            if (g == 0) sT[tb * ldsT + kb * 128 + c16 * 8 + j] = sc;
            if (present) {
                float col[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) col[i] = bf16_lane(raw[i], j);
                *reinterpret_cast<uint2 *>(qT + (kb * 128 + c16 * 8 + j) * M + tok0) = encode8(col, make_divisor(sc));
            }
        }
    }
    if (q != nullptr) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float a = fmaxf(rmax[i], rowmax[cb ^ 1][8 * g + i]);
            if (present) {
                float f[8];
                bf16x8_to_f32(raw[i], f);
                const float sc = __fdiv_rn(a, kE4M3Max);
                *reinterpret_cast<uint2 *>(q + (tok0 + i) * K + kb * 128 + c16 * 8) = encode8(f, make_divisor(sc));
                if (c16 == 0) s[kb * lds + tok0 + i] = sc;
            }
        }
    }
}

// ------------------------------------------------------------------------
// 128x128 weight blocks: one CTA per block.  The block (32 KB of BF16) is
// staged in shared memory with asynchronous 16-byte copies, so that registers
// do not limit how many blocks an SM keeps in flight; each thread then reads
// back the chunks it copied for the max-abs and again for the encode.
// ------------------------------------------------------------------------
constexpr int kBlockThreads = 256;
constexpr int kBlockChunks = 128 * 16 / kBlockThreads;     // 16-byte chunks per thread

__global__ void __launch_bounds__(kBlockThreads)
    quant_w_block_kernel(const __nv_bfloat16 *__restrict__ w, int64_t N, int64_t K, int64_t ldw,
                         uint8_t *__restrict__ q, float *__restrict__ s, int64_t lds)
{
    __shared__ __align__(16) uint4 tile[128 * 16];
    __shared__ float red[kBlockThreads / 32];
    const int64_t kb = blockIdx.x;
    const int64_t nb = blockIdx.y;
    // blockIdx.z: expert of a stacked [E][N][K] weight; its q and s follow it
    w += (int64_t)blockIdx.z * N * ldw;
    q += (int64_t)blockIdx.z * N * K;
    s += (int64_t)blockIdx.z * (K / 128) * lds;
    const int64_t n0 = nb * 128;
    const int rows = (int)((N - n0) < 128 ? (N - n0) : 128);
    const int tid = threadIdx.x;

#pragma unroll
    for (int i = 0; i < kBlockChunks; ++i) {
        const int c = tid + i * kBlockThreads;
        const int r = c >> 4, c16 = c & 15;
        if (r < rows) cp_async_16(&tile[c], w + (n0 + r) * ldw + kb * 128 + c16 * 8);
        else tile[c] = make_uint4(0, 0, 0, 0);
    }
    cp_async_wait_all();
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < kBlockChunks; ++i) {
        float f[8];
        bf16x8_to_f32(tile[tid + i * kBlockThreads], f);
        a = fmaxf(a, amax8(f));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((tid & 31) == 0) red[tid >> 5] = a;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int i = 1; i < kBlockThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    const float sc = __fdiv_rn(amax, kE4M3Max);
    const Divisor dv = make_divisor(sc);
    if (tid == 0) s[kb * lds + nb] = sc;
#pragma unroll
    for (int i = 0; i < kBlockChunks; ++i) {
        const int c = tid + i * kBlockThreads;
        const int r = c >> 4, c16 = c & 15;
        if (r < rows) {
            float f[8];
            bf16x8_to_f32(tile[c], f);
            *reinterpret_cast<uint2 *>(q + (n0 + r) * K + kb * 128 + c16 * 8) = encode8(f, dv);
        }
    }
}

// ------------------------------------------------------------------------
// 128x128 weight blocks written transposed: W^T, the B operand of the
// data-gradient GEMM dX = dY * W (inner dimension N).  A block of W^T holds the
// elements of one block of W, so scale and codes are those of the forward
// layout, transposed; the forward layout can be written in the same pass.
// Staging as in quant_w_block_kernel; afterwards each thread encodes an 8 x 8
// sub-block, and a warp (8 column octets x 4 row octets) writes 8 rows of W^T
// x 32 contiguous bytes per store.
// ------------------------------------------------------------------------
__global__ void __launch_bounds__(kBlockThreads, 3)
    quant_w_block_t_kernel(const __nv_bfloat16 *__restrict__ w, int64_t N, int64_t K, int64_t ldw,
                           uint8_t *__restrict__ qT, float *__restrict__ sT, int64_t ldsT,
                           uint8_t *__restrict__ q, float *__restrict__ s, int64_t lds)
{
    __shared__ __align__(16) uint4 tile[128 * 16];
    __shared__ float red[kBlockThreads / 32];
    const int64_t kb = blockIdx.x;
    const int64_t nb = blockIdx.y;
    const int64_t n0 = nb * 128;            // N % 128 == 0: every block is full
    const int tid = threadIdx.x;

#pragma unroll
    for (int i = 0; i < kBlockChunks; ++i) {
        const int c = tid + i * kBlockThreads;
        cp_async_16(&tile[c], w + (n0 + (c >> 4)) * ldw + kb * 128 + (c & 15) * 8);
    }
    cp_async_wait_all();
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < kBlockChunks; ++i) {
        float f[8];
        bf16x8_to_f32(tile[tid + i * kBlockThreads], f);
        a = fmaxf(a, amax8(f));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((tid & 31) == 0) red[tid >> 5] = a;
    __syncthreads();                        // also publishes every thread's staged chunks
    float amax = red[0];
#pragma unroll
    for (int i = 1; i < kBlockThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    const float sc = __fdiv_rn(amax, kE4M3Max);
    const Divisor dv = make_divisor(sc);
    if (tid == 0) {
        sT[nb * ldsT + kb] = sc;
        if (s != nullptr) s[kb * lds + nb] = sc;
    }
    const int lane = tid & 31, warp = tid >> 5;
    const int c8 = (warp & 1) * 8 + (lane & 7);     // columns 8*c8 .. +7 of the block (K direction)
    const int r8 = (warp >> 1) * 4 + (lane >> 3);   // rows 8*r8 .. +7 (N direction)
    uint4 raw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) raw[i] = tile[(8 * r8 + i) * 16 + c8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float col[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) col[i] = bf16_lane(raw[i], j);
        *reinterpret_cast<uint2 *>(qT + (kb * 128 + 8 * c8 + j) * N + n0 + 8 * r8) = encode8(col, dv);
    }
    if (q != nullptr) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float f[8];
            bf16x8_to_f32(raw[i], f);
            *reinterpret_cast<uint2 *>(q + (n0 + 8 * r8 + i) * K + kb * 128 + 8 * c8) = encode8(f, dv);
        }
    }
}

// Test hook: the quotient the encoders use next to CUDA's IEEE division.
__global__ void scaled_div_selftest_kernel(const float *__restrict__ x, const float *__restrict__ s, int64_t n,
                                           float *__restrict__ fast, float *__restrict__ ieee)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        fast[i] = scaled(x[i], make_divisor(s[i]));
        ieee[i] = __fdiv_rn(x[i], s[i]);
    }
}

}  // namespace

cudaError_t launch_scaled_div_selftest(const float *x, const float *s, int64_t n, float *fast, float *ieee,
                                       cudaStream_t stream)
{
    if (n <= 0) return cudaSuccess;
    scaled_div_selftest_kernel<<<1184, 256, 0, stream>>>(x, s, n, fast, ieee);
    return cudaGetLastError();
}

cudaError_t launch_quant_act_rows(const void *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, float *s,
                                  int64_t lds, cudaStream_t stream)
{
    const int64_t KB = K / 128;
    const int64_t tiles = M * KB;
    if (tiles >= (int64_t(1) << 31)) return cudaErrorInvalidValue;   // 2^31 tiles = 2^38 elements
    const int64_t per_block = (int64_t)kActWarps * kActRounds * 4;
    const int64_t blocks = (tiles + per_block - 1) / per_block;
    if (blocks == 0) return cudaSuccess;
    quant_act_rows_kernel<<<(unsigned)blocks, kActWarps * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(x), (uint32_t)M, (uint32_t)KB, ldx, q, s, lds);
    return cudaGetLastError();
}

cudaError_t launch_quant_act_tiles(const void *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, float *s,
                                   int64_t lds, uint8_t *qT, float *sT, int64_t ldsT, cudaStream_t stream)
{
    const dim3 grid((unsigned)(K / 128), (unsigned)((M + 127) / 128));
    if (grid.x == 0 || grid.y == 0) return cudaSuccess;
    quant_act_tile_kernel<<<grid, kTileThreads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(x), M, K, ldx, q,
                                                             s, lds, qT, sT, ldsT);
    return cudaGetLastError();
}

cudaError_t launch_quant_w_t(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *qT, float *sT, int64_t ldsT,
                             uint8_t *q, float *s, int64_t lds, cudaStream_t stream)
{
    const dim3 grid((unsigned)(K / 128), (unsigned)(N / 128));
    if (grid.x == 0 || grid.y == 0) return cudaSuccess;
    quant_w_block_t_kernel<<<grid, kBlockThreads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(w), N, K, ldw, qT,
                                                               sT, ldsT, q, s, lds);
    return cudaGetLastError();
}

cudaError_t launch_quant_w(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, float *s, int64_t lds,
                           int32_t num_experts, cudaStream_t stream)
{
    const dim3 grid((unsigned)(K / 128), (unsigned)((N + 127) / 128), (unsigned)num_experts);
    if (grid.x == 0 || grid.y == 0) return cudaSuccess;
    quant_w_block_kernel<<<grid, kBlockThreads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(w), N, K, ldw, q, s,
                                                             lds);
    return cudaGetLastError();
}

}  // namespace fgf8
