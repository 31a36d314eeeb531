// gemm_pair.cu -- block-scaled FP8 GEMM on CTA pairs (sm_103a, tcgen05
// .cta_group::2), 256 x 128 output tiles, ping-pong promotion.
//
// C[m][n] = sum_kb P_kb[m][n] * sa[kb][m] * sb[kb][n / 128],
// P_kb = sum_{k in kb} qa*qb over one 128-wide K group; every K group's
// partial product leaves the tensor cores, is multiplied by its scale pair
// and added in FP32 ("kailasan.com recruit post 147436", hardware-suggestion
// passage; "dssusan.co.kr Q&A post 93378", inner-dimension and Figure 7(b)
// passages).
//
// What sets the pace here is the hand-off of each K group's partial between
// the tensor core and the CUDA cores, not the tensor core itself: an MMA
// group issued into an idle pipe takes ~250 cycles longer than one queued
// behind another, and every mbarrier test costs ~110 cycles even when the
// phase has completed.  So:
//   - two SMs run their tensor cores as one (M = 256), each holding 128 rows
//     of A and 64 rows of B, and each keeps four 128-column FP32 partial
//     buffers in tensor memory, so the MMA runs up to three K groups ahead of
//     the promotion;
//   - the two promotion warps that share a scheduler take alternate K groups
//     (ping-pong) over all 128 columns of their 32 rows, so each has two MMA
//     periods per group and the fixed latencies of one overlap the FMAs of
//     the other; at the end of a tile the pair swaps halves of its two FP32
//     partial sums through shared memory and each stores 64 columns (even-
//     group sum + odd-group sum, a fixed order);
//   - the scale vectors of 8 K groups travel together, one barrier per 8.
//
// Roles, per CTA (384 threads):
//   - warp 0 (one lane): TMA loads of this CTA's A rows and B rows into a
//     6-stage ring; the bytes of both CTAs are counted on the leader's
//     barrier, which the leader's producer arms with the total;
//   - warps 1 and 3 of the leader (one lane each, even and odd K groups):
//     4 tcgen05.mma.cta_group::2 (K = 32) per K group into a fresh FP32
//     partial, buffers in turn; the commits arrive on both CTAs' barriers;
//   - warp 2: scale vectors (sa of this CTA's 128 rows, the tile's 128x128
//     block scale) of 8 K groups per slot, with cp.async;
//   - warps 4..7 (even K groups) and 8..11 (odd K groups): promotion, one
//     TMEM lane (= output row) per thread: tcgen05.ld, acc += P * s in FP32
//     registers.
// Tiles are walked persistently, tile t on cluster t mod G (n-outer); the
// tiles left over after the whole waves can be cut into K pieces, each
// piece's FP32 partial stored, and the last piece to take a ticket adds them
// in K order (no cluster waits for another).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "kernels.h"
#include "ptx.cuh"

namespace fgf8 {
namespace {

constexpr int kHalfM = 128;             // rows of A per CTA (TMEM lanes)
constexpr int kTileN = 128;             // output columns per pair tile
constexpr int kHalfN = kTileN / 2;      // rows of B per CTA
constexpr int kBK = 128;                // K bytes per group
constexpr int kPairThreads = 384;
constexpr int kStages = 6;
constexpr int kBufs = 4;                // TMEM partial buffers of kTileN columns
constexpr int kGroupsPerSlot = 8;       // K groups of scales per ring slot
constexpr int kSlots = 3;
constexpr int kProducer = 0, kMma = 1, kScale = 2, kMma2 = 3, kEpi0 = 4, kEpiWarps = 8;
constexpr uint32_t kCtrlRegs = 40, kEpiRegs = 232;
static_assert(128 * kCtrlRegs + 256 * kEpiRegs <= kPairThreads * 168, "register split exceeds the launch budget");
static_assert(kBufs * kTileN == 512, "the partial buffers fill tensor memory");
// Arrivals that free a TMEM buffer: every thread of the leader's four
// promotion warps of that group's parity, and one per such warp of the peer
// (a remote arrive).
constexpr uint32_t kTmEmptyCount = 4 * 32 + 4;

enum : int32_t {
    kSiteProducerEmpty = 21,
    kSiteScaleEmpty = 22,
    kSiteMmaTmemEmpty = 23,
    kSiteMmaFull = 24,
    kSiteEpiScale = 25,
    kSiteEpiTmemFull = 26,
};

struct PairParams {
    int64_t M, N, K;
    int32_t KB;
    int32_t num_mp, num_nt, num_tiles;  // 256-row pair blocks, 128-column tiles
    void *C;
    int64_t ldc;
    DeviceStatus *status;
    const float *sa;
    const float *sb;
    int64_t ldsa, ldsb;
    // tail split: tiles [0, dp_tiles) whole; the rest cut into tail_s K
    // pieces, unit v = piece * R + tail tile on cluster v
    int32_t dp_tiles, tail_s, tail_units;
    float *tail_partials;               // [R * tail_s][2 ranks][kTileN / 4][128][4]
    uint32_t *tail_tickets;             // [R][2], zero between calls
};

// Segments (tile, K groups kbeg..kend, piece or -1) of one cluster, in order.
struct PairSegIter {
    int32_t t, v, G;
    __device__ __forceinline__ PairSegIter()
        : t((int32_t)(blockIdx.x >> 1)), v((int32_t)(blockIdx.x >> 1)), G((int32_t)(gridDim.x >> 1))
    {
    }
    __device__ __forceinline__ bool next(const PairParams &p, int32_t &tile, int32_t &k0, int32_t &k1,
                                         int32_t &piece)
    {
        if (t < p.dp_tiles) {
            tile = t;
            k0 = 0;
            k1 = p.KB;
            piece = -1;
            t += G;
            return true;
        }
        if (v >= p.tail_units) return false;
        const int32_t R = p.num_tiles - p.dp_tiles;
        piece = v / R;
        tile = p.dp_tiles + (v - piece * R);
        k0 = piece * p.KB / p.tail_s;
        k1 = (piece + 1) * p.KB / p.tail_s;
        v += G;
        return true;
    }
};

__host__ __device__ constexpr size_t pair_align(size_t v, size_t a)
{
    return (v + a - 1) / a * a;
}

struct PairLayout {
    static constexpr size_t a_bytes = (size_t)kHalfM * kBK;     // 16 KB
    static constexpr size_t b_bytes = (size_t)kHalfN * kBK;     // 8 KB
    static constexpr size_t off_a = 0;
    static constexpr size_t off_b = off_a + kStages * a_bytes;
    // tile-end exchange: per promotion warp, 64 columns x 32 rows of FP32
    static constexpr size_t xch_warp = (size_t)32 * 64 * 4;    // 8 KB
    static constexpr size_t off_xch = off_b + kStages * b_bytes;
    static constexpr size_t off_sa = off_xch + kEpiWarps * xch_warp;
    static constexpr size_t sa_slot = (size_t)kGroupsPerSlot * kHalfM * 4;   // 4 KB
    static constexpr size_t off_sb = off_sa + kSlots * sa_slot;
    static constexpr size_t sb_slot = (size_t)kGroupsPerSlot * 16;             // one 16-byte chunk per group
    static constexpr size_t off_bar = pair_align(off_sb + kSlots * sb_slot, 16);
    static constexpr int num_bars = 2 * kStages + 2 * kSlots + 2 * kBufs + 1;
    static constexpr size_t off_misc = off_bar + (size_t)num_bars * 8;
    static constexpr size_t total = off_misc + 16;
    static constexpr size_t dyn_bytes = total + 1024;
};
static_assert(PairLayout::dyn_bytes <= 227 * 1024, "shared memory");

__device__ __forceinline__ void pair_tile_coords(int32_t tile, const PairParams &p, int32_t &mp, int32_t &nt)
{
    nt = tile / p.num_mp;               // n outer: the waves share B column tiles, A stays in L2
    mp = tile - nt * p.num_mp;
}

__device__ __forceinline__ void store_bf16x8_row(__nv_bfloat16 *dst, float2 a, float2 b, float2 c, float2 d)
{
    uint4 o;
    __nv_bfloat162 h0 = __float22bfloat162_rn(a);
    __nv_bfloat162 h1 = __float22bfloat162_rn(b);
    __nv_bfloat162 h2 = __float22bfloat162_rn(c);
    __nv_bfloat162 h3 = __float22bfloat162_rn(d);
    memcpy(&o.x, &h0, 4);
    memcpy(&o.y, &h1, 4);
    memcpy(&o.z, &h2, 4);
    memcpy(&o.w, &h3, 4);
    *reinterpret_cast<uint4 *>(dst) = o;
}

// Columns [64*H, 64*H + 64) of a 128-column accumulator (float2 pairs) to
// the exchange area, lane-interleaved 16-byte chunks.
template <int H>
__device__ __forceinline__ void xch_write(float4 *dst, const float2 (&acc)[64], uint32_t lane)
{
#pragma unroll
    for (int j = 0; j < 16; ++j)
        dst[j * 32 + lane] = make_float4(acc[H * 32 + 2 * j].x, acc[H * 32 + 2 * j].y, acc[H * 32 + 2 * j + 1].x,
                                         acc[H * 32 + 2 * j + 1].y);
}

template <int H>
__device__ __forceinline__ void xch_add(const float4 *src, float2 (&acc)[64], uint32_t lane)
{
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float4 v = src[j * 32 + lane];
        acc[H * 32 + 2 * j].x += v.x;
        acc[H * 32 + 2 * j].y += v.y;
        acc[H * 32 + 2 * j + 1].x += v.z;
        acc[H * 32 + 2 * j + 1].y += v.w;
    }
}

// Store columns [64*H, 64*H + 64) of the accumulator to row m (n0 = first
// column of the tile); columns past N are not written (N % 16 == 0).
template <int H, bool OUT_F32>
__device__ __forceinline__ void store_half(const PairParams &p, int64_t m, int64_t n0, const float2 (&acc)[64])
{
    const int64_t c0 = n0 + 64 * H;
    if (OUT_F32) {
        float *dst = static_cast<float *>(p.C) + m * p.ldc + c0;
#pragma unroll
        for (int c = 0; c < 64; c += 4)
            if (c0 + c < p.N)
                *reinterpret_cast<float4 *>(dst + c) = make_float4(acc[H * 32 + c / 2].x, acc[H * 32 + c / 2].y,
                                                                   acc[H * 32 + c / 2 + 1].x, acc[H * 32 + c / 2 + 1].y);
    } else {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.C) + m * p.ldc + c0;
#pragma unroll
        for (int c = 0; c < 64; c += 8)
            if (c0 + c < p.N)
                store_bf16x8_row(dst + c, acc[H * 32 + c / 2], acc[H * 32 + c / 2 + 1], acc[H * 32 + c / 2 + 2],
                                 acc[H * 32 + c / 2 + 3]);
    }
}

// FP32 partial of one tail piece: columns [64*H, +64) of row `row`, layout
// [kTileN / 4][128][4].
template <int H>
__device__ __forceinline__ void partial_store(float *part, uint32_t row, const float2 (&acc)[64])
{
#pragma unroll
    for (int c = 0; c < 64; c += 4)
        *reinterpret_cast<float4 *>(part + ((int64_t)((64 * H + c) / 4) * kHalfM + row) * 4) =
            make_float4(acc[H * 32 + c / 2].x, acc[H * 32 + c / 2].y, acc[H * 32 + c / 2 + 1].x,
                        acc[H * 32 + c / 2 + 1].y);
}

template <int H>
__device__ __forceinline__ void partial_accumulate(const float *part, uint32_t row, float2 (&acc)[64], bool first)
{
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(part + ((int64_t)((64 * H + c) / 4) * kHalfM + row) * 4));
        if (first) {
            acc[H * 32 + c / 2] = make_float2(v.x, v.y);
            acc[H * 32 + c / 2 + 1] = make_float2(v.z, v.w);
        } else {
            acc[H * 32 + c / 2].x += v.x;
            acc[H * 32 + c / 2].y += v.y;
            acc[H * 32 + c / 2 + 1].x += v.z;
            acc[H * 32 + c / 2 + 1].y += v.w;
        }
    }
}

// Tile end for the warp that keeps columns [64*H, +64): hand the other half
// of its partial sum to its partner, add the partner's half, then either
// store the 64 columns or (a tail piece) store this piece's FP32 partial and
// take part in the ticket; the last piece adds all pieces in K order and
// stores.  Both warps of a pair and all eight promotion warps pass the same
// named barriers whatever happened before, so a failed wait cannot strand the
// others at a barrier.
template <int H, bool OUT_F32>
__device__ __forceinline__ void tile_end(const PairParams &p, float2 (&acc)[64], float4 *xch_mine,
                                         const float4 *xch_partner, uint32_t quarter, uint32_t lane, uint32_t row,
                                         uint32_t rank, int64_t m, int64_t n0, int32_t tile, int32_t piece, bool &ok,
                                         volatile int *abort_flag, volatile int *tail_last)
{
    xch_write<1 - H>(xch_mine, acc, lane);
    named_barrier_sync(2 + quarter, 64);
    xch_add<H>(xch_partner, acc, lane);
    named_barrier_sync(2 + quarter, 64);
    if (piece >= 0) {
        const int32_t ti = tile - p.dp_tiles;
        const int64_t unit = ((int64_t)ti * p.tail_s + piece) * 2 + rank;
        if (ok) partial_store<H>(p.tail_partials + unit * (kHalfM * kTileN), row, acc);
        __threadfence();
        const bool all_ok = named_barrier_and(1, kEpiWarps * 32, ok && !*abort_flag);
        if (all_ok && threadIdx.x == kEpi0 * 32) {
            const uint32_t ticket = atomicAdd(p.tail_tickets + 2 * ti + rank, 1u);
            const int last = ticket == (uint32_t)(p.tail_s - 1);
            if (last) p.tail_tickets[2 * ti + rank] = 0u;      // ready for the next call
            *tail_last = last;
        }
        named_barrier_sync(1, kEpiWarps * 32);
        if (!all_ok) ok = false;
        if (!all_ok || !*tail_last) return;
        __threadfence();
        for (int32_t q = 0; q < p.tail_s; ++q)
            partial_accumulate<H>(p.tail_partials + (((int64_t)ti * p.tail_s + q) * 2 + rank) * (kHalfM * kTileN),
                                  row, acc, q == 0);
    } else if (!ok) {
        return;
    }
    if (m < p.M) store_half<H, OUT_F32>(p, m, n0, acc);
}

template <bool OUT_F32>
__global__ void __launch_bounds__(kPairThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const PairParams p)
{
    using L = PairLayout;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(pair_align(reinterpret_cast<uintptr_t>(smem_raw), 1024));
    uint8_t *sm_a = smem + L::off_a;
    uint8_t *sm_b = smem + L::off_b;
    float *sm_sa = reinterpret_cast<float *>(smem + L::off_sa);
    float *sm_sb = reinterpret_cast<float *>(smem + L::off_sb);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::off_bar);
    uint64_t *full = bars;                       // leader: both CTAs' stage bytes
    uint64_t *empty = bars + kStages;            // each CTA: its stage may be refilled
    uint64_t *sc_full = bars + 2 * kStages;
    uint64_t *sc_empty = bars + 2 * kStages + kSlots;
    uint64_t *tm_full = bars + 2 * kStages + 2 * kSlots;   // each CTA: partial in its TMEM
    uint64_t *tm_empty = tm_full + kBufs;                   // leader: both CTAs done with a buffer
    uint64_t *drain = tm_full + 2 * kBufs;
    uint32_t *tmem_base_slot = reinterpret_cast<uint32_t *>(smem + L::off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::off_misc + 4);
    volatile int *tail_last = reinterpret_cast<volatile int *>(smem + L::off_misc + 8);

    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();
    const uint32_t rank = cluster_ctarank();     // 0: leader

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&sc_full[i], 32);          // one cp.async arrival per scale-warp lane
            mbar_init(&sc_empty[i], kEpiWarps);
        }
        for (int i = 0; i < kBufs; ++i) {
            mbar_init(&tm_full[i], 1);
            mbar_init(&tm_empty[i], kTmEmptyCount);
        }
        mbar_init(drain, 2);                     // one commit per MMA issuer
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMma) tmem_alloc_pair(tmem_base_slot, 512);
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();                              // the peer may now signal the leader's barriers
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_base_slot;

    if (warp < kEpi0) regs_decrease<kCtrlRegs>();

    if (warp == kProducer) {
        if (elect_one()) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            uint32_t it = 0;
            bool ok = true;
            PairSegIter si;
            int32_t tile, kbeg, kend, piece;
            while (ok && si.next(p, tile, kbeg, kend, piece)) {
                int32_t mp, nt;
                pair_tile_coords(tile, p, mp, nt);
                const int32_t a_row = mp * 2 * kHalfM + (int32_t)rank * kHalfM;
                const int32_t b_row = nt * kTileN + (int32_t)rank * kHalfN;
                for (int32_t kb = kbeg; kb < kend; ++kb, ++it) {
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1;
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag)) {
                        record_timeout(p.status, kSiteProducerEmpty);
                        ok = false;
                        break;
                    }
                    if (rank == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * (L::a_bytes + L::b_bytes)));
                    const uint32_t full_leader = cluster_map(&full[s], 0);
                    tma_load_2d_pair(sm_a + s * L::a_bytes, &tmA, full_leader, kb * kBK, a_row);
                    tma_load_2d_pair(sm_b + s * L::b_bytes, &tmB, full_leader, kb * kBK, b_row);
                }
            }
            if (!ok) *abort_flag = 1;
        }
        __syncwarp();
    } else if (warp == kScale) {
        // sa of this CTA's 128 rows and the 16-byte chunk holding the tile's
        // block scale, up to 8 K groups per slot (every segment starts a new
        // slot), copied with cp.async by the whole warp; past the end of a
        // scale row nothing is read (zero fill).
        uint32_t nslot = 0;
        bool ok = true;
        PairSegIter si;
        int32_t tile, kbeg, kend, piece;
        while (ok && si.next(p, tile, kbeg, kend, piece)) {
            int32_t mp, nt;
            pair_tile_coords(tile, p, mp, nt);
            const int64_t sa_x = (int64_t)mp * 2 * kHalfM + rank * kHalfM + 4 * lane;
            const int64_t sb_x = (int64_t)nt & ~3ll;
            for (int32_t kb = kbeg; kb < kend; ++kb) {
                const uint32_t slot = nslot % kSlots, pos = (uint32_t)(kb - kbeg) % kGroupsPerSlot;
                if (pos == 0 && !mbar_wait(&sc_empty[slot], ((nslot / kSlots) & 1) ^ 1, abort_flag)) {
                    record_timeout(p.status, kSiteScaleEmpty);
                    ok = false;
                    break;
                }
                cp_async_16_zfill(sm_sa + ((size_t)slot * kGroupsPerSlot + pos) * kHalfM + 4 * lane,
                                  p.sa + (int64_t)kb * p.ldsa + (sa_x < p.ldsa ? sa_x : 0), sa_x < p.ldsa ? 16u : 0u);
                if (lane == 0)
                    cp_async_16_zfill(sm_sb + ((size_t)slot * kGroupsPerSlot + pos) * 4,
                                      p.sb + (int64_t)kb * p.ldsb + sb_x, 16u);
                if (pos == kGroupsPerSlot - 1 || kb == kend - 1) {
                    cp_async_arrive_noinc(&sc_full[slot]);
                    ++nslot;
                }
            }
        }
        if (!ok) *abort_flag = 1;
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncwarp();
    } else if (warp == kMma || warp == kMma2) {
        // Two issuers: warp 1 takes the even K groups, warp 3 the odd ones
        // (their stages and TMEM buffers never overlap), so each has two MMA
        // periods for its two barrier tests and four instructions per group.
        if (rank == 0) {
            const uint32_t mine = warp == kMma ? 0u : 1u;
            const uint32_t idesc = idesc_e4m3_f32(2 * kHalfM, kTileN);
            uint32_t it = 0;
            bool ok = true;
            PairSegIter si;
            int32_t tile, kbeg, kend, piece;
            while (ok && si.next(p, tile, kbeg, kend, piece)) {
                for (int32_t kb = kbeg; kb < kend; ++kb, ++it) {
                    if ((it & 1) != mine) continue;
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1;
                    const uint32_t buf = it % kBufs, phb = (it / kBufs) & 1;
                    if (!mbar_wait(&tm_empty[buf], phb ^ 1, abort_flag)) {
                        record_timeout(p.status, kSiteMmaTmemEmpty);
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(&full[s], ph, abort_flag)) {
                        record_timeout(p.status, kSiteMmaFull);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (elect_one()) {
                        const uint64_t da = smem_desc_kmajor_sw128(sm_a + s * L::a_bytes);
                        const uint64_t db = smem_desc_kmajor_sw128(sm_b + s * L::b_bytes);
                        const uint32_t d_tmem = tmem_base + buf * kTileN;
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k)
                            mma_e4m3_pair(d_tmem, da + 2 * k, db + 2 * k, idesc, k > 0 ? 1u : 0u);
                        mma_commit_pair(&empty[s], 0x3);
                        mma_commit_pair(&tm_full[buf], 0x3);
                    }
                    __syncwarp();
                }
            }
            if (!ok) *abort_flag = 1;
            // every pair MMA of this issuer has completed before tensor memory is released
            if (elect_one()) mma_commit_pair(drain, 0x1);
            __syncwarp();
            mbar_wait(drain, 0, nullptr, 20u * 1000u * 1000u);
        }
        __syncwarp();
    } else if (warp >= kEpi0) {
        regs_increase<kEpiRegs>();
        const uint32_t quarter = warp & 3;
        const uint32_t parity = (warp - kEpi0) >> 2;        // 0: even K groups, 1: odd K groups
        const uint32_t row = quarter * 32 + lane;
        const uint32_t lane_addr = (quarter * 32) << 16;
        float4 *xch_mine = reinterpret_cast<float4 *>(smem + L::off_xch + (warp - kEpi0) * L::xch_warp);
        const float4 *xch_partner =
            reinterpret_cast<const float4 *>(smem + L::off_xch + ((warp - kEpi0) ^ 4) * L::xch_warp);
        uint32_t it = 0;                         // K groups so far (TMEM buffer ring)
        uint32_t nslot = 0;                      // scale slots so far
        bool ok = true;
        PairSegIter si;
        int32_t tile, kbeg, kend, piece;
        while (si.next(p, tile, kbeg, kend, piece)) {
            int32_t mp, nt;
            pair_tile_coords(tile, p, mp, nt);
            float2 acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.0f, 0.0f);
            const int sb_sel = nt & 3;           // the tile's 128x128 block of B in its 16-byte chunk
            for (int32_t kb = kbeg; kb < kend; ++kb, ++it) {
                const uint32_t slot = nslot % kSlots, pos = (uint32_t)(kb - kbeg) % kGroupsPerSlot;
                if (ok && (pos & 1) == parity) {
                    if (pos == parity && !mbar_wait(&sc_full[slot], (nslot / kSlots) & 1, abort_flag)) {
                        record_timeout(p.status, kSiteEpiScale);
                        ok = false;
                        *abort_flag = 1;
                    }
                    const uint32_t buf = it % kBufs, phb = (it / kBufs) & 1;
                    if (ok && !mbar_wait(&tm_full[buf], phb, abort_flag)) {
                        record_timeout(p.status, kSiteEpiTmemFull);
                        ok = false;
                        *abort_flag = 1;
                    }
                    if (ok) {
                        const float sa_v = sm_sa[((size_t)slot * kGroupsPerSlot + pos) * kHalfM + row];
                        const float blk = sa_v * sm_sb[((size_t)slot * kGroupsPerSlot + pos) * 4 + sb_sel];
                        const float2 blk2 = make_float2(blk, blk);
                        tc_fence_after_sync();
                        const uint32_t taddr = tmem_base + lane_addr + buf * kTileN;
#pragma unroll
                        for (int g = 0; g < kTileN / 32; ++g) {
                            uint32_t r[32];
                            tmem_ld_sync<32>(taddr + g * 32, r);
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float2 pv =
                                    make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                                acc[g * 16 + i] = __ffma2_rn(pv, blk2, acc[g * 16 + i]);
                            }
                        }
                        tc_fence_before_sync();
                        if (rank == 0) {
                            mbar_arrive(&tm_empty[buf]);
                        } else {
                            __syncwarp();
                            if (lane == 0) mbar_arrive_cluster(cluster_map(&tm_empty[buf], 0));
                        }
                    }
                }
                // the last group of a slot: both parities release it (a warp
                // whose parity had no group in a one-group slot releases it too)
                if (pos == kGroupsPerSlot - 1 || kb == kend - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sc_empty[slot]);
                    ++nslot;
                }
            }
            const int64_t m = (int64_t)mp * 2 * kHalfM + rank * kHalfM + row;
            const int64_t n0 = (int64_t)nt * kTileN;
            if (parity == 0)
                tile_end<0, OUT_F32>(p, acc, xch_mine, xch_partner, quarter, lane, row, rank, m, n0, tile, piece, ok,
                                     abort_flag, tail_last);
            else
                tile_end<1, OUT_F32>(p, acc, xch_mine, xch_partner, quarter, lane, row, rank, m, n0, tile, piece, ok,
                                     abort_flag, tail_last);
        }
        if (!ok) *abort_flag = 1;
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();                              // no pair MMA, remote arrive or TMA is left in flight
    if (warp == kMma) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, 512);
    }
}

std::atomic<int> g_max_clusters[64];                          // co-resident CTA pairs per device (0: not yet known)

template <bool OUT_F32>
cudaError_t launch_pair_variant(const GemmArgs &a, const PairParams &p, int clusters, cudaStream_t stream)
{
    CUtensorMap tmA, tmB;
    if (!make_tensor_map_2d(&tmA, 1, false, a.A, a.K, a.M, a.K, kBK, kHalfM, true) ||
        !make_tensor_map_2d(&tmB, 1, false, a.B, a.K, a.N, a.K, kBK, kHalfN, true))
        return cudaErrorInvalidValue;
    auto kern = gemm_pair_kernel<OUT_F32>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PairLayout::dyn_bytes);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = PairLayout::dyn_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p);
}

}  // namespace

// Co-resident CTA pairs of the pair kernel on the current device (looked up
// once per device; 0 if the device cannot run it).
int pair_max_clusters()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (g_max_clusters[dev].load(std::memory_order_relaxed) == 0) {
        auto kern = gemm_pair_kernel<false>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PairLayout::dyn_bytes) !=
            cudaSuccess)
            return 0;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kPairThreads, 1, 1);
        cfg.dynamicSmemBytes = PairLayout::dyn_bytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            g_max_clusters[dev].store(-1, std::memory_order_relaxed);
        } else {
            g_max_clusters[dev].store(n, std::memory_order_relaxed);
        }
    }
    const int n = g_max_clusters[dev].load(std::memory_order_relaxed);
    return n > 0 ? n : 0;
}

int pair_tile_n()
{
    return kTileN;
}

size_t pair_tail_workspace_bytes()
{
    // a 128 x 128 FP32 partial per CTA, up to 148 CTAs in the tail wave
    return kWsPartialsOffset + (size_t)148 * kHalfM * kTileN * 4;
}

PairPlan pair_plan(const GemmArgs &a, int clusters)
{
    PairPlan pl{};
    const int64_t mp = (a.M + 2 * kHalfM - 1) / (2 * kHalfM), nt = (a.N + kTileN - 1) / kTileN;
    const int64_t tiles = mp * nt, KB = a.K / kBK;
    pl.tiles = (int32_t)tiles;
    pl.dp_tiles = (int32_t)tiles;
    pl.tail_s = 1;
    const int G = clusters;
    if (G <= 0) return pl;
    const int64_t W = tiles / G, R = tiles % G;
    pl.cost = (W + (R > 0 ? 1 : 0)) * KB;
    // Last-wave split, as for the single-SM kernel: K pieces of the R tail
    // tiles fill one more wave; a piece costs ceil(KB / s) K-group steps plus
    // about three for its partial (store, and the last piece's read-back).
    if (R > 0 && 2 * R <= kMaxCounters && a.ws_bytes >= pair_tail_workspace_bytes()) {
        for (int64_t s = 2; s <= KB && R * s <= G && 2 * R * s <= 148; ++s) {
            const int64_t c = W * KB + (KB + s - 1) / s + 2 * s + 1;
            if (c < pl.cost) {
                pl.cost = c;
                pl.dp_tiles = (int32_t)(W * G);
                pl.tail_s = (int32_t)s;
            }
        }
    }
    return pl;
}

cudaError_t launch_pair(const GemmArgs &a, cudaStream_t stream)
{
    const int G = pair_max_clusters();
    if (G <= 0) return cudaErrorNotSupported;
    const PairPlan pl = pair_plan(a, G);
    PairParams p{};
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.KB = (int32_t)(a.K / kBK);
    p.num_mp = (int32_t)((a.M + 2 * kHalfM - 1) / (2 * kHalfM));
    p.num_nt = (int32_t)((a.N + kTileN - 1) / kTileN);
    p.num_tiles = pl.tiles;
    p.C = a.C;
    p.ldc = a.ldc;
    p.status = reinterpret_cast<DeviceStatus *>(a.workspace);
    p.sa = a.sa;
    p.sb = a.sb;
    p.ldsa = a.ldsa;
    p.ldsb = a.ldsb;
    p.dp_tiles = pl.dp_tiles;
    int clusters = pl.tiles < G ? pl.tiles : G;
    if (pl.tail_s > 1) {
        const int32_t units = (pl.tiles - pl.dp_tiles) * pl.tail_s;
        clusters = pl.dp_tiles > 0 ? G : units;
        p.tail_s = pl.tail_s;
        p.tail_units = units;
        uint8_t *ws = static_cast<uint8_t *>(a.workspace);
        p.tail_tickets = reinterpret_cast<uint32_t *>(ws + kWsHeaderBytes);
        p.tail_partials = reinterpret_cast<float *>(ws + kWsPartialsOffset);
    }
    if (clusters <= 0) return cudaSuccess;
    return a.out_f32 ? launch_pair_variant<true>(a, p, clusters, stream)
                     : launch_pair_variant<false>(a, p, clusters, stream);
}

}  // namespace fgf8
