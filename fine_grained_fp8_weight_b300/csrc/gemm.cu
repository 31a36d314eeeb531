// gemm.cu -- block-scaled FP8 GEMM for sm_103a (tcgen05 + TMA + TMEM).
//
// C[m][n] = sum_kb P_kb[m][n] * sa[kb][m] * sb_kb(n),  P_kb = sum_{k in kb} qa*qb
//
// "dssusan.co.kr Q&A post 93378" (inner-dimension and E4M3 passages) scales
// every 128-wide group along K separately, so a K group's partial product
// must leave the tensor cores before it can be scaled; "kailasan.com
// recruit post 147436" (hardware-suggestion passage) has the partial results
// copied out at each interval, multiplied by the scaling factors and added
// into FP32.  Here that interval is one 128-wide K group.
//
// gemm_blockscaled_kernel (128 x 256 or 128 x 128 output tiles, persistent,
// dense and grouped layouts):
//   - warp 0 (one lane) streams the A/B tiles with TMA into a ring of
//     shared-memory stages;
//   - warp 2 copies each K group's scale vectors (sa, and block or per-row
//     sb) into a separate ring with cp.async, 8 K groups per slot (4 with
//     per-row B scales) and three slots;
//   - warp 1 (one lane) issues 4 tcgen05.mma (K = 32 each) per K group into a
//     fresh FP32 partial in tensor memory, alternating between two TMEM
//     buffers so that the next group's MMAs run while this one is promoted;
//   - warps 4..11 (two promotion warpgroups, half of the tile's columns
//     each) read each partial with tcgen05.ld, multiply by sa*sb and add into
//     FP32 registers, then write the finished tile (BF16 or FP32).  With
//     block B scales a thread owns one TMEM lane (one output row); with
//     per-row B scales it reads the 16x256b shape (4 rows x 32 columns), so
//     that it needs a quarter of the column scales.
//   Schedule: tile t runs on CTA t mod grid.  When the tiles leave the last
//   wave over the SMs partly empty (dense GEMMs, workspace permitting), the
//   whole waves keep that order and each remaining tile is cut into K pieces
//   on otherwise idle CTAs; the last piece to finish (an atomic ticket) adds
//   the FP32 partials in K order and writes the tile.  No CTA waits for
//   another.  A test switch runs the same kernel in clusters of two CTAs on
//   vertically adjacent tiles that share the B panel by TMA multicast.
// gemm_smallm_kernel (decode, dense M <= 128 tokens): the weight tile takes
// the MMA's M side and the tokens its N side, K is split over the CTAs of a
// thread-block cluster, which add their partials in split order through
// distributed shared memory; the same kernel serves the masked grouped layout
// (per-expert token slots of up to 256 rows with device-side counts; the
// K groups per barrier handshake follow each expert's count) and, for
// M <= 256, the variant that quantizes BF16 tokens inside the kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "e4m3_rule.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace fgf8 {
namespace {

constexpr int BM = 128;                 // rows of A per tile (TMEM lanes)
constexpr int BK = 128;                 // K elements (= bytes) per group
constexpr int kThreads = 384;           // 12 warps: one control warpgroup, two promotion warpgroups
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kScaleWarp = 2;
constexpr int kEpiWarp0 = 4;            // warps 4..11; warp w may read TMEM lanes 32*(w%4) .. +31
constexpr int kEpiWarps = 8;
// Registers per thread after the split (the launch gives 168 to every thread):
// the control warpgroup gives some back, the promotion warpgroups take them.
constexpr uint32_t kCtrlRegs = 40;
constexpr uint32_t kEpiRegs = 232;
static_assert(128 * kCtrlRegs + 256 * kEpiRegs <= 384 * 168, "register split exceeds the launch budget");

// wait-site ids reported in the status word
enum : int32_t {
    kSiteProducerEmpty = 1,
    kSiteProducerScale = 2,
    kSiteMmaTmemEmpty = 3,
    kSiteMmaFull = 4,
    kSiteEpiScale = 5,
    kSiteEpiTmemFull = 6,
    kSiteProbe = 7,
    kSiteQuantFull = 8,
    kSiteSelftest = 99
};

struct Params {
    int64_t M, N, K;
    int32_t KB;
    int32_t num_m_blocks, num_n_blocks, num_tiles;   // with multicast clusters: rows of MC M blocks
    int32_t m_blocks;                   // 128-row blocks of A
    int32_t m_major;                    // tile order: 1 = m outer, 0 = n outer within bands of M blocks
    int32_t band;                       // n outer: M blocks per band (all of them when A fits in L2)
    void *C;
    int64_t ldc;
    const int32_t *m_indices;           // grouped layout when non-null
    int64_t b_rows_per_expert;          // N (grouped)
    int32_t sb_rows_per_expert;         // KB (grouped)
    DeviceStatus *status;
    const float *sa;                    // scales, copied by the scale warp with cp.async
    const float *sb;
    int64_t ldsa, ldsb;
    // Tail split (with multicast: cluster tiles on clusters):
    // tiles [0, dp_tiles) run whole, tile t on CTA t mod G; the
    // other R = num_tiles - dp_tiles tiles (fewer than G) are each cut into
    // tail_s contiguous K-group pieces, unit v = piece * R + tail tile on CTA v,
    // so the last wave keeps every SM busy.  The last piece of a tail tile to
    // finish adds the FP32 partials in piece (K) order.  Without a tail,
    // dp_tiles = num_tiles and tail_units = 0.
    int32_t dp_tiles, tail_s, tail_units;
    float *tail_partials;               // [R * tail_s][BN / 4][128][4]
    uint32_t *tail_tickets;             // [R], zero between calls
};

// The segments (tile, K groups k0..k1, tail piece or -1) one CTA processes, in
// order; every role of the CTA walks the same sequence.  With clusters of MC
// CTAs (multicast) both CTAs of a cluster walk the same cluster tiles: the
// walk goes by cluster index and cluster count.
template <int MC>
struct SegIter {
    int32_t t, v;
    __device__ __forceinline__ SegIter() : t((int32_t)(blockIdx.x / MC)), v((int32_t)(blockIdx.x / MC)) {}
    __device__ __forceinline__ bool next(const Params &p, int32_t &tile, int32_t &k0, int32_t &k1, int32_t &piece)
    {
        if (t < p.dp_tiles) {
            tile = t;
            k0 = 0;
            k1 = p.KB;
            piece = -1;
            t += gridDim.x / MC;
            return true;
        }
        if (v >= p.tail_units) return false;
        const int32_t R = p.num_tiles - p.dp_tiles;
        piece = v / R;
        tile = p.dp_tiles + (v - piece * R);
        k0 = piece * p.KB / p.tail_s;
        k1 = (piece + 1) * p.KB / p.tail_s;
        v += gridDim.x / MC;
        return true;
    }
};

__host__ __device__ constexpr size_t align_up(size_t v, size_t a)
{
    return (v + a - 1) / a * a;
}

// Scale ring: SS slots of SG K groups each (one barrier handshake per SG
// groups): per group 128 floats of sa and either the 16-byte chunk holding
// the tile's 128x128 block scales or BN per-row scales of B.
template <int BN, int STAGES, int SG, int SS, bool ROW_SB>
struct Layout {
    static constexpr size_t a_bytes = (size_t)BM * BK;
    static constexpr size_t b_bytes = (size_t)BN * BK;
    static constexpr int sb_pitch = ROW_SB ? BN : 4;         // floats of B scales per K group
    static constexpr size_t off_a = 0;
    static constexpr size_t off_b = off_a + STAGES * a_bytes;
    static constexpr size_t off_sa = off_b + STAGES * b_bytes;
    static constexpr size_t off_sb = off_sa + (size_t)SS * SG * BM * 4;
    static constexpr size_t off_bar = align_up(off_sb + (size_t)SS * SG * sb_pitch * 4, 16);
    static constexpr int num_bars = 2 * STAGES + 2 * SS + 4 + 1;
    static constexpr size_t off_misc = off_bar + (size_t)num_bars * 8;
    static constexpr size_t total = off_misc + 16;
    static constexpr size_t dyn_bytes = total + 1024;    // slack to align the base to 1024
    static constexpr uint32_t tmem_cols = 2 * BN;        // two partial buffers
};

// Wait until this thread's cp.async copies have landed (before a CTA exits).
__device__ __forceinline__ void scale_copies_wait()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void tile_coords(int32_t tile, const Params &p, int32_t &mb, int32_t &nb)
{
    if (p.m_major) {
        mb = tile / p.num_n_blocks;
        nb = tile - mb * p.num_n_blocks;
    } else {
        // n outer inside a band of p.band M blocks: the band's A panels stay
        // in L2 while every B column panel streams past them once
        const int32_t band_tiles = p.band * p.num_n_blocks;
        const int32_t b = tile / band_tiles;
        const int32_t r = tile - b * band_tiles;
        const int32_t h = min(p.band, p.num_m_blocks - b * p.band);
        nb = r / h;
        mb = b * p.band + (r - nb * h);
    }
}

// Expert of an M block in the grouped layout (-1: padding block, skipped).
__device__ __forceinline__ int32_t block_expert(const Params &p, int32_t mb)
{
    return p.m_indices ? __ldg(p.m_indices + (int64_t)mb * BM) : 0;
}

__device__ __forceinline__ void store_bf16x8(__nv_bfloat16 *dst, float2 a, float2 b, float2 c, float2 d)
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

// MC = 2: the kernel runs in clusters of two CTAs on vertically adjacent
// tiles (M blocks 2r and 2r + 1, the same N block).  Each CTA loads its own
// A panel and one half of the shared B panel, multicast into both CTAs'
// stages; a stage is refilled once both CTAs' MMAs have read it (each MMA
// warp's commit arrives on the stage's barrier in both CTAs).
template <int BN, int STAGES, int SG, int SS, bool ROW_SB, bool OUT_F32, int MC>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_blockscaled_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const Params p)
{
    using L = Layout<BN, STAGES, SG, SS, ROW_SB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
    uint8_t *sm_a = smem + L::off_a;
    uint8_t *sm_b = smem + L::off_b;
    float *sm_sa = reinterpret_cast<float *>(smem + L::off_sa);
    float *sm_sb = reinterpret_cast<float *>(smem + L::off_sb);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::off_bar);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *sc_full = bars + 2 * STAGES;
    uint64_t *sc_empty = bars + 2 * STAGES + SS;
    uint64_t *tm_full = bars + 2 * STAGES + 2 * SS;
    uint64_t *tm_empty = tm_full + 2;
    uint64_t *drain = tm_full + 4;
    uint32_t *tmem_base_slot = reinterpret_cast<uint32_t *>(smem + L::off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::off_misc + 4);
    volatile int *tail_last = reinterpret_cast<volatile int *>(smem + L::off_misc + 8);

    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();
    static_assert(MC == 1 || MC == 2, "clusters of one or two CTAs");
    const uint32_t crank = MC > 1 ? cluster_ctarank() : 0;
    // this CTA's M block and the N block of a (cluster) tile
    auto tile_mb = [&](int32_t tile, int32_t &mb, int32_t &nb) {
        tile_coords(tile, p, mb, nb);
        mb = mb * MC + (int32_t)crank;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], MC);                   // every CTA's MMA warp frees the stage
        }
        for (int i = 0; i < SS; ++i) {
            mbar_init(&sc_full[i], 32);                 // one cp.async arrival per scale-warp lane
            mbar_init(&sc_empty[i], kEpiWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tm_full[i], 1);
            mbar_init(&tm_empty[i], kEpiWarps * 32);    // every promotion thread arrives
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_base_slot, L::tmem_cols);
    tc_fence_before_sync();
    __syncthreads();
    if (MC > 1) cluster_sync();                         // the peer may now fill this CTA's stages
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_base_slot;

    if (warp < kEpiWarp0) regs_decrease<kCtrlRegs>();

    if (warp == kProducerWarp) {
        if (elect_one()) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            uint32_t it = 0;
            bool ok = true;
            SegIter<MC> si;
            int32_t tile, kbeg, kend, piece;
            while (ok && si.next(p, tile, kbeg, kend, piece)) {
                int32_t mb, nb;
                tile_mb(tile, mb, nb);
                const int32_t e = block_expert(p, mb);
                if (e < 0) continue;
                const int32_t b_row = (int32_t)(e * p.b_rows_per_expert) + nb * BN;
                // an M block past the end (odd block count, second CTA of the
                // last cluster row) loads the last block; its rows are not stored
                const int32_t a_row = (MC == 1 || mb < p.m_blocks ? mb : p.m_blocks - 1) * BM;
                for (int32_t kb = kbeg; kb < kend; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag)) {
                        record_timeout(p.status, kSiteProducerEmpty);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], (uint32_t)(L::a_bytes + L::b_bytes));
                    tma_load_2d(sm_a + s * L::a_bytes, &tmA, &full[s], kb * BK, a_row);
                    if (MC > 1)
                        tma_load_2d_multicast(sm_b + s * L::b_bytes + crank * (L::b_bytes / MC), &tmB, &full[s],
                                              kb * BK, b_row + (int32_t)crank * (BN / MC), (uint16_t)((1u << MC) - 1));
                    else
                        tma_load_2d(sm_b + s * L::b_bytes, &tmB, &full[s], kb * BK, b_row);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                // let the copies already issued land before the CTA exits
                const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0;
                for (uint32_t i = first; i <= it; ++i)
                    mbar_wait(&full[i % STAGES], (i / STAGES) & 1, nullptr, 20u * 1000u * 1000u);
            }
        }
        __syncwarp();
    } else if (warp == kScaleWarp) {
        // The scale vectors of each K group (128 floats of sa, and 4 floats of
        // block sb or BN floats of per-row sb) are copied by the whole warp
        // with 16-byte cp.async copies: generic-proxy writes that do not queue
        // behind the operand tiles in the TMA unit.  Chunks past the end of a
        // scale row are zero-filled without a read.
        // Every segment (tile or tail piece) starts a new slot.
        uint32_t nslot = 0;
        bool ok = true;
        SegIter<MC> si;
        int32_t tile, kbeg, kend, piece;
        while (ok && si.next(p, tile, kbeg, kend, piece)) {
            int32_t mb, nb;
            tile_mb(tile, mb, nb);
            const int32_t e = block_expert(p, mb);
            if (e < 0) continue;
            const int64_t s_row0 = (int64_t)e * p.sb_rows_per_expert;
            const int64_t sa_x = (int64_t)mb * BM + 4 * lane;
            for (int32_t kb = kbeg; kb < kend; ++kb) {
                const uint32_t slot = nslot % SS, pos = (uint32_t)(kb - kbeg) % SG;
                if (pos == 0 && !mbar_wait(&sc_empty[slot], ((nslot / SS) & 1) ^ 1, abort_flag)) {
                    record_timeout(p.status, kSiteProducerScale);
                    ok = false;
                    break;
                }
                const uint32_t g = slot * SG + pos;              // K group's place in the ring
                cp_async_16_zfill(sm_sa + g * BM + 4 * lane, p.sa + (int64_t)kb * p.ldsa + (sa_x < p.ldsa ? sa_x : 0),
                                  sa_x < p.ldsa ? 16u : 0u);
                const float *sb_row = p.sb + (s_row0 + kb) * p.ldsb;
                if constexpr (ROW_SB) {
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h) {
                        const int64_t x = (int64_t)nb * BN + h * 128 + 4 * lane;
                        cp_async_16_zfill(sm_sb + g * L::sb_pitch + h * 128 + 4 * lane, sb_row + (x < p.ldsb ? x : 0),
                                          x < p.ldsb ? 16u : 0u);
                    }
                } else if (lane == 0) {
                    cp_async_16_zfill(sm_sb + g * L::sb_pitch, sb_row + ((nb * BN / 128) & ~3), 16u);
                }
                if (pos == SG - 1 || kb == kend - 1) {
                    cp_async_arrive_noinc(&sc_full[slot]);
                    ++nslot;
                }
            }
        }
        if (!ok) *abort_flag = 1;
        scale_copies_wait();
        __syncwarp();
    } else if (warp == kMmaWarp) {
        const uint32_t idesc = idesc_e4m3_f32(BM, BN);
        uint32_t it = 0;
        bool ok = true;
        SegIter<MC> si;
        int32_t tile, kbeg, kend, piece;
        while (ok && si.next(p, tile, kbeg, kend, piece)) {
            int32_t mb, nb;
            tile_mb(tile, mb, nb);
            if (block_expert(p, mb) < 0) continue;
            for (int32_t kb = kbeg; kb < kend; ++kb, ++it) {
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                const uint32_t buf = it & 1, phb = (it >> 1) & 1;
                // The operand stage is normally loaded long before its TMEM
                // buffer comes free: test it first, so that the buffer's
                // release is followed directly by the MMAs.
                if (!mbar_wait(&full[s], ph, abort_flag)) {
                    record_timeout(p.status, kSiteMmaFull);
                    ok = false;
                    break;
                }
                if (!mbar_wait(&tm_empty[buf], phb ^ 1, abort_flag)) {
                    record_timeout(p.status, kSiteMmaTmemEmpty);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                if (elect_one()) {
                    const uint64_t da = smem_desc_kmajor_sw128(sm_a + s * L::a_bytes);
                    const uint64_t db = smem_desc_kmajor_sw128(sm_b + s * L::b_bytes);
                    const uint32_t d_tmem = tmem_base + buf * BN;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)       // 32 bytes = 2 x 16-byte descriptor units
                        mma_e4m3(d_tmem, da + 2 * k, db + 2 * k, idesc, k > 0 ? 1u : 0u);
                    if (MC > 1)
                        mma_commit_multicast(&empty[s], (uint16_t)((1u << MC) - 1));
                    else
                        mma_commit(&empty[s]);
                    mma_commit(&tm_full[buf]);
                }
                __syncwarp();
            }
        }
        if (!ok) *abort_flag = 1;
        // every MMA issued by this warp completes before TMEM is released
        if (elect_one()) mma_commit(drain);
        __syncwarp();
        mbar_wait(drain, 0, nullptr, 20u * 1000u * 1000u);
    } else if (warp >= kEpiWarp0) {
        regs_increase<kEpiRegs>();
        // Promotion warpgroups: warps 4..7 cover TMEM lane quarters 0..3 for the
        // first half of the tile's columns, warps 8..11 for the second half.
        constexpr int HALF = BN / 2;                        // columns per promotion warp
        constexpr int NCH = HALF / 32;                      // 32-column TMEM loads per K group
        const uint32_t quarter = warp & 3;
        const uint32_t half = (warp - kEpiWarp0) >> 2;
        const uint32_t row = quarter * 32 + lane;
        const uint32_t lane_addr = (quarter * 32) << 16;
        const uint32_t col0 = half * HALF;
        // Per-row B scales: the partial is read in the 16x256b shape, so a
        // thread holds 4 rows x HALF/4 columns (instead of 1 row x HALF) and
        // reads a quarter of the column scales.  acc[a], a = (j*NREP + i)*2 + k:
        // row quarter*32 + 16j + 8k + lane/4, columns col0 + 8i + 2(lane%4), +1.
        constexpr int NREP = HALF / 8;
        const uint32_t rs_r = quarter * 32 + (lane >> 2);
        const uint32_t rs_c = col0 + 2 * (lane & 3);
        uint32_t it = 0;                                    // K groups so far (TMEM buffers)
        uint32_t nslot = 0;                                 // scale slots so far
        bool ok = true;
        // After a failed wait a warp still walks its remaining segments (without
        // waiting), so that all eight reach the tail's named barrier together.
        SegIter<MC> si;
        int32_t tile, kbeg, kend, piece;
        while (si.next(p, tile, kbeg, kend, piece)) {
            int32_t mb, nb;
            tile_mb(tile, mb, nb);
            if (block_expert(p, mb) < 0) continue;
            float2 acc[HALF / 2];
#pragma unroll
            for (int i = 0; i < HALF / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);
            const int sb_sel = ROW_SB ? 0 : ((nb * BN / 128) & 3) + (int)(col0 / 128);
            for (int32_t kb = kbeg; ok && kb < kend; ++kb, ++it) {
                const uint32_t slot = nslot % SS, pos = (uint32_t)(kb - kbeg) % SG;
                if (pos == 0 && !mbar_wait(&sc_full[slot], (nslot / SS) & 1, abort_flag)) {
                    record_timeout(p.status, kSiteEpiScale);
                    ok = false;
                    *abort_flag = 1;
                    break;
                }
                const uint32_t g = slot * SG + pos;
                const float blk = ROW_SB ? 0.0f : sm_sa[g * BM + row] * sm_sb[g * L::sb_pitch + sb_sel];
                const float2 blk2 = make_float2(blk, blk);
                const uint32_t buf = it & 1, phb = (it >> 1) & 1;
                if (!mbar_wait(&tm_full[buf], phb, abort_flag)) {
                    record_timeout(p.status, kSiteEpiTmemFull);
                    ok = false;
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t taddr = tmem_base + lane_addr + buf * BN + col0;
                if constexpr (ROW_SB) {
                    // per-column B scales: the scales of this thread's 4 rows,
                    // then per 8 column blocks their B scales (one pair each)
                    // and the two 16-lane loads
                    float sa_r[4];
#pragma unroll
                    for (int jk = 0; jk < 4; ++jk) sa_r[jk] = sm_sa[g * BM + rs_r + 16 * (jk >> 1) + 8 * (jk & 1)];
                    const float *sbc = sm_sb + g * L::sb_pitch + rs_c;
#pragma unroll
                    for (int i0 = 0; i0 < NREP; i0 += 8) {
                        // both 16-lane halves of 8 column blocks, then each
                        // column pair's B scale once for the thread's 4 rows
                        uint32_t r0[32], r1[32];
                        tmem_ld_16x256b_x8_sync(tmem_base + ((quarter * 32) << 16) + buf * BN + col0 + 8 * i0, r0);
                        tmem_ld_16x256b_x8_sync(tmem_base + ((quarter * 32 + 16) << 16) + buf * BN + col0 + 8 * i0, r1);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float2 sb2 = *reinterpret_cast<const float2 *>(sbc + 8 * (i0 + i));
                            const int a0 = (i0 + i) * 2, a1 = (NREP + i0 + i) * 2;
                            acc[a0] = __ffma2_rn(make_float2(__uint_as_float(r0[4 * i]), __uint_as_float(r0[4 * i + 1])),
                                                 __fmul2_rn(make_float2(sa_r[0], sa_r[0]), sb2), acc[a0]);
                            acc[a0 + 1] = __ffma2_rn(make_float2(__uint_as_float(r0[4 * i + 2]), __uint_as_float(r0[4 * i + 3])),
                                                     __fmul2_rn(make_float2(sa_r[1], sa_r[1]), sb2), acc[a0 + 1]);
                            acc[a1] = __ffma2_rn(make_float2(__uint_as_float(r1[4 * i]), __uint_as_float(r1[4 * i + 1])),
                                                 __fmul2_rn(make_float2(sa_r[2], sa_r[2]), sb2), acc[a1]);
                            acc[a1 + 1] = __ffma2_rn(make_float2(__uint_as_float(r1[4 * i + 2]), __uint_as_float(r1[4 * i + 3])),
                                                     __fmul2_rn(make_float2(sa_r[3], sa_r[3]), sb2), acc[a1 + 1]);
                        }
                    }
                } else {
                    // 64 columns per load and wait, then the FMAs
#pragma unroll
                    for (int g = 0; g < NCH / 2; ++g) {
                        uint32_t r[64];
                        tmem_ld_sync<64>(taddr + g * 64, r);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float2 pv = make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                            acc[g * 32 + i] = __ffma2_rn(pv, blk2, acc[g * 32 + i]);
                        }
                    }
                }
                tc_fence_before_sync();
                mbar_arrive(&tm_empty[buf]);
                if (pos == SG - 1 || kb == kend - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sc_empty[slot]);
                    ++nslot;
                }
            }
            if (piece >= 0) {
                // A piece of a tail tile: store the FP32 partial, take a ticket;
                // the last piece to arrive adds all of them in K order.  (With
                // multicast clusters each CTA of a tail cluster tile owns one.)
                const int32_t ti = (tile - p.dp_tiles) * MC + (int32_t)crank;
                if (ok) {
                    float *mine = p.tail_partials + (int64_t)(ti * p.tail_s + piece) * (BM * BN);
                    if constexpr (ROW_SB) {
#pragma unroll
                        for (int a = 0; a < HALF / 2; ++a) {
                            const uint32_t rr = rs_r + 16 * (a / (2 * NREP)) + 8 * (a & 1);
                            const uint32_t cc = rs_c + 8 * ((a / 2) % NREP);
                            *reinterpret_cast<float2 *>(mine + ((int64_t)(cc / 4) * BM + rr) * 4 + (cc & 3)) = acc[a];
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < HALF; c += 4)
                            *reinterpret_cast<float4 *>(mine + ((int64_t)((col0 + c) / 4) * BM + row) * 4) =
                                make_float4(acc[c / 2].x, acc[c / 2].y, acc[c / 2 + 1].x, acc[c / 2 + 1].y);
                    }
                }
                __threadfence();
                const bool all_ok = named_barrier_and(1, kEpiWarps * 32, ok && !*abort_flag);
                if (all_ok && threadIdx.x == kEpiWarp0 * 32) {
                    const uint32_t ticket = atomicAdd(p.tail_tickets + ti, 1u);
                    const int last = ticket == (uint32_t)(p.tail_s - 1);
                    if (last) p.tail_tickets[ti] = 0u;          // ready for the next call
                    *tail_last = last;
                }
                named_barrier_sync(1, kEpiWarps * 32);
                if (!all_ok) ok = false;
                if (!all_ok || !*tail_last) continue;
                __threadfence();
                const float *part = p.tail_partials + (int64_t)ti * p.tail_s * (BM * BN);
                if constexpr (ROW_SB) {
                    // in K order, 8 values of one piece in flight at a time
                    // (keeps the 128 accumulator registers clear of spills)
#pragma unroll
                    for (int a = 0; a < HALF / 2; ++a) acc[a] = make_float2(0.0f, 0.0f);
                    for (int32_t q = 0; q < p.tail_s; ++q) {
                        const float *pq = part + (int64_t)q * (BM * BN);
#pragma unroll
                        for (int a0 = 0; a0 < HALF / 2; a0 += 8) {
                            float2 v[8];
#pragma unroll
                            for (int a = a0; a < a0 + 8; ++a) {
                                const uint32_t rr = rs_r + 16 * (a / (2 * NREP)) + 8 * (a & 1);
                                const uint32_t cc = rs_c + 8 * ((a / 2) % NREP);
                                v[a - a0] = __ldcg(reinterpret_cast<const float2 *>(pq + ((int64_t)(cc / 4) * BM + rr) * 4 + (cc & 3)));
                            }
#pragma unroll
                            for (int a = a0; a < a0 + 8; ++a) {
                                acc[a].x += v[a - a0].x;
                                acc[a].y += v[a - a0].y;
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < HALF; c += 4) {
                        const float4 v = __ldcg(reinterpret_cast<const float4 *>(part + ((int64_t)((col0 + c) / 4) * BM + row) * 4));
                        acc[c / 2] = make_float2(v.x, v.y);
                        acc[c / 2 + 1] = make_float2(v.z, v.w);
                    }
                    for (int32_t q = 1; q < p.tail_s; ++q) {
                        const float *pq = part + (int64_t)q * (BM * BN);
#pragma unroll
                        for (int c = 0; c < HALF; c += 4) {
                            const float4 v = __ldcg(reinterpret_cast<const float4 *>(pq + ((int64_t)((col0 + c) / 4) * BM + row) * 4));
                            acc[c / 2].x += v.x;
                            acc[c / 2].y += v.y;
                            acc[c / 2 + 1].x += v.z;
                            acc[c / 2 + 1].y += v.w;
                        }
                    }
                }
            } else if (!ok) {
                continue;
            }
            if constexpr (ROW_SB) {
                // this thread's 4 rows x HALF/4 columns, a pair of columns per store
#pragma unroll
                for (int a = 0; a < HALF / 2; ++a) {
                    const int64_t m = (int64_t)mb * BM + rs_r + 16 * (a / (2 * NREP)) + 8 * (a & 1);
                    const int64_t n = (int64_t)nb * BN + rs_c + 8 * ((a / 2) % NREP);
                    bool write = m < p.M && n < p.N;
                    if (write && p.m_indices) write = __ldg(p.m_indices + m) >= 0;
                    if (!write) continue;
                    if (OUT_F32)
                        *reinterpret_cast<float2 *>(static_cast<float *>(p.C) + m * p.ldc + n) = acc[a];
                    else
                        *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(p.C) + m * p.ldc + n) =
                            __float22bfloat162_rn(acc[a]);
                }
                continue;
            }
            // write this thread's finished row segment
            const int64_t m = (int64_t)mb * BM + row;
            bool write = m < p.M;
            if (write && p.m_indices) write = __ldg(p.m_indices + m) >= 0;
            if (write) {
                const int64_t n0 = (int64_t)nb * BN + col0;
                if (OUT_F32) {
                    float *dst = static_cast<float *>(p.C) + m * p.ldc + n0;
#pragma unroll
                    for (int c = 0; c < HALF; c += 4)
                        if (n0 + c < p.N)
                            *reinterpret_cast<float4 *>(dst + c) =
                                make_float4(acc[c / 2].x, acc[c / 2].y, acc[c / 2 + 1].x, acc[c / 2 + 1].y);
                } else {
                    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.C) + m * p.ldc + n0;
#pragma unroll
                    for (int c = 0; c < HALF; c += 8)
                        if (n0 + c < p.N) store_bf16x8(dst + c, acc[c / 2], acc[c / 2 + 1], acc[c / 2 + 2], acc[c / 2 + 3]);
                }
            }
        }
        if (!ok) *abort_flag = 1;
    }

    tc_fence_before_sync();
    __syncthreads();
    // no multicast copy or commit arrival of the peer is left in flight
    if (MC > 1) cluster_sync();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, L::tmem_cols);
    }
}


// ------------------------------------------------------------------------
// Small M (decode, M <= 256 tokens): the weight tile fills the MMA's M = 128
// side and the tokens its N side (NT = M rounded up to 16), i.e. D^T = W X^T
// per 128 weight rows, so the MMA shape suits a handful of tokens.  Such GEMMs
// read 128 x K bytes of weights per 2*128*NT*K FLOP, far below the tensor
// cores' ridge ("kailasan.com recruit post 147436", decode passage: the batch
// per expert is small and memory access is the bottleneck), so the K groups
// are split across CTAs until the SMs stream weights.  The S splits of one
// weight tile form a thread-block cluster: after its last K group each CTA
// leaves its FP32 partial in its own (by then idle) stage memory, the cluster
// synchronises once, and CTA r adds the r-th slice of all S partials in split
// order (deterministic) straight from the peers' shared memory and writes
// that slice of the output; a second cluster barrier keeps every CTA resident
// until its partial has been read.  Nothing goes through global memory but
// the output.
// Promotion: acc[token] += P[w_row][token] * (sb[w block][kb] * sa[kb][token]).
// ------------------------------------------------------------------------
constexpr int kMaxSplits = 8;   // split-K factor (= cluster size) of the small-M kernel, at most

struct SmallParams {
    int64_t M, N, K;
    int32_t KB, S, n_tiles;   // S: CTAs per cluster (blockIdx.x mod S = split = cluster rank)
    void *C;
    int64_t ldc;
    DeviceStatus *status;
    // masked grouped layout (decode MoE): expert e owns token rows
    // e*cap .. e*cap+cap-1 of A and C (and those columns of sa) and weight
    // rows e*N .. of B; only its first counts[e] tokens are real.  Dense:
    // counts == nullptr, cap == M.
    const int32_t *counts;
    int64_t cap;
    const float *sb;          // QX: weight block scales read directly
    int64_t ldsb;
};

// Shared memory of the small-M kernel.  Work goes in batches of up to GB K
// groups: one stage holds the weight and token tiles of a batch (one barrier
// handshake per batch), one scale slot their scales, one TMEM buffer their
// partials side by side.  A stage and a TMEM buffer hold XR token rows
// (columns) in all.  A batch has GB groups of NT token rows; with VAR (the
// masked layout, where the slot size NT is fixed but the expert's count is
// known only on the device) gb = min(GB, XR / n) groups of n token rows, n
// the count rounded up to 16.
template <int NT, int STAGES, int SC, int GB, bool QX = false>
struct SmallLayout {
    static constexpr int XR = GB * NT < 256 ? GB * NT : 256;  // token rows per stage / TMEM columns per buffer
    static constexpr size_t w_group = (size_t)BM * BK;        // 16 KB of weights per K group
    static constexpr size_t xb_group = QX ? (size_t)NT * BK * 2 : 0;   // tokens as BF16 (quantized in the kernel)
    static constexpr size_t w_bytes = GB * w_group;           // per stage (batch)
    static constexpr size_t x_bytes = (size_t)XR * BK;        // tokens, E4M3 (swizzled, read by the MMA)
    static constexpr size_t xb_bytes = GB * xb_group;
    static constexpr size_t off_w = 0;
    static constexpr size_t off_x = off_w + STAGES * w_bytes;
    static constexpr size_t off_xb = align_up(off_x + STAGES * x_bytes, 1024);
    static constexpr size_t sa_slot = align_up((size_t)GB * NT * 4, 128);   // [GB][NT] floats (a TMA box)
    static constexpr size_t sb_slot = align_up((size_t)GB * 16, 128);       // [GB][4] floats (a TMA box)
    // the split's FP32 partial [NT][128] reuses the stage memory after the
    // last K group (extended where the stages are smaller)
    static constexpr size_t part_bytes = (size_t)NT * BM * 4;
    static constexpr size_t stage_end = align_up(off_xb + STAGES * xb_bytes, 1024);
    static constexpr size_t off_sa = stage_end > part_bytes ? stage_end : part_bytes;
    static constexpr size_t off_sb = off_sa + (size_t)SC * sa_slot;
    static constexpr size_t off_bar = align_up(off_sb + (size_t)SC * sb_slot, 16);
    static constexpr int bufcols = XR;                         // TMEM columns of one batch's partials
    static_assert(!QX || GB * NT <= 256, "quantize-in-GEMM batches are whole");
    // as many TMEM buffers as fit (up to 8): the MMA runs that many batches ahead
    static constexpr int nbuf = (512 / bufcols) < 8 ? (512 / bufcols) : 8;
    static constexpr int num_bars = 2 * STAGES + 2 * SC + 2 * nbuf + 1 + (QX ? STAGES : SC);
    static constexpr size_t off_misc = off_bar + (size_t)num_bars * 8;
    static constexpr size_t total = off_misc + 16;
    static constexpr size_t dyn_bytes = total + 1024;
    static constexpr uint32_t tmem_cols = nbuf * bufcols < 32 ? 32 : nbuf * bufcols;   // power of two
    static_assert(dyn_bytes <= 227 * 1024, "shared memory");
};

// QX: the token operand arrives as BF16 and is quantized 1x128 inside the
// kernel (no E4M3 round trip through HBM): warps 2 and 3 turn each K group's
// BF16 token tile into the swizzled E4M3 tile the MMA reads and its scales,
// by the same rule and code as the quantization kernels (e4m3_rule.cuh).
template <int NT, int STAGES, int SC, int GB, bool OUT_F32, bool QX, bool VAR>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_smallm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                       const SmallParams p)
{
    using L = SmallLayout<NT, STAGES, SC, GB, QX>;
    constexpr int COLS = NT / 2;                 // token columns per promotion warp and K group
    constexpr int CH = COLS < 32 ? COLS : 32;    // columns per TMEM load
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
    uint8_t *sm_w = smem + L::off_w;
    uint8_t *sm_x = smem + L::off_x;
    uint8_t *sm_sa = smem + L::off_sa;
    uint8_t *sm_sb = smem + L::off_sb;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::off_bar);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *sc_full = bars + 2 * STAGES;
    uint64_t *sc_empty = bars + 2 * STAGES + SC;
    uint64_t *tm_full = bars + 2 * STAGES + 2 * SC;
    uint64_t *tm_empty = tm_full + L::nbuf;
    uint64_t *drain = tm_full + 2 * L::nbuf;
    uint64_t *qfull = drain + 1;                 // QX: stage s quantized (after full[s])
    uint64_t *pr_full = drain + 1;               // not QX: scale slot j holds the products sb * sa
    uint8_t *sm_xb = smem + L::off_xb;
    uint32_t *tmem_base_slot = reinterpret_cast<uint32_t *>(smem + L::off_misc);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + L::off_misc + 4);   // [0] abort, [1] partial ok

    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();
    const int32_t per_expert = p.n_tiles * p.S;
    const int32_t e = blockIdx.x / per_expert;   // expert (0 for a dense GEMM)
    const int32_t rem = blockIdx.x - e * per_expert;
    const int32_t tile = rem / p.S;              // 128 weight rows
    const int32_t split = rem - tile * p.S;
    int64_t m_real = p.M;                        // token columns that are written
    if (p.counts != nullptr) {
        int32_t c = __ldg(p.counts + e);
        c = c < 0 ? 0 : (c > p.cap ? (int32_t)p.cap : c);
        if (c == 0) return;                      // idle expert: its weights are not even read
        m_real = c;
    }
    // token columns actually computed: the real tokens rounded up to the MMA's
    // N granularity (16); loads, MMAs and promotion stop there
    const int32_t nt_run = m_real >= NT ? NT : (int32_t)((m_real + 15) / 16 * 16);
    const int32_t kb0 = (int32_t)((int64_t)split * p.KB / p.S);
    const int32_t kb1 = (int32_t)((int64_t)(split + 1) * p.KB / p.S);
    const int32_t ngroups = kb1 - kb0;
    // K groups per batch and the token rows (TMEM columns) of each group's tile
    const int32_t ncol = VAR ? nt_run : NT;
    const int32_t gb = VAR ? (L::XR / nt_run < GB ? L::XR / nt_run : GB) : GB;
    const uint32_t xg = (uint32_t)ncol * BK;
    const int32_t nbatch = (ngroups + gb - 1) / gb;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < SC; ++i) {
            mbar_init(&sc_full[i], QX ? 2 : 1);        // QX: one arrival per quantizer warp
            mbar_init(&sc_empty[i], kEpiWarps * 32);   // every promotion thread
        }
        if (QX)
            for (int i = 0; i < STAGES; ++i) mbar_init(&qfull[i], 2);
        else
            for (int i = 0; i < SC; ++i) mbar_init(&pr_full[i], 1);
        for (int i = 0; i < L::nbuf; ++i) {
            mbar_init(&tm_full[i], 1);
            mbar_init(&tm_empty[i], kEpiWarps * 32);
        }
        mbar_init(drain, 1);
        flags[0] = 0;
        flags[1] = 0;
        fence_barrier_init();
    }
    // one batch of weight and token tiles into stage b % STAGES
    auto issue_batch = [&](int32_t b) {
        const uint32_t s = b % STAGES;
        const int32_t gn = min(gb, ngroups - b * gb);
        mbar_arrive_expect_tx(&full[s], (uint32_t)(gn * (L::w_group + nt_run * BK * (QX ? 2 : 1))));
        for (int32_t jj = 0; jj < gn; ++jj) {
            const int32_t kx = (kb0 + b * gb + jj) * BK;
            tma_load_2d(sm_w + s * L::w_bytes + jj * L::w_group, &tmW, &full[s], kx, (int32_t)(e * p.N) + tile * BM);
            for (int32_t r = 0; r < nt_run; r += 16) {   // 16-row boxes: whole 128B-swizzle atoms
                if (QX)
                    tma_load_2d(sm_xb + s * L::xb_bytes + jj * L::xb_group + r * BK * 2, &tmX, &full[s], kx,
                                (int32_t)(e * p.cap) + r);
                else
                    tma_load_2d(sm_x + s * L::x_bytes + jj * xg + r * BK, &tmX, &full[s], kx,
                                (int32_t)(e * p.cap) + r);
            }
        }
    };
    // the scales of batch b: a (NT x GB) box of sa and a (4 x GB) box of the
    // weight tile's block scales from the batch's first K group (rows past
    // the batch are not used; boxes past the tensor read zeros)
    auto issue_scales = [&](int32_t b) {
        const uint32_t j = b % SC;
        mbar_arrive_expect_tx(&sc_full[j], (uint32_t)(GB * NT * 4 + GB * 16));
        tma_load_2d(sm_sa + j * L::sa_slot, &tmSA, &sc_full[j], (int32_t)(e * p.cap), kb0 + b * gb);
        tma_load_2d(sm_sb + j * L::sb_slot, &tmSB, &sc_full[j], tile & ~3, e * p.KB + kb0 + b * gb);
    };
    // The first batch goes out before the block-wide barrier (the TMEM
    // allocation runs meanwhile): its stage and scale slot are unused, and
    // this thread initialised the barriers they complete on.  (Issuing every
    // free stage here would hold the other warps at the barrier while the
    // TMA unit accepts the copies.)
    const int32_t pre_w = 1;
    const int32_t pre_s = QX ? 0 : 1;
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
        if (!QX) {
            tma_prefetch_desc(&tmSA);
            tma_prefetch_desc(&tmSB);
        }
        for (int32_t b = 0; b < pre_w; ++b) issue_batch(b);
        for (int32_t b = 0; b < pre_s; ++b) issue_scales(b);
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_base_slot, L::tmem_cols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_base_slot;
    volatile int *abort_flag = flags;
    // register split: the promotion warpgroups' increase below draws on what
    // the control warpgroup gives back here (128*40 + 256*232 <= 384*168)
    if (warp < kEpiWarp0) regs_decrease<kCtrlRegs>();

    // Waits on a stage, scale slot or TMEM buffer that has not been used yet
    // are skipped: its first phase counts as released.
    if (warp == kProducerWarp) {
        if (elect_one()) {
            for (int32_t b = pre_w; b < nbatch; ++b) {
                const uint32_t s = b % STAGES, ph = (b / STAGES) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1, abort_flag)) {
                    record_timeout(p.status, kSiteProducerEmpty);
                    *abort_flag = 1;
                    break;
                }
                issue_batch(b);
            }
        }
        __syncwarp();
    } else if (QX && (warp == kScaleWarp || warp == kScaleWarp + 1)) {
        // Quantize each K group's token tile: a warp takes two token rows per
        // pass (16 lanes x 8 values each), amax over the row by shuffles, the
        // codes into the 128B-swizzled E4M3 tile (16-byte chunk c of row r at
        // chunk c ^ (r & 7) of its 1024-byte atom), the scales into the ring.
        const int wq = (int)warp - kScaleWarp;
        const int c16 = (int)(lane & 15);
        bool ok = true;
        for (int32_t b = 0; b < nbatch; ++b) {
            const uint32_t s = b % STAGES, ph = (b / STAGES) & 1;
            const uint32_t j = b % SC, phj = (b / SC) & 1;
            if (!mbar_wait(&full[s], ph, abort_flag)) {
                record_timeout(p.status, kSiteQuantFull);
                ok = false;
                break;
            }
            if (b >= SC && !mbar_wait(&sc_empty[j], phj ^ 1, abort_flag)) {
                record_timeout(p.status, kSiteProducerScale);
                ok = false;
                break;
            }
            const int32_t gn = min(gb, ngroups - b * gb);
            float *sav = reinterpret_cast<float *>(sm_sa + j * L::sa_slot);
            for (int32_t jj = 0; jj < gn; ++jj) {
                const uint8_t *xb = sm_xb + s * L::xb_bytes + jj * L::xb_group;
                uint8_t *xq = sm_x + s * L::x_bytes + jj * xg;
                const float sbw = __ldg(p.sb + (int64_t)(e * p.KB + kb0 + b * gb + jj) * p.ldsb + tile);
                for (int32_t r0 = 0; r0 < nt_run; r0 += 4) {
                    const int r = r0 + 2 * wq + (int)(lane >> 4);
                    float f[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xb + r * (BK * 2) + c16 * 16), f);
                    float a = amax8(f);
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
                    const float sc = __fdiv_rn(a, kE4M3Max);
                    const uint2 c = encode8(f, make_divisor(sc));
                    uint8_t *row = xq + (r >> 3) * 1024 + (r & 7) * 128;
                    *reinterpret_cast<uint2 *>(row + (((c16 >> 1) ^ (r & 7)) * 16) + (c16 & 1) * 8) = c;
                    if (c16 == 0) sav[jj * NT + r] = sbw * sc;   // the promotion's scale of this token
                }
            }
            fence_proxy_async_smem();     // E4M3 tiles -> the MMA; BF16 stage -> its next TMA refill
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&qfull[s]);
                mbar_arrive(&sc_full[j]);
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (!QX && warp == kScaleWarp + 1) {
        // The promotion's per-token scale of each K group, sb(weight block) *
        // sa(token), formed once per CTA in place in the scale slot (instead of
        // once per weight row by every promotion thread).
        for (int32_t b = 0; b < nbatch; ++b) {
            const uint32_t j = b % SC, phj = (b / SC) & 1;
            if (!mbar_wait(&sc_full[j], phj, abort_flag)) {
                record_timeout(p.status, kSiteEpiScale);
                *abort_flag = 1;
                break;
            }
            const int32_t gn = min(gb, ngroups - b * gb);
            float *sav = reinterpret_cast<float *>(sm_sa + j * L::sa_slot);
            const float *sbv = reinterpret_cast<const float *>(sm_sb + j * L::sb_slot);
            for (int32_t jj = 0; jj < gn; ++jj) {
                const float sbw = sbv[jj * 4 + (tile & 3)];
                for (int32_t t = (int32_t)lane; t < nt_run; t += 32) sav[jj * NT + t] = sbw * sav[jj * NT + t];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&pr_full[j]);
        }
    } else if (!QX && warp == kScaleWarp) {
        if (elect_one()) {
            for (int32_t b = pre_s; b < nbatch; ++b) {
                const uint32_t j = b % SC, phj = (b / SC) & 1;
                if (!mbar_wait(&sc_empty[j], phj ^ 1, abort_flag)) {
                    record_timeout(p.status, kSiteProducerScale);
                    *abort_flag = 1;
                    break;
                }
                issue_scales(b);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        const uint32_t idesc = idesc_e4m3_f32(BM, (uint32_t)nt_run);
        bool ok = true;
        for (int32_t b = 0; b < nbatch; ++b) {
            const uint32_t s = b % STAGES, ph = (b / STAGES) & 1;
            const uint32_t buf = b % L::nbuf, phb = (b / L::nbuf) & 1;
            if (!mbar_wait(QX ? &qfull[s] : &full[s], ph, abort_flag)) {
                record_timeout(p.status, kSiteMmaFull);
                ok = false;
                break;
            }
            if (b >= L::nbuf && !mbar_wait(&tm_empty[buf], phb ^ 1, abort_flag)) {
                record_timeout(p.status, kSiteMmaTmemEmpty);
                ok = false;
                break;
            }
            tc_fence_after_sync();
            if (elect_one()) {
                const int32_t gn = min(gb, ngroups - b * gb);
                for (int32_t jj = 0; jj < gn; ++jj) {
                    const uint64_t dw = smem_desc_kmajor_sw128(sm_w + s * L::w_bytes + jj * L::w_group);
                    const uint64_t dx = smem_desc_kmajor_sw128(sm_x + s * L::x_bytes + jj * xg);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_e4m3(tmem_base + buf * L::bufcols + jj * ncol, dw + 2 * k, dx + 2 * k, idesc,
                                 k > 0 ? 1u : 0u);
                }
                mma_commit(&empty[s]);
                mma_commit(&tm_full[buf]);
            }
            __syncwarp();
        }
        if (!ok) *abort_flag = 1;
        if (elect_one()) mma_commit(drain);
        __syncwarp();
        mbar_wait(drain, 0, nullptr, 20u * 1000u * 1000u);
    } else if (warp >= kEpiWarp0) {
        regs_increase<kEpiRegs>();
        const uint32_t quarter = warp & 3;
        const uint32_t half = (warp - kEpiWarp0) >> 2;
        const uint32_t wrow = quarter * 32 + lane;              // weight row in the tile
        const uint32_t lane_addr = (quarter * 32) << 16;
        const uint32_t col0 = half * COLS;                      // first token column
        float2 acc[COLS / 2];
#pragma unroll
        for (int i = 0; i < COLS / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);
        bool ok = true;
        for (int32_t b = 0; b < nbatch; ++b) {
            const uint32_t j = b % SC, phj = (b / SC) & 1;
            if (!mbar_wait(QX ? &sc_full[j] : &pr_full[j], phj, abort_flag)) {
                record_timeout(p.status, kSiteEpiScale);
                ok = false;
                break;
            }
            const uint32_t buf = b % L::nbuf, phb = (b / L::nbuf) & 1;
            if (!mbar_wait(&tm_full[buf], phb, abort_flag)) {
                record_timeout(p.status, kSiteEpiTmemFull);
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const int32_t gn = min(gb, ngroups - b * gb);
            // per token: sb(weight block) * sa(token), the same for every weight row
            const float *scl = reinterpret_cast<const float *>(sm_sa + j * L::sa_slot);
#pragma unroll
            for (int jj = 0; jj < GB; ++jj) {
                if (jj >= gn) break;                            // warp-uniform
#pragma unroll
                for (int c = 0; c < COLS; c += CH) {
                    if ((int32_t)(col0 + c) >= nt_run) break;  // no token columns left (warp-uniform)
                    uint32_t r[CH];
                    tmem_ld_sync<CH>(tmem_base + lane_addr + buf * L::bufcols + jj * ncol + col0 + c, r);
#pragma unroll
                    for (int i = 0; i < CH / 4; ++i) {
                        const float4 s4 = *reinterpret_cast<const float4 *>(scl + jj * NT + col0 + c + 4 * i);
                        const float2 p0 = make_float2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]));
                        const float2 p1 = make_float2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                        acc[c / 2 + 2 * i] = __ffma2_rn(p0, make_float2(s4.x, s4.y), acc[c / 2 + 2 * i]);
                        acc[c / 2 + 2 * i + 1] = __ffma2_rn(p1, make_float2(s4.z, s4.w), acc[c / 2 + 2 * i + 1]);
                    }
                }
            }
            fence_proxy_async_smem();         // scale slot j is refilled by TMA once released
            tc_fence_before_sync();
            mbar_arrive(&tm_empty[buf]);
            mbar_arrive(&sc_empty[j]);
        }
        if (!ok) *abort_flag = 1;
        const int64_t n = (int64_t)tile * BM + wrow;
        if (ok && p.S == 1) {
            if (n < p.N) {
#pragma unroll
                for (int i = 0; i < COLS / 2; ++i) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int64_t m = col0 + 2 * i + h;
                        const float v = h ? acc[i].y : acc[i].x;
                        if (m < m_real) {
                            const int64_t row = e * p.cap + m;
                            if (OUT_F32) static_cast<float *>(p.C)[row * p.ldc + n] = v;
                            else static_cast<__nv_bfloat16 *>(p.C)[row * p.ldc + n] = __float2bfloat16_rn(v);
                        }
                    }
                }
            }
        } else if (p.S > 1) {
            // this split's partial, [token column][weight row], into this CTA's
            // stage memory: every TMA load into it has landed and every MMA
            // reading it has completed (the last tm_full wait above)
            float *part = reinterpret_cast<float *>(smem + L::off_w);
            if (ok) {
#pragma unroll
                for (int i = 0; i < COLS / 2; ++i) {
                    part[(col0 + 2 * i) * BM + wrow] = acc[i].x;
                    part[(col0 + 2 * i + 1) * BM + wrow] = acc[i].y;
                }
            }
            // all eight promotion warps done, none gave up?
            const bool mine_ok = named_barrier_and(1, kEpiWarps * 32, ok && !*abort_flag);
            if (threadIdx.x == kEpiWarp0 * 32) flags[1] = mine_ok ? 1 : 0;
            // Split-K reduction across the cluster.  Every thread of every CTA
            // in the cluster passes both cluster barriers (the other warps at
            // the end of the kernel); the CTAs of one cluster share the
            // expert, so an idle expert's CTAs have all returned above.
            __syncwarp();
            cluster_sync();                      // partials and ok flags visible cluster-wide
            uint32_t peer[kMaxSplits];
            int32_t peer_ok[kMaxSplits];
#pragma unroll
            for (int q = 0; q < kMaxSplits; ++q) {
                if (q < p.S) {
                    peer[q] = cluster_map(smem + L::off_w, (uint32_t)q);
                    peer_ok[q] = ld_cluster_s32(cluster_map((const void *)&flags[1], (uint32_t)q));
                }
            }
            bool all_ok = true;
#pragma unroll
            for (int q = 0; q < kMaxSplits; ++q)
                if (q < p.S) all_ok = all_ok && peer_ok[q] != 0;
            if (all_ok) {
                // slice `split` of the computed float4s (four outputs each),
                // summed over the splits in order; kRedUnroll float4s of every
                // split in flight per thread
                constexpr int kRedUnroll = 4;
                constexpr int kStride = kEpiWarps * 32;
                const int E4 = nt_run * BM / 4;
                const int lo = split * E4 / p.S, hi = (split + 1) * E4 / p.S;
                const int t = (int)threadIdx.x - kEpiWarp0 * 32;   // 0 .. 255
                for (int e0 = lo + t; e0 < hi; e0 += kStride * kRedUnroll) {
                    float4 v[kRedUnroll][kMaxSplits];
#pragma unroll
                    for (int u = 0; u < kRedUnroll; ++u) {
                        const int e4 = e0 + u * kStride;
#pragma unroll
                        for (int q = 0; q < kMaxSplits; ++q)
                            if (q < p.S && e4 < hi) v[u][q] = ld_cluster_f4(peer[q] + (uint32_t)e4 * 16u);
                    }
#pragma unroll
                    for (int u = 0; u < kRedUnroll; ++u) {
                        const int e4 = e0 + u * kStride;
                        if (e4 >= hi) break;
                        float4 sum = v[u][0];
#pragma unroll
                        for (int q = 1; q < kMaxSplits; ++q) {
                            if (q < p.S) {
                                sum.x += v[u][q].x;
                                sum.y += v[u][q].y;
                                sum.z += v[u][q].z;
                                sum.w += v[u][q].w;
                            }
                        }
                        const int col = (e4 * 4) / BM, r = e4 * 4 - col * BM;
                        const int64_t n = (int64_t)tile * BM + r;
                        if (col >= m_real || n >= p.N) continue;   // N % 16 == 0: all four in or out
                        const int64_t row = e * p.cap + col;
                        if (OUT_F32) {
                            *reinterpret_cast<float4 *>(static_cast<float *>(p.C) + row * p.ldc + n) = sum;
                        } else {
                            const __nv_bfloat162 lo2 = __floats2bfloat162_rn(sum.x, sum.y);
                            const __nv_bfloat162 hi2 = __floats2bfloat162_rn(sum.z, sum.w);
                            uint2 o;
                            memcpy(&o.x, &lo2, 4);
                            memcpy(&o.y, &hi2, 4);
                            *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.C) + row * p.ldc + n) = o;
                        }
                    }
                }
            }
            __syncwarp();
            cluster_sync();                      // no CTA leaves while a peer still reads its partial
        }
    }
    if (p.S > 1 && warp < kEpiWarp0) {
        // the control warps' part in the two cluster barriers of the reduction
        __syncwarp();
        cluster_sync();
        cluster_sync();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, L::tmem_cols);
    }
}

// ------------------------------------------------------------------------
// Accumulation-precision probe: one CTA, D = A * B^T chained over all of K
// in one TMEM accumulator (no promotion), raw FP32 written out.
// ------------------------------------------------------------------------
constexpr int kProbeMaxN = 256;
constexpr int kProbeThreads = 256;      // warp 0 loads, warp 1 issues MMAs, warps 4..7 read TMEM

__global__ void __launch_bounds__(kProbeThreads, 1)
    mma_probe_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, float *D, int N,
                     int K, DeviceStatus *status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
    uint8_t *sm_a = smem;                         // 16 KB
    uint8_t *sm_b = smem + BM * BK;               // up to 32 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + BM * BK + kProbeMaxN * BK);
    uint64_t *full = bars, *done = bars + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);
    const uint32_t warp = warp_id(), lane = lane_id();

    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        mbar_init(done, 1);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, kProbeMaxN);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    __shared__ int ok_all;
    if (threadIdx.x == 0) ok_all = 1;
    __syncthreads();

    const int KB = K / BK;
    for (int kb = 0; kb < KB; ++kb) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(full, (uint32_t)(BM * BK + N * BK));
            tma_load_2d(sm_a, &tmA, full, kb * BK, 0);
            tma_load_2d(sm_b, &tmB, full, kb * BK, 0);
        }
        if (warp == kMmaWarp) {
            bool ok = mbar_wait(full, kb & 1, nullptr);
            if (ok) {
                tc_fence_after_sync();
                if (elect_one()) {
                    const uint64_t da = smem_desc_kmajor_sw128(sm_a);
                    const uint64_t db = smem_desc_kmajor_sw128(sm_b);
                    const uint32_t idesc = idesc_e4m3_f32(BM, N);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k) mma_e4m3(tmem, da + 2 * k, db + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    mma_commit(done);
                }
                __syncwarp();
                ok = mbar_wait(done, kb & 1, nullptr);
            }
            if (!ok && lane == 0) {
                record_timeout(status, kSiteProbe);
                ok_all = 0;
            }
        }
        __syncthreads();                 // stage buffers are reused next iteration
        if (!ok_all) break;
    }
    if (warp >= kEpiWarp0 && ok_all) {
        tc_fence_after_sync();
        const uint32_t quarter = warp - kEpiWarp0;
        const uint32_t row = quarter * 32 + lane;
        for (int c = 0; c < N; c += 32) {
            uint32_t r[32];
            tmem_ld_sync<32>(tmem + ((quarter * 32) << 16) + c, r);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (c + i < N) D[(int64_t)row * N + c + i] = __uint_as_float(r[i]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kProbeMaxN);
    }
}

// A wait on a barrier that nothing arrives on: exercises the bounded-wait
// path (status word set, TMEM released, kernel returns) without any fault.
__global__ void wait_timeout_selftest_kernel(DeviceStatus *status, uint64_t budget_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_slot;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    tmem_alloc(&tmem_slot, 32);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const bool ok = mbar_wait(&bar, 0, nullptr, budget_ns);
    if (!ok && threadIdx.x == 0) record_timeout(status, kSiteSelftest);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    tmem_dealloc(tmem_slot, 32);
}

// ------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

template <int BN, int STAGES, int SG, int SS, bool ROW_SB, bool OUT_F32, int MC = 1>
cudaError_t launch_variant(const GemmArgs &a, const Params &p, int grid, cudaStream_t stream)
{
    using L = Layout<BN, STAGES, SG, SS, ROW_SB>;
    CUtensorMap tmA, tmB;
    const int64_t b_rows = a.m_indices ? (int64_t)a.num_experts * a.N : a.N;
    // with multicast each CTA of a cluster loads one of MC row slices of the B panel
    if (!make_tensor_map_2d(&tmA, 1, false, a.A, a.K, a.M, a.K, BK, BM, true) ||
        !make_tensor_map_2d(&tmB, 1, false, a.B, a.K, b_rows, a.K, BK, BN / MC, true))
        return cudaErrorInvalidValue;
    auto kern = gemm_blockscaled_kernel<BN, STAGES, SG, SS, ROW_SB, OUT_F32, MC>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::dyn_bytes);
    if (err != cudaSuccess) return err;
    if (MC == 1) {
        kern<<<grid, kThreads, L::dyn_bytes, stream>>>(tmA, tmB, p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::dyn_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = MC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p);
}

std::atomic<int> g_mc_clusters[64];          // concurrent clusters of the multicast variant per device (0: not yet known)

}  // namespace

// Concurrent clusters of two of the multicast variant on the current device
// (looked up once per device; 0 if it cannot run).
int mc_max_clusters()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (g_mc_clusters[dev].load(std::memory_order_relaxed) == 0) {
        using L = Layout<256, 4, 8, 3, false>;
        auto kern = gemm_blockscaled_kernel<256, 4, 8, 3, false, false, 2>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::dyn_bytes) !=
            cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = L::dyn_bytes;
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
            g_mc_clusters[dev].store(-1, std::memory_order_relaxed);
        } else {
            g_mc_clusters[dev].store(n, std::memory_order_relaxed);
        }
    }
    const int n = g_mc_clusters[dev].load(std::memory_order_relaxed);
    return n > 0 ? n : 0;
}

bool make_tensor_map_2d(void *map, int dtype_bytes, bool is_float, const void *base, uint64_t inner, uint64_t outer,
                        uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128)
{
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const CUtensorMapDataType dt =
        dtype_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
        : dtype_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
        : (is_float ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_INT32);
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(reinterpret_cast<CUtensorMap *>(map), dt, 2, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

// Token columns of the small-M kernel: M rounded up to 16, 32, 64, 128 or 256.
int small_nt(int64_t M)
{
    return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
}

// Dense GEMMs with up to 128 tokens and few weight tiles take the small-M
// kernel.  From 129 tokens on, the 128 x 256 tiles of the large kernel (token
// scale per row, one paired FMA per two elements, last-wave split along K)
// are faster on the B300: 256 x 4096 x 7168 in 19.4 us instead of 24.3 us,
// 256 x 7168 x 2048 in 11.7 us instead of 18.1 us; at 128 tokens the small-M
// kernel still wins (15.0 us against 16.5 us for 128 x 4096 x 7168).
bool use_small_m(int64_t M, int64_t N, int32_t num_experts_or_dense, int num_sms)
{
    (void)num_experts_or_dense;
    return M <= 128 && (N + BM - 1) / BM <= (num_sms > 0 ? num_sms / 2 : 74);
}

int g_small_splits = 0;     // testing: forced split count of the dense small-M kernel (0: planner)

int small_splits(int64_t N, int64_t K, int num_sms)
{
    const int64_t tiles = (N + BM - 1) / BM, KB = K / BK;
    if (g_small_splits > 0) return (int)(g_small_splits < KB ? g_small_splits : KB);
    int64_t S = (num_sms > 0 ? num_sms : 148) / tiles;
    if (S > kMaxSplits) S = kMaxSplits;
    if (S > KB) S = KB;
    return S < 1 ? 1 : (int)S;
}

// Split count of the masked layout and the last-wave split's grid, from the
// B300's 148 SMs rather than the device's, so that the workspace size a caller
// queries and the launch agree.
constexpr int kNominalSms = 148;

// Last-wave split of a dense GEMM: with W = tiles / G whole waves, the
// R = tiles mod G tail tiles are cut into s K pieces each (R * s <= G, one
// round).  Cost in K-group steps of one tile: ceil(KB / s) for the pieces,
// plus about two steps per 128 x BN FP32 partial that the last piece reads
// back from L2 and one to store its own; s = 1 (no split) costs KB.
struct TailPlan {
    int32_t dp_tiles, s;
    int64_t cost;               // K-group steps of the whole schedule on one CTA
};

TailPlan plan_tail(const GemmArgs &a, int64_t tiles, int64_t KB, int G, bool ws_ok)
{
    const int64_t W = tiles / G, R = tiles % G;
    TailPlan t{(int32_t)tiles, 1, (W + (R > 0 ? 1 : 0)) * KB};
    if (a.m_indices != nullptr || a.counts != nullptr || R == 0 || !ws_ok) return t;
    for (int64_t s = 2; s <= KB && R * s <= G; ++s) {
        const int64_t c = W * KB + (KB + s - 1) / s + 2 * s + 1;
        if (c < t.cost) t = TailPlan{(int32_t)(W * G), (int32_t)s, c};
    }
    return t;
}

// Status header, counters (one per tail tile, fewer than 148) and up to 148
// FP32 partial tiles of 128 x BN.
static_assert(kNominalSms <= kMaxCounters, "one counter per tail tile");
size_t tail_workspace_bytes(int BN)
{
    return kWsPartialsOffset + (size_t)kNominalSms * BM * BN * 4;
}
int masked_splits(int32_t E, int64_t n_tiles, int64_t KB)
{
    int64_t S = kNominalSms / ((int64_t)E * n_tiles);
    if (S > kMaxSplits) S = kMaxSplits;
    if (S > KB) S = KB;
    return S < 1 ? 1 : (int)S;
}

}  // namespace

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t num_experts, int)
{
    size_t bytes = gemm_workspace_min_bytes(M, N, K, num_experts);
    // room for the last-wave split with 128 x 256 tiles
    if (num_experts <= 1 && tail_workspace_bytes(256) > bytes) bytes = tail_workspace_bytes(256);
    return bytes;
}

size_t gemm_workspace_min_bytes(int64_t, int64_t, int64_t, int32_t)
{
    // whole tiles, and the small-M split (reduced within its cluster), need
    // the status header alone
    return kWsHeaderBytes;
}

size_t masked_workspace_bytes(int32_t, int64_t, int64_t, int64_t)
{
    return kWsHeaderBytes;
}

size_t gemm_workspace_zeroed_bytes(int64_t, int64_t, int64_t, int32_t)
{
    // status word and the arrival counters
    return kWsPartialsOffset;
}

namespace {

// A panels that a band of the n-outer walk keeps in the 126 MB L2 (with room
// for the B panels and output passing through).
constexpr int64_t kBandBytes = 48ll << 20;

template <int BN, int MC = 1>
Params make_params(const GemmArgs &a)
{
    Params p{};
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.KB = (int32_t)(a.K / BK);
    p.m_blocks = (int32_t)((a.M + BM - 1) / BM);
    p.num_m_blocks = (p.m_blocks + MC - 1) / MC;
    p.num_n_blocks = (int32_t)((a.N + BN - 1) / BN);
    p.num_tiles = p.num_m_blocks * p.num_n_blocks;
    p.m_major = a.m_indices != nullptr ? 1 : 0;
    // Bands of M blocks whose A panels take at most kBandBytes, as even as
    // possible: the down projection 4096 x 7168 x 18432 (A 75.5 MB) walks two
    // bands, reading A once and B twice instead of A once per wave.
    {
        const int64_t a_bytes = (int64_t)p.m_blocks * BM * a.K;
        const int64_t nbands = (a_bytes + kBandBytes - 1) / kBandBytes;
        p.band = (int32_t)((p.num_m_blocks + nbands - 1) / nbands);
    }
    p.C = a.C;
    p.ldc = a.ldc;
    p.m_indices = a.m_indices;
    p.b_rows_per_expert = a.m_indices ? a.N : 0;
    p.sb_rows_per_expert = a.m_indices ? p.KB : 0;
    p.status = reinterpret_cast<DeviceStatus *>(a.workspace);
    p.sa = a.sa;
    p.sb = a.sb;
    p.ldsa = a.ldsa;
    p.ldsb = a.ldsb;
    return p;
}

template <int BN, int STAGES>
cudaError_t launch_bn(const GemmArgs &a, cudaStream_t stream, int num_sms)
{
    Params p = make_params<BN>(a);
    int grid = p.num_tiles < num_sms ? p.num_tiles : num_sms;
    if (grid <= 0) return cudaSuccess;
    const int G = num_sms < kNominalSms ? num_sms : kNominalSms;
    const TailPlan t = plan_tail(a, p.num_tiles, p.KB, G, a.ws_bytes >= tail_workspace_bytes(BN));
    p.dp_tiles = t.dp_tiles;
    if (t.s > 1) {
        const int32_t units = (p.num_tiles - t.dp_tiles) * t.s;
        grid = t.dp_tiles > 0 ? G : units;
        p.tail_s = t.s;
        p.tail_units = units;
        uint8_t *ws = static_cast<uint8_t *>(a.workspace);
        p.tail_tickets = reinterpret_cast<uint32_t *>(ws + kWsHeaderBytes);
        p.tail_partials = reinterpret_cast<float *>(ws + kWsPartialsOffset);
    }
    // block scales: slots of 8 K groups; per-row B scales (BN floats per
    // group): slots of 4
    if (a.bkind == 1)
        return a.out_f32 ? launch_variant<BN, STAGES, 4, 3, true, true>(a, p, grid, stream)
                         : launch_variant<BN, STAGES, 4, 3, true, false>(a, p, grid, stream);
    return a.out_f32 ? launch_variant<BN, STAGES, 8, 3, false, true>(a, p, grid, stream)
                     : launch_variant<BN, STAGES, 8, 3, false, false>(a, p, grid, stream);
}

// Clusters of two vertically adjacent 128 x 256 tiles sharing the B panel by
// TMA multicast (dense GEMMs, 128x128 block B scales), the last wave split
// along K over clusters as launch_bn does over CTAs.
cudaError_t launch_multicast(const GemmArgs &a, cudaStream_t stream)
{
    Params p = make_params<256, 2>(a);
    const int G = mc_max_clusters();
    if (G <= 0) return cudaErrorNotSupported;
    int clusters = p.num_tiles < G ? p.num_tiles : G;
    if (clusters <= 0) return cudaSuccess;
    const TailPlan t = plan_tail(a, p.num_tiles, p.KB, G, a.ws_bytes >= tail_workspace_bytes(256));
    p.dp_tiles = t.dp_tiles;
    if (t.s > 1) {
        const int32_t units = (p.num_tiles - t.dp_tiles) * t.s;
        clusters = t.dp_tiles > 0 ? G : units;
        p.tail_s = t.s;
        p.tail_units = units;
        uint8_t *ws = static_cast<uint8_t *>(a.workspace);
        p.tail_tickets = reinterpret_cast<uint32_t *>(ws + kWsHeaderBytes);
        p.tail_partials = reinterpret_cast<float *>(ws + kWsPartialsOffset);
    }
    const int grid = 2 * clusters;
    return a.out_f32 ? launch_variant<256, 4, 8, 3, false, true, 2>(a, p, grid, stream)
                     : launch_variant<256, 4, 8, 3, false, false, 2>(a, p, grid, stream);
}

template <int NT, int STAGES, int SC, int GB, bool OUT_F32, bool QX = false, bool VAR = false>
cudaError_t launch_small(const GemmArgs &a, cudaStream_t stream, int num_sms)
{
    using L = SmallLayout<NT, STAGES, SC, GB, QX>;
    SmallParams p{};
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.KB = (int32_t)(a.K / BK);
    p.n_tiles = (int32_t)((a.N + BM - 1) / BM);
    const int32_t E = a.counts != nullptr ? a.num_experts : 1;
    p.S = a.counts != nullptr ? masked_splits(E, p.n_tiles, p.KB) : small_splits(a.N, a.K, num_sms);
    p.C = a.C;
    p.ldc = a.ldc;
    p.counts = a.counts;
    p.cap = a.counts != nullptr ? a.cap : a.M;
    p.sb = a.sb;
    p.ldsb = a.ldsb;
    p.status = reinterpret_cast<DeviceStatus *>(a.workspace);
    CUtensorMap tmW, tmX, tmSA, tmSB;
    memset(&tmSA, 0, sizeof(tmSA));
    memset(&tmSB, 0, sizeof(tmSB));
    if (!make_tensor_map_2d(&tmW, 1, false, a.B, a.K, (uint64_t)E * a.N, a.K, BK, BM, true))
        return cudaErrorInvalidValue;
    if (QX) {
        // BF16 tokens, plain row-major 16 x 128 boxes (the kernel quantizes them)
        if (!make_tensor_map_2d(&tmX, 2, false, a.xbf16, a.K, (uint64_t)E * p.cap, a.ldx * 2, BK, 16, false))
            return cudaErrorInvalidValue;
    } else if (!make_tensor_map_2d(&tmX, 1, false, a.A, a.K, (uint64_t)E * p.cap, a.K, BK, 16, true) ||
               !make_tensor_map_2d(&tmSA, 4, true, a.sa, a.ldsa, p.KB, a.ldsa * 4, NT, GB, false) ||
               !make_tensor_map_2d(&tmSB, 4, true, a.sb, a.ldsb, (uint64_t)E * p.KB, a.ldsb * 4, 4, GB, false)) {
        return cudaErrorInvalidValue;
    }
    auto kern = gemm_smallm_kernel<NT, STAGES, SC, GB, OUT_F32, QX, VAR>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::dyn_bytes);
    if (err != cudaSuccess) return err;
    // the S splits of a weight tile: one cluster of S consecutive CTAs
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(E * p.n_tiles * p.S));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::dyn_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmW, tmX, tmSA, tmSB, p);
}

template <bool OUT_F32>
cudaError_t launch_small_nt(const GemmArgs &a, cudaStream_t stream, int num_sms)
{
    switch (small_nt(a.M)) {
    // <tokens, stages, scale slots, K groups per batch>: batches of 4 K groups
    // (2 and 1 where four partials would not fit in tensor memory), stages
    // up to ~220 KB of shared memory
    case 16: return launch_small<16, 3, 4, 4, OUT_F32>(a, stream, num_sms);
    case 32: return launch_small<32, 2, 4, 4, OUT_F32>(a, stream, num_sms);
    case 64: return launch_small<64, 2, 4, 4, OUT_F32>(a, stream, num_sms);
    case 128: return launch_small<128, 3, 4, 2, OUT_F32>(a, stream, num_sms);
    default: return launch_small<256, 4, 8, 1, OUT_F32>(a, stream, num_sms);
    }
}

// Tile width: 256 columns unless 128-column tiles fill the SMs' last wave
// enough better to pay for their lower per-tile efficiency.
int choose_bn(const GemmArgs &a, int num_sms)
{
    // K-group steps on one CTA, a 128 x 256 step costing about 2 / 1.15 times
    // a 128 x 128 one
    const int G = num_sms < kNominalSms ? num_sms : kNominalSms;
    const int64_t mb = (a.M + BM - 1) / BM, KB = a.K / BK;
    const TailPlan t256 = plan_tail(a, mb * ((a.N + 255) / 256), KB, G, a.ws_bytes >= tail_workspace_bytes(256));
    const TailPlan t128 = plan_tail(a, mb * ((a.N + 127) / 128), KB, G, a.ws_bytes >= tail_workspace_bytes(128));
    return (double)t128.cost * 1.15 < (double)t256.cost * 2.0 ? 128 : 256;
}

}  // namespace

// The CTA-pair kernel (gemm_pair.cu) serves dense GEMMs with 128x128 block
// scales and at least two 128-row blocks only when it has been switched on
// (fgf8_testing_set_pair): on the B300 it is slower than the 128 x 256
// single-SM tile on every shape measured, so the planner does not pick it.
int g_pair_mode = 0;

bool use_pair(const GemmArgs &a)
{
    return g_pair_mode == 1 && a.m_indices == nullptr && a.counts == nullptr && a.bkind == 0 && a.M > BM;
}

// Mode 2: dense block-scaled GEMMs of more than 128 rows run the 128 x 256
// kernel in clusters of two that share B by TMA multicast.
bool use_multicast(const GemmArgs &a)
{
    return g_pair_mode == 2 && a.m_indices == nullptr && a.counts == nullptr && a.bkind == 0 && a.M > BM;
}

void set_pair_mode(int mode)
{
    g_pair_mode = mode;
}

void set_small_splits(int s)
{
    g_small_splits = s;
}

GemmSchedule gemm_schedule(const GemmArgs &a, int num_sms)
{
    GemmSchedule g{};
    if (a.m_indices == nullptr && a.bkind == 0 && use_small_m(a.M, a.N, 1, num_sms)) {
        g.small_m = 1;
        g.tail_s = small_splits(a.N, a.K, num_sms);
        return g;
    }
    if (use_pair(a)) {
        const PairPlan pl = pair_plan(a, num_sms / 2);
        g.pair = 1;
        g.bn = pair_tile_n();
        g.dp_tiles = pl.dp_tiles;
        g.tail_s = pl.tail_s;
        return g;
    }
    if (use_multicast(a)) {
        const int64_t tiles = ((a.M + 2 * BM - 1) / (2 * BM)) * ((a.N + 255) / 256);
        const TailPlan t = plan_tail(a, tiles, a.K / BK, num_sms / 2, a.ws_bytes >= tail_workspace_bytes(256));
        g.pair = 2;
        g.bn = 256;
        g.dp_tiles = t.dp_tiles;
        g.tail_s = t.s;
        return g;
    }
    g.bn = choose_bn(a, num_sms);
    const int G = num_sms < kNominalSms ? num_sms : kNominalSms;
    const int64_t tiles = ((a.M + BM - 1) / BM) * ((a.N + g.bn - 1) / g.bn);
    const TailPlan t = plan_tail(a, tiles, a.K / BK, G, a.ws_bytes >= tail_workspace_bytes(g.bn));
    g.dp_tiles = t.dp_tiles;
    g.tail_s = t.s;
    return g;
}

size_t gemm_required_bytes(const GemmArgs &a, int num_sms)
{
    const GemmSchedule g = gemm_schedule(a, num_sms);
    if (g.tail_s > 1) return g.pair == 1 ? pair_tail_workspace_bytes() : tail_workspace_bytes(g.bn);
    return kWsHeaderBytes;
}

cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t stream, int num_sms)
{
    // Few tokens: weights on the MMA's M side, K split across the SMs.
    if (a.m_indices == nullptr && a.bkind == 0 && use_small_m(a.M, a.N, 1, num_sms))
        return a.out_f32 ? launch_small_nt<true>(a, stream, num_sms) : launch_small_nt<false>(a, stream, num_sms);
    if (use_pair(a)) {
        const cudaError_t e = launch_pair(a, stream);
        if (e != cudaErrorNotSupported) return e;
    }
    if (use_multicast(a)) {
        const cudaError_t e = launch_multicast(a, stream);
        if (e != cudaErrorNotSupported) return e;
    }
    if (choose_bn(a, num_sms) == 128) return launch_bn<128, 6>(a, stream, num_sms);
    return launch_bn<256, 4>(a, stream, num_sms);
}

namespace {
// Masked layout: the slot capacity fixes the layout, the expert's count (on
// the device) the token rows computed.  Up to four K groups per batch, as
// many as the 256 token rows of a stage and a TMEM buffer hold at the
// expert's count (a full 256-row slot: one).
template <bool OUT_F32>
cudaError_t launch_masked_cap(const GemmArgs &a, cudaStream_t stream, int num_sms)
{
    switch (small_nt(a.cap)) {
    case 16: return launch_small<16, 3, 3, 4, OUT_F32, false, true>(a, stream, num_sms);
    case 32: return launch_small<32, 2, 4, 4, OUT_F32, false, true>(a, stream, num_sms);
    case 64: return launch_small<64, 2, 4, 4, OUT_F32, false, true>(a, stream, num_sms);
    case 128: return launch_small<128, 2, 4, 4, OUT_F32, false, true>(a, stream, num_sms);
    default: return launch_small<256, 2, 4, 4, OUT_F32, false, true>(a, stream, num_sms);
    }
}
}  // namespace

cudaError_t launch_masked(const GemmArgs &a, cudaStream_t stream, int num_sms)
{
    return a.out_f32 ? launch_masked_cap<true>(a, stream, num_sms) : launch_masked_cap<false>(a, stream, num_sms);
}

namespace {
template <bool OUT_F32>
cudaError_t launch_small_qx(const GemmArgs &a, cudaStream_t stream, int num_sms)
{
    // stages so that the BF16 token staging fits next to the E4M3 tiles
    // (the BF16 staging tile of 128 and 256 tokens takes 32 and 64 KB per K
    // group: one group per stage, three stages and one)
    switch (small_nt(a.M)) {
    case 16: return launch_small<16, 2, 4, 4, OUT_F32, true>(a, stream, num_sms);
    case 32: return launch_small<32, 3, 4, 2, OUT_F32, true>(a, stream, num_sms);
    case 64: return launch_small<64, 2, 4, 2, OUT_F32, true>(a, stream, num_sms);
    case 128: return launch_small<128, 3, 4, 1, OUT_F32, true>(a, stream, num_sms);
    default: return launch_small<256, 1, 4, 1, OUT_F32, true>(a, stream, num_sms);
    }
}
}  // namespace

cudaError_t launch_bf16a(const GemmArgs &a, cudaStream_t stream, int num_sms)
{
    return a.out_f32 ? launch_small_qx<true>(a, stream, num_sms) : launch_small_qx<false>(a, stream, num_sms);
}

cudaError_t launch_mma_probe(const uint8_t *A, const uint8_t *B, float *D, int N, int K, void *workspace,
                             cudaStream_t stream)
{
    CUtensorMap tmA, tmB;
    if (!make_tensor_map_2d(&tmA, 1, false, A, K, BM, K, BK, BM, true) ||
        !make_tensor_map_2d(&tmB, 1, false, B, K, N, K, BK, N, true))
        return cudaErrorInvalidValue;
    const size_t smem = 1024 + BM * BK + kProbeMaxN * BK + 64;
    cudaError_t err = cudaFuncSetAttribute(mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    mma_probe_kernel<<<1, kProbeThreads, smem, stream>>>(tmA, tmB, D, N, K, reinterpret_cast<DeviceStatus *>(workspace));
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(void *workspace, uint32_t budget_us, cudaStream_t stream)
{
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(reinterpret_cast<DeviceStatus *>(workspace),
                                                      (uint64_t)budget_us * 1000ull);
    return cudaGetLastError();
}

}  // namespace fgf8
