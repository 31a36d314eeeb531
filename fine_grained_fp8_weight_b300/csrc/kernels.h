// kernels.h -- launchers shared between the kernel files and the C ABI layer.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace fgf8 {

cudaError_t launch_quant_act_rows(const void *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, float *s,
                                  int64_t lds, cudaStream_t stream);
cudaError_t launch_quant_act_tiles(const void *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, float *s,
                                   int64_t lds, uint8_t *qT, float *sT, int64_t ldsT, cudaStream_t stream);
cudaError_t launch_scaled_div_selftest(const float *x, const float *s, int64_t n, float *fast, float *ieee,
                                       cudaStream_t stream);
cudaError_t launch_quant_w(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, float *s, int64_t lds,
                           int32_t num_experts, cudaStream_t stream);
cudaError_t launch_quant_w_t(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *qT, float *sT, int64_t ldsT,
                             uint8_t *q, float *s, int64_t lds, cudaStream_t stream);

struct GemmArgs {
    const uint8_t *A;
    const float *sa;
    int64_t ldsa;
    const uint8_t *B;
    const float *sb;
    int64_t ldsb;
    int bkind;              // 0: 128x128 block scales, 1: per-row scales
    void *C;
    int64_t ldc;
    int out_f32;            // 0: BF16 output, 1: FP32 output
    int64_t M, N, K;
    const int32_t *m_indices;   // grouped contiguous layout when non-null
    int32_t num_experts;
    void *workspace;
    size_t ws_bytes;
    // masked grouped layout (decode MoE): when counts != nullptr, A and C hold
    // num_experts slots of `cap` token rows (sa their scales, slot e at column
    // e*cap), B num_experts weight matrices of N rows, sb num_experts scale
    // blocks of K/128 rows
    const int32_t *counts = nullptr;
    int64_t cap = 0;
    // token operand as BF16 [M][ldx], quantized 1x128 inside the GEMM
    // (M <= 256); A and sa are unused then
    const void *xbf16 = nullptr;
    int64_t ldx = 0;
};

// Workspace layout, the same for every GEMM kernel so that one workspace can
// serve all of them in turn: [0, 256) status word; [256, 1280) 256 arrival
// counters, written by nothing but the last-wave split's atomics and their
// resets to zero (one per tail tile); from 1280 on, its FP32 partial sums.
// The small-M kernel's K split is reduced within a thread-block cluster and
// needs the status word only.
constexpr size_t kWsHeaderBytes = 256;
constexpr int kMaxCounters = 256;
constexpr size_t kWsPartialsOffset = kWsHeaderBytes + kMaxCounters * 4;

// Workspace that enables every schedule (for dense GEMMs, the last-wave
// split's partial tiles), and the least a call accepts.
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t num_experts, int num_sms);
size_t gemm_workspace_min_bytes(int64_t M, int64_t N, int64_t K, int32_t num_experts);
// Leading part of the workspace that must be zero when a call starts (the
// status word and the arrival counters).
size_t gemm_workspace_zeroed_bytes(int64_t M, int64_t N, int64_t K, int32_t num_experts);
// The schedule launch_gemm picks: small-M kernel (tail_s = its K split), or
// tile width, whole-tile count and pieces per last-wave tile (1: no split);
// pair = 1 for the CTA-pair kernel (256 x 128 tiles on two SMs).
struct GemmSchedule {
    int small_m, bn, dp_tiles, tail_s, pair;
};
GemmSchedule gemm_schedule(const GemmArgs &a, int num_sms);
// 1: dense block-scaled GEMMs of more than 128 rows run on CTA pairs; 2: they
// run single-SM tiles in clusters of two sharing B by TMA multicast; 0: the planner's choice (single-SM tiles).
// Process-wide, for tests.
void set_pair_mode(int mode);
// Concurrent two-CTA clusters of the multicast variant on the current device.
int mc_max_clusters();
// 1..8: the dense small-M kernel splits K over this many CTAs (at most K/128);
// 0: the planner's choice.  Process-wide, for tests.
void set_small_splits(int s);
cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t stream, int num_sms);
// Workspace bytes the schedule launch_gemm picks for `a` (with a.ws_bytes of
// workspace) reads and writes: the status header, plus the last-wave split's
// counters and partials when it splits.
size_t gemm_required_bytes(const GemmArgs &a, int num_sms);
// CTA-pair kernel (gemm_pair.cu): 256 x 128 tiles on two SMs whose tensor
// cores run as one.  pair_max_clusters() is the number of co-resident pairs on
// the current device (0: not available); pair_plan the tile count and the
// last-wave split for `clusters` pairs; launch_pair returns
// cudaErrorNotSupported when the device cannot run it.
struct PairPlan {
    int32_t tiles, dp_tiles, tail_s;
    int64_t cost;               // K-group steps of the whole schedule on one pair
};
int pair_max_clusters();
int pair_tile_n();          // output columns of a pair tile (128 or 256)
size_t pair_tail_workspace_bytes();
PairPlan pair_plan(const GemmArgs &a, int clusters);
cudaError_t launch_pair(const GemmArgs &a, cudaStream_t stream);
// Masked grouped layout: scratch size, launch.
size_t masked_workspace_bytes(int32_t num_experts, int64_t cap, int64_t N, int64_t K);
cudaError_t launch_masked(const GemmArgs &a, cudaStream_t stream, int num_sms);
// Token operand given as BF16 and quantized in the GEMM's producer (M <= 256).
cudaError_t launch_bf16a(const GemmArgs &a, cudaStream_t stream, int num_sms);
cudaError_t launch_mma_probe(const uint8_t *A, const uint8_t *B, float *D, int N, int K, void *workspace,
                             cudaStream_t stream);
cudaError_t launch_wait_timeout_selftest(void *workspace, uint32_t budget_us, cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).  Returns false if the driver rejects the map.
bool make_tensor_map_2d(void *map, int dtype_bytes, bool is_float, const void *base, uint64_t inner, uint64_t outer,
                        uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128);

}  // namespace fgf8
