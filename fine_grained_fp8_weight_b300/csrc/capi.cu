// capi.cu -- the extern "C" boundary declared in include/fgf8.h: argument
// checks on the host, device checks, then the kernel launchers.  Nothing here
// allocates device memory.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/fgf8.h"
#include "../../include/fgf8_testing.h"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int checked;     // 0 = not yet, 1 = supported, -1 = unsupported
    int num_sms;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mutex;

// Compute capability 10.3 (B300) only: the kernels are built for sm_103a.
fgf8_status current_device(int *num_sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FGF8_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FGF8_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_devices_mutex);
    DeviceInfo &d = g_devices[dev];
    if (d.checked == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FGF8_ERR_CUDA;
        d.num_sms = sms;
        d.checked = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (d.checked < 0) return FGF8_ERR_UNSUPPORTED_DEVICE;
    if (num_sms) *num_sms = d.num_sms;
    return FGF8_OK;
}

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

fgf8_status from_cuda(cudaError_t e)
{
    return e == cudaSuccess ? FGF8_OK : FGF8_ERR_CUDA;
}

}  // namespace

extern "C" {

const char *fgf8_status_string(fgf8_status st)
{
    switch (st) {
    case FGF8_OK: return "ok";
    case FGF8_ERR_INVALID_ARG: return "invalid argument";
    case FGF8_ERR_MISALIGNED: return "misaligned pointer or stride";
    case FGF8_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case FGF8_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case FGF8_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FGF8_ERR_CUDA: return "CUDA error";
    case FGF8_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

const char *fgf8_version(void)
{
    return "fgf8 0.13 sm_103a";
}

fgf8_status fp8_quant_act_1x128(const void *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, float *s,
                                int64_t lds, uint8_t *qT, float *sT, int64_t ldsT, void *stream)
{
    if (M < 0 || K <= 0) return FGF8_ERR_INVALID_ARG;
    if (K % 128 != 0) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return FGF8_OK;                 // empty input: nothing to read or write
    if (x == nullptr || ldx < K) return FGF8_ERR_INVALID_ARG;
    if ((q == nullptr) != (s == nullptr) || (qT == nullptr) != (sT == nullptr)) return FGF8_ERR_INVALID_ARG;
    if (q == nullptr && qT == nullptr) return FGF8_ERR_INVALID_ARG;
    if (K % 128 != 0) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (q != nullptr && (lds < M || lds % 4 != 0)) return FGF8_ERR_INVALID_ARG;
    if (qT != nullptr && (ldsT < K || ldsT % 4 != 0)) return FGF8_ERR_INVALID_ARG;
    if (qT != nullptr && M % 16 != 0) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (M * (K / 128) >= (int64_t(1) << 31)) return FGF8_ERR_UNSUPPORTED_SHAPE;   // 2^31 tiles
    if (!aligned(x, 16) || ldx % 8 != 0) return FGF8_ERR_MISALIGNED;
    if ((q && (!aligned(q, 16) || !aligned(s, 16))) || (qT && (!aligned(qT, 16) || !aligned(sT, 16))))
        return FGF8_ERR_MISALIGNED;
    fgf8_status st = current_device(nullptr);
    if (st != FGF8_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (qT == nullptr) return from_cuda(fgf8::launch_quant_act_rows(x, M, K, ldx, q, s, lds, cs));
    return from_cuda(fgf8::launch_quant_act_tiles(x, M, K, ldx, q, s, lds, qT, sT, ldsT, cs));
}

fgf8_status fp8_quant_w_128x128(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, float *s,
                                int64_t lds, void *stream)
{
    if (N < 0 || K <= 0) return FGF8_ERR_INVALID_ARG;
    if (K % 128 != 0) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (N == 0) return FGF8_OK;                 // empty input: nothing to read or write
    if (w == nullptr || q == nullptr || s == nullptr || ldw < K) return FGF8_ERR_INVALID_ARG;
    if (lds < (N + 127) / 128 || lds % 4 != 0) return FGF8_ERR_INVALID_ARG;
    if (!aligned(w, 16) || ldw % 8 != 0 || !aligned(q, 16) || !aligned(s, 16)) return FGF8_ERR_MISALIGNED;
    fgf8_status st = current_device(nullptr);
    if (st != FGF8_OK) return st;
    return from_cuda(fgf8::launch_quant_w(w, N, K, ldw, q, s, lds, 1, static_cast<cudaStream_t>(stream)));
}

fgf8_status fp8_quant_w_128x128_grouped(const void *w, int32_t num_experts, int64_t N, int64_t K, int64_t ldw,
                                        uint8_t *q, float *s, int64_t lds, void *stream)
{
    if (num_experts < 0 || num_experts > 65535 || N < 0 || K <= 0) return FGF8_ERR_INVALID_ARG;
    if (K % 128 != 0) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (N == 0 || num_experts == 0) return FGF8_OK;
    if (w == nullptr || q == nullptr || s == nullptr || ldw < K) return FGF8_ERR_INVALID_ARG;
    if (lds < (N + 127) / 128 || lds % 4 != 0) return FGF8_ERR_INVALID_ARG;
    if (!aligned(w, 16) || ldw % 8 != 0 || !aligned(q, 16) || !aligned(s, 16)) return FGF8_ERR_MISALIGNED;
    fgf8_status st = current_device(nullptr);
    if (st != FGF8_OK) return st;
    return from_cuda(
        fgf8::launch_quant_w(w, N, K, ldw, q, s, lds, num_experts, static_cast<cudaStream_t>(stream)));
}

fgf8_status fp8_quant_w_128x128_t(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *qT, float *sT,
                                  int64_t ldsT, uint8_t *q, float *s, int64_t lds, void *stream)
{
    if (N < 0 || K <= 0) return FGF8_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 128 != 0) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (N == 0) return FGF8_OK;                 // empty input: nothing to read or write
    if (w == nullptr || qT == nullptr || sT == nullptr || ldw < K) return FGF8_ERR_INVALID_ARG;
    if (ldsT < K / 128 || ldsT % 4 != 0) return FGF8_ERR_INVALID_ARG;
    if ((q == nullptr) != (s == nullptr)) return FGF8_ERR_INVALID_ARG;
    if (q != nullptr && (lds < N / 128 || lds % 4 != 0)) return FGF8_ERR_INVALID_ARG;
    if (!aligned(w, 16) || ldw % 8 != 0 || !aligned(qT, 16) || !aligned(sT, 16)) return FGF8_ERR_MISALIGNED;
    if (q != nullptr && (!aligned(q, 16) || !aligned(s, 16))) return FGF8_ERR_MISALIGNED;
    fgf8_status st = current_device(nullptr);
    if (st != FGF8_OK) return st;
    return from_cuda(fgf8::launch_quant_w_t(w, N, K, ldw, qT, sT, ldsT, q, s, lds, static_cast<cudaStream_t>(stream)));
}

size_t fgf8_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t num_experts)
{
    return fgf8::gemm_workspace_bytes(M, N, K, num_experts, 0);
}

size_t fgf8_gemm_workspace_min_bytes(int64_t M, int64_t N, int64_t K, int32_t num_experts)
{
    return fgf8::gemm_workspace_min_bytes(M, N, K, num_experts);
}

// Host checks of a GEMM call; the workspace size is checked only when
// `check_ws_size` (the allocation-free entry point checks its own scratch).
static fgf8_status check_gemm(const uint8_t *A, const float *sa, int64_t ldsa, const uint8_t *B, const float *sb,
                              int64_t ldsb, int bkind, void *C, int64_t ldc, int cdt, int64_t M, int64_t N,
                              int64_t K, void *workspace, size_t ws_bytes, int32_t num_experts,
                              bool check_ws_size = true)
{
    if (!A || !sa || !B || !sb || !C || !workspace) return FGF8_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return FGF8_ERR_INVALID_ARG;
    if (bkind != FGF8_BSCALE_BLOCK128 && bkind != FGF8_BSCALE_ROW1x128) return FGF8_ERR_INVALID_ARG;
    if (cdt != FGF8_OUT_BF16 && cdt != FGF8_OUT_FP32) return FGF8_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 16 != 0) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (ldsa < M || ldsa % 4 != 0) return FGF8_ERR_INVALID_ARG;
    const int64_t sb_min = bkind == FGF8_BSCALE_BLOCK128 ? (N + 127) / 128 : N;
    if (ldsb < sb_min || ldsb % 4 != 0) return FGF8_ERR_INVALID_ARG;
    if (ldc < N) return FGF8_ERR_INVALID_ARG;
    const int64_t esz = cdt == FGF8_OUT_BF16 ? 2 : 4;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sa, 16) || !aligned(sb, 16) || !aligned(C, 16) ||
        (ldc * esz) % 16 != 0 || !aligned(workspace, 256))
        return FGF8_ERR_MISALIGNED;
    if (check_ws_size && ws_bytes < fgf8::gemm_workspace_min_bytes(M, N, K, num_experts))
        return FGF8_ERR_WORKSPACE_TOO_SMALL;
    return FGF8_OK;
}

fgf8_status fp8_gemm_blockscaled(const uint8_t *A, const float *sa, int64_t ldsa, const uint8_t *B, const float *sb,
                                 int64_t ldsb, fgf8_bscale_kind bkind, void *C, int64_t ldc, fgf8_out_dtype cdt,
                                 int64_t M, int64_t N, int64_t K, void *workspace, size_t ws_bytes, void *stream)
{
    fgf8_status st = check_gemm(A, sa, ldsa, B, sb, ldsb, bkind, C, ldc, cdt, M, N, K, workspace, ws_bytes, 1);
    if (st != FGF8_OK) return st;
    int num_sms = 0;
    st = current_device(&num_sms);
    if (st != FGF8_OK) return st;
    fgf8::GemmArgs a{A, sa, ldsa, B, sb, ldsb, (int)bkind, C, ldc, cdt == FGF8_OUT_FP32 ? 1 : 0, M, N, K,
                     nullptr, 1, workspace, ws_bytes};
    return from_cuda(fgf8::launch_gemm(a, static_cast<cudaStream_t>(stream), num_sms));
}

fgf8_status fp8_grouped_gemm_blockscaled(const uint8_t *A, const float *sa, int64_t ldsa, const uint8_t *B,
                                         const float *sb, int64_t ldsb, const int32_t *m_indices,
                                         int32_t num_experts, void *C, int64_t ldc, fgf8_out_dtype cdt,
                                         int64_t M_total, int64_t N, int64_t K, void *workspace, size_t ws_bytes,
                                         void *stream)
{
    if (m_indices == nullptr || num_experts < 1) return FGF8_ERR_INVALID_ARG;
    if (M_total % 128 != 0) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)num_experts * N > INT32_MAX / 2) return FGF8_ERR_UNSUPPORTED_SHAPE;
    fgf8_status st = check_gemm(A, sa, ldsa, B, sb, ldsb, FGF8_BSCALE_BLOCK128, C, ldc, cdt, M_total, N, K,
                                workspace, ws_bytes, num_experts);
    if (st != FGF8_OK) return st;
    if (!aligned(m_indices, 4)) return FGF8_ERR_MISALIGNED;
    int num_sms = 0;
    st = current_device(&num_sms);
    if (st != FGF8_OK) return st;
    fgf8::GemmArgs a{A, sa, ldsa, B, sb, ldsb, 0, C, ldc, cdt == FGF8_OUT_FP32 ? 1 : 0, M_total, N, K,
                     m_indices, num_experts, workspace, ws_bytes};
    return from_cuda(fgf8::launch_gemm(a, static_cast<cudaStream_t>(stream), num_sms));
}

fgf8_status fp8_gemm_bf16a_blockscaled(const void *x, int64_t ldx, const uint8_t *B, const float *sb, int64_t ldsb,
                                       void *C, int64_t ldc, fgf8_out_dtype cdt, int64_t M, int64_t N, int64_t K,
                                       void *workspace, size_t ws_bytes, void *stream)
{
    if (M == 0 || N == 0) return FGF8_OK;                // empty output: nothing to read or write
    if (!x || !B || !sb || !C || !workspace) return FGF8_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 1) return FGF8_ERR_INVALID_ARG;
    if (cdt != FGF8_OUT_BF16 && cdt != FGF8_OUT_FP32) return FGF8_ERR_INVALID_ARG;
    if (M > 256 || K % 128 != 0 || N % 16 != 0) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (N > INT32_MAX / 2 || K > INT32_MAX / 2) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (ldx < K || ldsb < (N + 127) / 128 || ldsb % 4 != 0 || ldc < N) return FGF8_ERR_INVALID_ARG;
    const int64_t esz = cdt == FGF8_OUT_BF16 ? 2 : 4;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(B, 16) || !aligned(sb, 16) || !aligned(C, 16) ||
        (ldc * esz) % 16 != 0 || !aligned(workspace, 256))
        return FGF8_ERR_MISALIGNED;
    if (ws_bytes < fgf8::gemm_workspace_min_bytes(M, N, K, 1)) return FGF8_ERR_WORKSPACE_TOO_SMALL;
    int num_sms = 0;
    fgf8_status st = current_device(&num_sms);
    if (st != FGF8_OK) return st;
    fgf8::GemmArgs a{nullptr, nullptr, 0, B, sb, ldsb, 0, C, ldc, cdt == FGF8_OUT_FP32 ? 1 : 0, M, N, K,
                     nullptr, 1, workspace, ws_bytes};
    a.xbf16 = x;
    a.ldx = ldx;
    return from_cuda(fgf8::launch_bf16a(a, static_cast<cudaStream_t>(stream), num_sms));
}

size_t fgf8_masked_gemm_workspace_bytes(int32_t num_experts, int64_t cap, int64_t N, int64_t K)
{
    if (num_experts < 1 || cap < 1 || N < 1 || K < 128) return fgf8::kWsHeaderBytes;
    return fgf8::masked_workspace_bytes(num_experts, cap, N, K);
}

fgf8_status fp8_masked_grouped_gemm_blockscaled(const uint8_t *A, const float *sa, int64_t ldsa, const uint8_t *B,
                                                const float *sb, int64_t ldsb, const int32_t *counts,
                                                int32_t num_experts, int64_t cap, void *C, int64_t ldc,
                                                fgf8_out_dtype cdt, int64_t N, int64_t K, void *workspace,
                                                size_t ws_bytes, void *stream)
{
    if (num_experts < 0 || num_experts > 65535) return FGF8_ERR_INVALID_ARG;
    if (num_experts == 0) return FGF8_OK;                // nothing to read or write
    if (!A || !sa || !B || !sb || !counts || !C || !workspace) return FGF8_ERR_INVALID_ARG;
    if (cap < 1 || N < 1 || K < 1) return FGF8_ERR_INVALID_ARG;
    if (cdt != FGF8_OUT_BF16 && cdt != FGF8_OUT_FP32) return FGF8_ERR_INVALID_ARG;
    if (cap > 256 || cap % 16 != 0 || K % 128 != 0 || N % 16 != 0) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)num_experts * N > INT32_MAX / 2 || (int64_t)num_experts * cap > INT32_MAX / 2 ||
        (int64_t)num_experts * (K / 128) > INT32_MAX / 2 || K > INT32_MAX / 2)
        return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (ldsa < (int64_t)num_experts * cap || ldsa % 4 != 0) return FGF8_ERR_INVALID_ARG;
    if (ldsb < (N + 127) / 128 || ldsb % 4 != 0) return FGF8_ERR_INVALID_ARG;
    if (ldc < N) return FGF8_ERR_INVALID_ARG;
    const int64_t esz = cdt == FGF8_OUT_BF16 ? 2 : 4;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sa, 16) || !aligned(sb, 16) || !aligned(C, 16) ||
        !aligned(counts, 4) || (ldc * esz) % 16 != 0 || !aligned(workspace, 256))
        return FGF8_ERR_MISALIGNED;
    if (ws_bytes < fgf8::masked_workspace_bytes(num_experts, cap, N, K)) return FGF8_ERR_WORKSPACE_TOO_SMALL;
    int num_sms = 0;
    fgf8_status st = current_device(&num_sms);
    if (st != FGF8_OK) return st;
    fgf8::GemmArgs a{A, sa, ldsa, B, sb, ldsb, 0, C, ldc, cdt == FGF8_OUT_FP32 ? 1 : 0, cap, N, K,
                     nullptr, num_experts, workspace, ws_bytes};
    a.counts = counts;
    a.cap = cap;
    return from_cuda(fgf8::launch_masked(a, static_cast<cudaStream_t>(stream), num_sms));
}

// ---------------------------------------------------------------------------
// Allocation-free GEMM entry point.  Its scratch -- the device status word,
// the split-K arrival counters and, for the decode-sized GEMMs that split K,
// their FP32 partial sums -- lives in this file-scope device array instead of
// a workspace the caller allocates.  Every device that loads the library
// holds the array until the process exits; all calls on a device share it.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 10;        // 4 KiB per device: status header and counters
static_assert(kStaticScratchBytes >= fgf8::kWsPartialsOffset, "the cleared header and counters fit");
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mutex;
void *g_static_scratch_ptr[kMaxDevices];

// Device address of g_static_scratch on the current device, looked up once per
// device (the host-side name is only a stand-in, not a device address).
fgf8_status static_scratch(void **ptr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FGF8_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FGF8_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (g_static_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return FGF8_ERR_CUDA;
        g_static_scratch_ptr[dev] = p;
    }
    *ptr = g_static_scratch_ptr[dev];
    return FGF8_OK;
}

}  // namespace

fgf8_status fp8_gemm_blockscaled_noalloc(const uint8_t *A, const float *sa, int64_t ldsa, const uint8_t *B,
                                         const float *sb, int64_t ldsb, fgf8_bscale_kind bkind, void *C,
                                         int64_t ldc, fgf8_out_dtype cdt, int64_t M, int64_t N, int64_t K,
                                         void *stream)
{
    int num_sms = 0;
    fgf8_status st = current_device(&num_sms);
    if (st != FGF8_OK) return st;
    void *ws = nullptr;
    st = static_scratch(&ws);
    if (st != FGF8_OK) return st;
    st = check_gemm(A, sa, ldsa, B, sb, ldsb, bkind, C, ldc, cdt, M, N, K, ws, kStaticScratchBytes, 1, false);
    if (st != FGF8_OK) return st;
    fgf8::GemmArgs a{A, sa, ldsa, B, sb, ldsb, (int)bkind, C, ldc, cdt == FGF8_OUT_FP32 ? 1 : 0, M, N, K,
                     nullptr, 1, ws, kStaticScratchBytes};
    // the scratch the schedule for this shape really uses (on this device,
    // with this scratch) must fit
    if (fgf8::gemm_required_bytes(a, num_sms) > kStaticScratchBytes) return FGF8_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // the previous call's status word (and split-K counters) must not leak into this one
    if (cudaMemsetAsync(ws, 0, fgf8::gemm_workspace_zeroed_bytes(M, N, K, 1), cs) != cudaSuccess) return FGF8_ERR_CUDA;
    return from_cuda(fgf8::launch_gemm(a, cs, num_sms));
}

fgf8_status fgf8_noalloc_read_status(void *stream, int32_t *site)
{
    void *ws = nullptr;
    fgf8_status st = static_scratch(&ws);
    if (st != FGF8_OK) return st;
    return fgf8_read_status(ws, stream, site);
}

fgf8_status fgf8_read_status(void *workspace, void *stream, int32_t *site)
{
    if (workspace == nullptr) return FGF8_ERR_INVALID_ARG;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int32_t word[2] = {0, 0};
    if (cudaMemcpyAsync(word, workspace, sizeof word, cudaMemcpyDeviceToHost, cs) != cudaSuccess) return FGF8_ERR_CUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return FGF8_ERR_CUDA;
    if (site) *site = word[1];
    if (word[0] != 0) {
        const int32_t zero[2] = {0, 0};
        if (cudaMemcpyAsync(workspace, zero, sizeof zero, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
            cudaStreamSynchronize(cs) != cudaSuccess)
            return FGF8_ERR_CUDA;
    }
    return static_cast<fgf8_status>(word[0]);
}

fgf8_status fgf8_mma_probe(const uint8_t *A, const uint8_t *B, float *D, int32_t N, int32_t K, void *workspace,
                           void *stream)
{
    if (!A || !B || !D || !workspace) return FGF8_ERR_INVALID_ARG;
    if (N < 16 || N > 256 || N % 16 != 0 || K < 128 || K > 16384 || K % 128 != 0) return FGF8_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16) || !aligned(workspace, 256)) return FGF8_ERR_MISALIGNED;
    fgf8_status st = current_device(nullptr);
    if (st != FGF8_OK) return st;
    return from_cuda(fgf8::launch_mma_probe(A, B, D, N, K, workspace, static_cast<cudaStream_t>(stream)));
}

fgf8_status fgf8_selftest_wait_timeout(void *workspace, uint32_t budget_us, void *stream)
{
    if (!workspace || budget_us == 0 || budget_us > 2000000u) return FGF8_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return FGF8_ERR_MISALIGNED;
    fgf8_status st = current_device(nullptr);
    if (st != FGF8_OK) return st;
    return from_cuda(fgf8::launch_wait_timeout_selftest(workspace, budget_us, static_cast<cudaStream_t>(stream)));
}

fgf8_status fgf8_selftest_scaled_div(const float *x, const float *s, int64_t n, float *q_encoder,
                                     float *q_ieee, void *stream)
{
    if (n < 0 || (n > 0 && (!x || !s || !q_encoder || !q_ieee))) return FGF8_ERR_INVALID_ARG;
    fgf8_status st = current_device(nullptr);
    if (st != FGF8_OK) return st;
    return from_cuda(fgf8::launch_scaled_div_selftest(x, s, n, q_encoder, q_ieee, static_cast<cudaStream_t>(stream)));
}

fgf8_status fgf8_testing_gemm_schedule(int64_t M, int64_t N, int64_t K, int32_t bkind, size_t ws_bytes,
                                       int32_t num_sms, int32_t *schedule)
{
    if (M < 1 || N < 1 || K < 128 || K % 128 != 0 || (bkind != 0 && bkind != 1) || num_sms < 1 || !schedule)
        return FGF8_ERR_INVALID_ARG;
    fgf8::GemmArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.bkind = bkind;
    a.ws_bytes = ws_bytes;
    const fgf8::GemmSchedule g = fgf8::gemm_schedule(a, num_sms);
    schedule[0] = g.small_m;
    schedule[1] = g.bn;
    schedule[2] = g.dp_tiles;
    schedule[3] = g.tail_s;
    schedule[4] = g.pair;
    return FGF8_OK;
}

fgf8_status fgf8_testing_set_pair(int32_t mode)
{
    if (mode < 0 || mode > 2) return FGF8_ERR_INVALID_ARG;
    fgf8::set_pair_mode(mode);
    return FGF8_OK;
}

fgf8_status fgf8_testing_set_small_splits(int32_t splits)
{
    if (splits < 0 || splits > 8) return FGF8_ERR_INVALID_ARG;
    fgf8::set_small_splits(splits);
    return FGF8_OK;
}

int32_t fgf8_testing_pair_clusters(void)
{
    if (current_device(nullptr) != FGF8_OK) return 0;
    return fgf8::pair_max_clusters();
}

int32_t fgf8_testing_multicast_clusters(void)
{
    if (current_device(nullptr) != FGF8_OK) return 0;
    return fgf8::mc_max_clusters();
}

}  // extern "C"
