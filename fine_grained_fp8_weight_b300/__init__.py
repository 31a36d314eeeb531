"""Fine-grained FP8 quantization and block-scaled FP8 GEMM for B300 (sm_103a).

Thin ctypes binding over ``libfgf8.so`` (the C ABI in ``include/fgf8.h``).
The functions here only marshal arguments: they allocate outputs with torch,
pass raw device pointers and the current CUDA stream to the library, and turn
a non-zero status into an exception.  Every step of the computation runs in
the library's CUDA kernels; there is no CPU or library fallback, and importing
this package fails if the library has not been built.

Scale layouts ("K-group major", as in the C header):
  activation 1x128 scales  s  [K/128, round_up(M, 4)]
  activation 128x1 scales  sT [ceil(M/128), round_up(K, 4)]
  weight 128x128 scales    s  [K/128, round_up(ceil(N/128), 4)]
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "FGF8Error", "lib", "fp8_quant_act_1x128", "fp8_quant_w_128x128", "fp8_quant_w_128x128_grouped",
    "fp8_gemm_blockscaled",
    "fp8_grouped_gemm_blockscaled", "fp8_masked_grouped_gemm_blockscaled", "fp8_gemm_bf16a_blockscaled",
    "fp8_quant_w_128x128_t", "fgf8_mma_probe", "fgf8_read_status", "fgf8_noalloc_read_status", "workspace_for",
    "BSCALE_BLOCK128", "BSCALE_ROW1x128", "OUT_BF16", "OUT_FP32",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfgf8.so")

BSCALE_BLOCK128 = 0
BSCALE_ROW1x128 = 1
OUT_BF16 = 0
OUT_FP32 = 1

STATUS_NAMES = {0: "FGF8_OK", 1: "FGF8_ERR_INVALID_ARG", 2: "FGF8_ERR_MISALIGNED",
                3: "FGF8_ERR_UNSUPPORTED_SHAPE", 4: "FGF8_ERR_UNSUPPORTED_DEVICE",
                5: "FGF8_ERR_WORKSPACE_TOO_SMALL", 6: "FGF8_ERR_CUDA", 7: "FGF8_ERR_TIMEOUT"}

# Every symbol declared in include/fgf8.h and include/fgf8_testing.h.
EXPORTED = ["fgf8_status_string", "fgf8_version", "fp8_quant_act_1x128", "fp8_quant_w_128x128",
            "fp8_quant_w_128x128_grouped", "fp8_quant_w_128x128_t",
            "fp8_gemm_blockscaled", "fp8_gemm_blockscaled_noalloc", "fp8_grouped_gemm_blockscaled",
            "fp8_masked_grouped_gemm_blockscaled", "fp8_gemm_bf16a_blockscaled", "fgf8_gemm_workspace_bytes", "fgf8_gemm_workspace_min_bytes",
            "fgf8_masked_gemm_workspace_bytes",
            "fgf8_read_status", "fgf8_mma_probe", "fgf8_selftest_wait_timeout", "fgf8_selftest_scaled_div",
            "fgf8_testing_gemm_schedule", "fgf8_testing_pair_clusters", "fgf8_testing_set_pair",
            "fgf8_testing_multicast_clusters",
            "fgf8_testing_set_small_splits",
            "fgf8_noalloc_read_status"]


class FGF8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library with argument types declared (no compute call)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libfgf8.so is not built ({LIB_PATH}); run "
                              "`python -m fine_grained_fp8_weight_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        L.fgf8_status_string.argtypes = [ctypes.c_int]
        L.fgf8_status_string.restype = ctypes.c_char_p
        L.fgf8_version.argtypes = []
        L.fgf8_version.restype = ctypes.c_char_p
        L.fp8_quant_act_1x128.argtypes = [P, I64, I64, I64, P, P, I64, P, P, I64, P]
        L.fp8_quant_w_128x128.argtypes = [P, I64, I64, I64, P, P, I64, P]
        L.fp8_quant_w_128x128_grouped.argtypes = [P, I32, I64, I64, I64, P, P, I64, P]
        L.fp8_quant_w_128x128_t.argtypes = [P, I64, I64, I64, P, P, I64, P, P, I64, P]
        L.fp8_gemm_blockscaled.argtypes = [P, P, I64, P, P, I64, ctypes.c_int, P, I64, ctypes.c_int,
                                           I64, I64, I64, P, SZ, P]
        L.fp8_gemm_blockscaled_noalloc.argtypes = [P, P, I64, P, P, I64, ctypes.c_int, P, I64, ctypes.c_int,
                                                   I64, I64, I64, P]
        L.fp8_grouped_gemm_blockscaled.argtypes = [P, P, I64, P, P, I64, P, I32, P, I64, ctypes.c_int,
                                                   I64, I64, I64, P, SZ, P]
        L.fgf8_gemm_workspace_bytes.argtypes = [I64, I64, I64, I32]
        L.fgf8_gemm_workspace_bytes.restype = SZ
        L.fgf8_gemm_workspace_min_bytes.argtypes = [I64, I64, I64, I32]
        L.fgf8_gemm_workspace_min_bytes.restype = SZ
        L.fp8_masked_grouped_gemm_blockscaled.argtypes = [P, P, I64, P, P, I64, P, I32, I64, P, I64, ctypes.c_int,
                                                          I64, I64, P, SZ, P]
        L.fgf8_masked_gemm_workspace_bytes.argtypes = [I32, I64, I64, I64]
        L.fp8_gemm_bf16a_blockscaled.argtypes = [P, I64, P, P, I64, P, I64, ctypes.c_int, I64, I64, I64, P, SZ, P]
        L.fgf8_masked_gemm_workspace_bytes.restype = SZ
        L.fgf8_read_status.argtypes = [P, P, ctypes.POINTER(I32)]
        L.fgf8_noalloc_read_status.argtypes = [P, ctypes.POINTER(I32)]
        L.fgf8_noalloc_read_status.restype = ctypes.c_int
        L.fgf8_mma_probe.argtypes = [P, P, P, I32, I32, P, P]
        L.fgf8_selftest_wait_timeout.argtypes = [P, ctypes.c_uint32, P]
        L.fgf8_selftest_scaled_div.argtypes = [P, P, I64, P, P, P]
        L.fgf8_testing_gemm_schedule.argtypes = [I64, I64, I64, I32, SZ, I32, P]
        L.fgf8_testing_pair_clusters.argtypes = []
        L.fgf8_testing_pair_clusters.restype = I32
        L.fgf8_testing_multicast_clusters.argtypes = []
        L.fgf8_testing_multicast_clusters.restype = I32
        L.fgf8_testing_set_pair.argtypes = [I32]
        L.fgf8_testing_set_pair.restype = ctypes.c_int
        L.fgf8_testing_set_small_splits.argtypes = [I32]
        L.fgf8_testing_set_small_splits.restype = ctypes.c_int
        for name in ("fp8_quant_act_1x128", "fp8_quant_w_128x128", "fp8_quant_w_128x128_grouped",
                     "fp8_gemm_blockscaled", "fp8_gemm_blockscaled_noalloc",
                     "fp8_grouped_gemm_blockscaled", "fgf8_read_status", "fgf8_mma_probe",
                     "fgf8_selftest_wait_timeout", "fgf8_selftest_scaled_div"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise FGF8Error(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def round_up(v: int, m: int) -> int:
    return (v + m - 1) // m * m


_workspaces: dict = {}

# Bytes at the start of every GEMM workspace that must be zero when a call
# starts: the device status word and the split kernels' arrival counters.
WS_ZEROED_BYTES = 256 + 256 * 4


def workspace_for(device, nbytes: int, stream=None) -> torch.Tensor:
    """A zero-filled, 256-byte aligned device workspace of at least nbytes,
    cached per (device, stream): calls on one stream run in order and may share
    one (the kernels leave it zeroed for the next call); calls on different
    streams could overlap and get different ones."""
    device = torch.device(device)
    if stream is None:
        stream = torch.cuda.current_stream(device)
    key = (device, stream.cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 4096), dtype=torch.uint8, device=device)
        assert ws.data_ptr() % 256 == 0
        _workspaces[key] = ws
    return ws


def _check_device(ws: torch.Tensor, where: str):
    """Read the workspace's device status (synchronizes the stream).  After an
    expired device-side wait the kernels may have left arrival counters
    non-zero: clear them, then raise FGF8Error(FGF8_ERR_TIMEOUT)."""
    st, site = fgf8_read_status(ws)
    if st != 0:
        ws[:WS_ZEROED_BYTES].zero_()
        raise FGF8Error(st, f"{where} (device wait site {site})")


def fp8_quant_act_1x128(x: torch.Tensor, rows: bool = True, transposed: bool = False):
    """1x128 activation quantization (and/or the transposed 128x1 output).

    x: BF16 [M, K] CUDA tensor (row stride may exceed K).  Returns
    (q, s, qT, sT); the ones not requested are None."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    dev = x.device
    q = s = qT = sT = None
    if rows:
        q = torch.empty((M, K), dtype=torch.uint8, device=dev)
        s = torch.empty((K // 128, round_up(max(M, 1), 4)), dtype=torch.float32, device=dev)
    if transposed:
        qT = torch.empty((K, M), dtype=torch.uint8, device=dev)
        sT = torch.empty(((M + 127) // 128, round_up(K, 4)), dtype=torch.float32, device=dev)
    st = lib().fp8_quant_act_1x128(_ptr(x), M, K, x.stride(0), _ptr(q), _ptr(s),
                                   s.shape[1] if s is not None else 0, _ptr(qT), _ptr(sT),
                                   sT.shape[1] if sT is not None else 0, _stream(dev))
    _check(st, "fp8_quant_act_1x128")
    return q, s, qT, sT


def fp8_quant_w_128x128(w: torch.Tensor):
    """128x128 weight quantization.  w: BF16 [N, K].  Returns (q, s)."""
    assert w.dtype == torch.bfloat16 and w.dim() == 2 and w.stride(1) == 1
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((K // 128, round_up((N + 127) // 128, 4)), dtype=torch.float32, device=w.device)
    st = lib().fp8_quant_w_128x128(_ptr(w), N, K, w.stride(0), _ptr(q), _ptr(s), s.shape[1], _stream(w.device))
    _check(st, "fp8_quant_w_128x128")
    return q, s


def fp8_quant_w_128x128_t(w: torch.Tensor, forward: bool = False):
    """128x128 weight quantization written as W^T for the data-gradient GEMM.
    w: BF16 [N, K], N % 128 == 0.  Returns (qT [K, N], sT [N/128, round_up(K/128, 4)])
    and, with forward=True, also (q [N, K], s) as fp8_quant_w_128x128."""
    assert w.dtype == torch.bfloat16 and w.dim() == 2 and w.stride(1) == 1
    N, K = w.shape
    qT = torch.empty((K, N), dtype=torch.uint8, device=w.device)
    sT = torch.empty((N // 128, round_up(K // 128, 4)), dtype=torch.float32, device=w.device)
    q = s = None
    if forward:
        q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
        s = torch.empty((K // 128, round_up(N // 128, 4)), dtype=torch.float32, device=w.device)
    st = lib().fp8_quant_w_128x128_t(_ptr(w), N, K, w.stride(0), _ptr(qT), _ptr(sT), sT.shape[1],
                                     _ptr(q) if forward else None, _ptr(s) if forward else None,
                                     s.shape[1] if forward else 0, _stream(w.device))
    _check(st, "fp8_quant_w_128x128_t")
    return (qT, sT, q, s) if forward else (qT, sT)


def fp8_quant_w_128x128_grouped(w: torch.Tensor):
    """128x128 block quantization of stacked expert weights w: BF16 [E, N, K].
    Returns (q [E, N, K], s [E, K/128, round_up(ceil(N/128), 4)])."""
    assert w.dtype == torch.bfloat16 and w.dim() == 3 and w.is_contiguous()
    E, N, K = w.shape
    q = torch.empty((E, N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((E, K // 128, round_up((N + 127) // 128, 4)), dtype=torch.float32, device=w.device)
    st = lib().fp8_quant_w_128x128_grouped(_ptr(w), E, N, K, K, _ptr(q), _ptr(s), s.shape[2], _stream(w.device))
    _check(st, "fp8_quant_w_128x128_grouped")
    return q, s


def fp8_gemm_blockscaled(A, sa, B, sb, bkind: int = BSCALE_BLOCK128, out_dtype=torch.bfloat16,
                         out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                         check: bool = False):
    """C = A_hat * B_hat^T.  A [M,K] and B [N,K] uint8 E4M3 codes, sa [K/128, ldsa],
    sb [K/128, ldsb] float32 (block or per-row kind).  check=True waits for
    the GEMM and raises FGF8Error if a device-side wait expired."""
    M, K = A.shape
    N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    cdt = OUT_FP32 if out.dtype == torch.float32 else OUT_BF16
    need = lib().fgf8_gemm_workspace_bytes(M, N, K, 1)
    ws = workspace if workspace is not None else workspace_for(A.device, need)
    st = lib().fp8_gemm_blockscaled(_ptr(A), _ptr(sa), sa.stride(0), _ptr(B), _ptr(sb), sb.stride(0), bkind,
                                    _ptr(out), out.stride(0), cdt, M, N, K, _ptr(ws), ws.numel(),
                                    _stream(A.device))
    _check(st, "fp8_gemm_blockscaled")
    if check:
        _check_device(ws, "fp8_gemm_blockscaled")
    return out


def fp8_gemm_bf16a_blockscaled(x, B, sb, out_dtype=torch.bfloat16, out: torch.Tensor | None = None,
                               workspace: torch.Tensor | None = None, check: bool = False):
    """C = quant_1x128(x) * B_hat^T with x: BF16 [M, K] (M <= 256) quantized inside the GEMM.
    check=True waits for the GEMM and raises FGF8Error if a device-side wait expired."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    cdt = OUT_FP32 if out.dtype == torch.float32 else OUT_BF16
    need = lib().fgf8_gemm_workspace_bytes(M, N, K, 1)
    ws = workspace if workspace is not None else workspace_for(x.device, need)
    st = lib().fp8_gemm_bf16a_blockscaled(_ptr(x), x.stride(0), _ptr(B), _ptr(sb), sb.stride(0), _ptr(out),
                                          out.stride(0), cdt, M, N, K, _ptr(ws), ws.numel(), _stream(x.device))
    _check(st, "fp8_gemm_bf16a_blockscaled")
    if check:
        _check_device(ws, "fp8_gemm_bf16a_blockscaled")
    return out


def fp8_grouped_gemm_blockscaled(A, sa, B, sb, m_indices, out_dtype=torch.bfloat16,
                                 out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                                 check: bool = False):
    """Contiguous-layout grouped GEMM.  A [M_total,K], B [E,N,K], sb [E,K/128,ldsb],
    m_indices int32 [M_total] (-1 = padding row, left unwritten).  check=True
    waits for the GEMM and raises FGF8Error if a device-side wait expired."""
    M, K = A.shape
    E, N, _ = B.shape
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    cdt = OUT_FP32 if out.dtype == torch.float32 else OUT_BF16
    need = lib().fgf8_gemm_workspace_bytes(M, N, K, E)
    ws = workspace if workspace is not None else workspace_for(A.device, need)
    st = lib().fp8_grouped_gemm_blockscaled(_ptr(A), _ptr(sa), sa.stride(0), _ptr(B), _ptr(sb), sb.stride(1),
                                            _ptr(m_indices), E, _ptr(out), out.stride(0), cdt, M, N, K,
                                            _ptr(ws), ws.numel(), _stream(A.device))
    _check(st, "fp8_grouped_gemm_blockscaled")
    if check:
        _check_device(ws, "fp8_grouped_gemm_blockscaled")
    return out


def fp8_masked_grouped_gemm_blockscaled(A, sa, B, sb, counts, out_dtype=torch.bfloat16,
                                        out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                                        check: bool = False):
    """Masked-layout grouped GEMM (decode MoE).  A [E, cap, K] uint8 with sa [K/128, ldsa]
    (the 1x128 scales of the stacked [E*cap, K] slots), B [E, N, K] with sb [E, K/128, ldsb],
    counts int32 [E] on the device.  Returns C [E, cap, N]; rows past each expert's count
    are left as they were in `out`.  check=True waits for the GEMM and raises
    FGF8Error if a device-side wait expired."""
    E, cap, K = A.shape
    N = B.shape[1]
    assert sa.dim() == 2 and sa.stride(1) == 1
    assert sb.stride(2) == 1 and sb.stride(0) == sb.shape[1] * sb.stride(1)
    if out is None:
        out = torch.empty((E, cap, N), dtype=out_dtype, device=A.device)
    assert out.stride(0) == cap * out.stride(1)
    cdt = OUT_FP32 if out.dtype == torch.float32 else OUT_BF16
    need = lib().fgf8_masked_gemm_workspace_bytes(E, cap, N, K)
    ws = workspace if workspace is not None else workspace_for(A.device, need)
    st = lib().fp8_masked_grouped_gemm_blockscaled(_ptr(A), _ptr(sa), sa.stride(0), _ptr(B), _ptr(sb), sb.stride(1),
                                                   _ptr(counts), E, cap, _ptr(out), out.stride(1), cdt, N, K,
                                                   _ptr(ws), ws.numel(), _stream(A.device))
    _check(st, "fp8_masked_grouped_gemm_blockscaled")
    if check:
        _check_device(ws, "fp8_masked_grouped_gemm_blockscaled")
    return out


def fgf8_mma_probe(A: torch.Tensor, B: torch.Tensor, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Raw tensor-core accumulation of A [128,K] * B [N,K]^T (E4M3 codes), no promotion."""
    N, K = B.shape
    D = torch.empty((128, N), dtype=torch.float32, device=A.device)
    ws = workspace if workspace is not None else workspace_for(A.device, 256)
    st = lib().fgf8_mma_probe(_ptr(A), _ptr(B), _ptr(D), N, K, _ptr(ws), _stream(A.device))
    _check(st, "fgf8_mma_probe")
    return D


def fgf8_testing_gemm_schedule(M: int, N: int, K: int, bkind: int = BSCALE_BLOCK128,
                               ws_bytes: int | None = None, num_sms: int = 148) -> dict:
    """The schedule fp8_gemm_blockscaled picks (host only, nothing launched).
    ws_bytes defaults to fgf8_gemm_workspace_bytes(M, N, K, 1)."""
    if ws_bytes is None:
        ws_bytes = lib().fgf8_gemm_workspace_bytes(M, N, K, 1)
    out = (ctypes.c_int32 * 5)()
    _check(lib().fgf8_testing_gemm_schedule(M, N, K, bkind, ws_bytes, num_sms, out), "fgf8_testing_gemm_schedule")
    return {"small_m": out[0], "bn": out[1], "dp_tiles": out[2], "tail_s": out[3], "pair": out[4]}


def fgf8_read_status(workspace: torch.Tensor):
    """(status, site) of the device status word; resets it.  Synchronizes the stream."""
    site = ctypes.c_int32(0)
    st = lib().fgf8_read_status(_ptr(workspace), _stream(workspace.device), ctypes.byref(site))
    return st, site.value


def fgf8_noalloc_read_status(device=None):
    """(status, site) of the allocation-free GEMM's scratch on the current
    device; resets it.  Synchronizes the current stream."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    site = ctypes.c_int32(0)
    st = lib().fgf8_noalloc_read_status(_stream(dev), ctypes.byref(site))
    return st, site.value
