"""The allocation-free GEMM entry point (fp8_gemm_blockscaled_noalloc), for
callers that may not allocate device memory -- a plugin whose host framework
owns all GPU memory, or a loop where an allocation could stall.  It keeps its
scratch in a library-owned device array instead of a caller workspace.

Checked through the C ABI against the workspace entry point
(fp8_gemm_blockscaled) on two calls in a row with different shapes, output
types and scale kinds, within the GEMM tolerance used throughout the tests:
|C_noalloc - C_workspace| <= 2^-7 * sum|a_hat*b_hat| + 1e-6.  This file is
collected last so that a failure here stops a -x run only after every other
test has run."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import fine_grained_fp8_weight_b300 as fg
from fine_grained_fp8_weight_b300 import workloads as wl
from tests.gpu_util import DEV, ensure_built

pytestmark = pytest.mark.gpu


def _d(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _case(seed, M, N, K, bkind):
    rng = np.random.default_rng(seed)
    A = wl.bf16_normal(rng, (M, K), 1.0, 0.01, 100.0)
    B = wl.bf16_normal(rng, (N, K), 0.02 if bkind == 0 else 1.0)
    qa, sa = oracle.quant_act_1x128(A)
    qb, sb = oracle.quant_w_128x128(B) if bkind == 0 else oracle.quant_act_1x128(B)
    return qa, sa, qb, sb


def _call_noalloc(L, qa, sa, qb, sb, bkind, out):
    M, K = qa.shape
    N = qb.shape[0]
    cdt = fg.OUT_FP32 if out.dtype == torch.float32 else fg.OUT_BF16
    return L.fp8_gemm_blockscaled_noalloc(fg._ptr(qa), fg._ptr(sa), sa.stride(0), fg._ptr(qb), fg._ptr(sb),
                                          sb.stride(0), bkind, fg._ptr(out), out.stride(0), cdt, M, N, K,
                                          fg._stream(out.device))


def _call_workspace(L, qa, sa, qb, sb, bkind, out):
    M, K = qa.shape
    N = qb.shape[0]
    cdt = fg.OUT_FP32 if out.dtype == torch.float32 else fg.OUT_BF16
    ws = torch.zeros(L.fgf8_gemm_workspace_bytes(M, N, K, 1) + 4096, dtype=torch.uint8, device=DEV)
    return L.fp8_gemm_blockscaled(fg._ptr(qa), fg._ptr(sa), sa.stride(0), fg._ptr(qb), fg._ptr(sb), sb.stride(0),
                                  bkind, fg._ptr(out), out.stride(0), cdt, M, N, K, fg._ptr(ws), ws.numel(),
                                  fg._stream(out.device))


def test_noalloc_matches_workspace_entry_point_twice():
    L = ensure_built()
    cases = [(1, 128, 256, 512, 0, torch.bfloat16),      # first call on the device: looks up the array
             (2, 300, 400, 1024, 1, torch.float32)]      # second call: different shape, kind and output
    for seed, M, N, K, bkind, dt in cases:
        qa, sa, qb, sb = _case(seed, M, N, K, bkind)
        ref_out = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
        got_out = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
        dqa, dsa, dqb, dsb = _d(qa), _d(sa), _d(qb), _d(sb)
        assert _call_workspace(L, dqa, dsa, dqb, dsb, bkind, ref_out) == 0
        assert _call_noalloc(L, dqa, dsa, dqb, dsb, bkind, got_out) == 0
        torch.cuda.synchronize()
        _, S = oracle.gemm_blockscaled(qa, sa, qb, sb, bkind)
        ref = ref_out.float().cpu().numpy().astype(np.float64)
        got = got_out.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), "the no-allocation call left outputs unwritten"
        assert np.all(np.abs(got - ref) <= 2.0 ** -7 * S + 1e-6)


def test_noalloc_rejects_bad_arguments_without_launching():
    L = ensure_built()
    a = ctypes.c_void_p(0x10000)
    # K not a multiple of 128
    assert L.fp8_gemm_blockscaled_noalloc(a, a, 4, a, a, 4, 0, a, 128, 0, 4, 128, 200, None) == 3
    # null operand
    assert L.fp8_gemm_blockscaled_noalloc(None, a, 4, a, a, 4, 0, a, 128, 0, 4, 128, 128, None) == 1
