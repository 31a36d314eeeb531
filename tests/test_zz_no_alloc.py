"""The allocation-free GEMM entry point (fp8_gemm_blockscaled_noalloc), for
callers that may not allocate device memory -- a plugin whose host framework
owns all GPU memory, or a loop where an allocation could stall.  It keeps its
scratch in a library-owned device array instead of a caller workspace.

Checked through the C ABI on calls in a row with different shapes, output
types and scale kinds -- large tiles and the decode-size path that splits K
over a thread-block cluster, twice in a row on the shared scratch -- against
the oracle's binary64 result within the GEMM tolerance used throughout the
tests, |C - C_ref| <= 2^-7 * sum|a_hat*b_hat| + 1e-6, and against the
workspace entry point (fp8_gemm_blockscaled) within the same tolerance;
decode shapes of 16 and 256 tokens run on the scratch.  This file is
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


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def test_noalloc_matches_oracle_and_workspace_entry_point():
    L = ensure_built()
    cases = [(1, 128, 256, 512, 0, torch.bfloat16),      # first call on the device: looks up the array; splits K
             (2, 300, 400, 1024, 1, torch.float32),      # large tiles, per-row B scales
             (3, 128, 512, 2048, 0, torch.float32),      # split K again, after a large-tile call
             (3, 128, 512, 2048, 0, torch.float32),      # ... and the same call once more
             (4, 128, 512, 1024, 1, torch.bfloat16)]     # M <= 256 with per-row B scales: large tiles
    for seed, M, N, K, bkind, dt in cases:
        qa, sa, qb, sb = _case(seed, M, N, K, bkind)
        ref_out = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
        got_out = torch.full((M, N), float("nan"), dtype=dt, device=DEV)
        dqa, dsa, dqb, dsb = _d(qa), _d(sa), _d(qb), _d(sb)
        assert _call_workspace(L, dqa, dsa, dqb, dsb, bkind, ref_out) == 0
        assert _call_noalloc(L, dqa, dsa, dqb, dsb, bkind, got_out) == 0
        torch.cuda.synchronize()
        Cr, S = oracle.gemm_blockscaled(qa, sa, qb, sb, bkind)
        got = _f64(got_out)
        bound = 2.0 ** -7 * S + 1e-6
        assert np.all(np.isfinite(got)), "the no-allocation call left outputs unwritten"
        assert np.all(np.abs(got - Cr) <= bound), f"{M}x{N}x{K}: outside the bound against the oracle"
        assert np.all(np.abs(got - _f64(ref_out)) <= bound), f"{M}x{N}x{K}: differs from the workspace entry point"
        assert fg.fgf8_noalloc_read_status() == (0, 0)


def test_noalloc_decode_shapes_fit():
    # decode token counts up to 128 split K over a thread-block cluster whose
    # CTAs reduce through distributed shared memory, more tokens run whole
    # large tiles: nothing but the status header is needed, so M = 16 and
    # M = 256 with N = 4096, K = 7168 both run
    L = ensure_built()
    for seed, M in ((5, 16), (6, 256)):
        sch = fg.fgf8_testing_gemm_schedule(M, 4096, 7168, 0, ws_bytes=4096)
        assert sch["small_m"] == (1 if M <= 128 else 0) and (M <= 128 or sch["tail_s"] == 1)
        qa, sa, qb, sb = _case(seed, M, 4096, 7168, 0)
        out = torch.full((M, 4096), float("nan"), dtype=torch.bfloat16, device=DEV)
        assert _call_noalloc(L, _d(qa), _d(sa), _d(qb), _d(sb), 0, out) == 0
        torch.cuda.synchronize()
        rows = np.array([0, 7, M - 1])
        Cr, S = oracle.gemm_blockscaled(qa, sa, qb, sb, 0, rows=rows)
        assert np.all(np.abs(_f64(out)[rows] - Cr) <= 2.0 ** -7 * S + 1e-6)
        assert fg.fgf8_noalloc_read_status() == (0, 0)


def test_noalloc_rejects_bad_arguments_without_launching():
    L = ensure_built()
    a = ctypes.c_void_p(0x10000)
    # K not a multiple of 128
    assert L.fp8_gemm_blockscaled_noalloc(a, a, 4, a, a, 4, 0, a, 128, 0, 4, 128, 200, None) == 3
    # null operand
    assert L.fp8_gemm_blockscaled_noalloc(None, a, 4, a, a, 4, 0, a, 128, 0, 4, 128, 128, None) == 1
