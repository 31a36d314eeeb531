"""Failure detection without a GPU fault: a bounded wait that nothing
satisfies expires, the kernel records FGF8_ERR_TIMEOUT in the status word,
releases its tensor memory and returns; the context stays usable and the next
GEMM is correct."""
import numpy as np
import pytest
import torch

import oracle
import fine_grained_fp8_weight_b300 as fg
from fine_grained_fp8_weight_b300 import workloads as wl
from tests.gpu_util import DEV, assert_within_bound, bf16_out_to_f64, ensure_built

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_context_survives():
    L = ensure_built()
    ws = torch.zeros(max(4096, L.fgf8_gemm_workspace_bytes(128, 256, 512, 1)), dtype=torch.uint8, device=DEV)
    st = L.fgf8_selftest_wait_timeout(fg._ptr(ws), 20000, fg._stream(ws.device))
    assert st == 0
    status, site = fg.fgf8_read_status(ws)
    assert status == 7 and site == 99
    assert fg.fgf8_read_status(ws) == (0, 0), "status word is reset after reading"
    g = wl.tiny().gemms[0]
    qa, sa = oracle.quant_act_1x128(g.A)
    qb, sb = oracle.quant_w_128x128(g.B)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    C = fg.fp8_gemm_blockscaled(d(qa), d(sa), d(qb), d(sb), workspace=ws)
    assert fg.fgf8_read_status(ws) == (0, 0)
    Cr, S = oracle.gemm_blockscaled(qa, sa, qb, sb)
    assert_within_bound(bf16_out_to_f64(C), Cr, S)


def test_check_raises_on_timeout_and_next_call_succeeds():
    # an expired wait left in the wrapper's own cached workspace: the next
    # call with check=True raises FGF8_ERR_TIMEOUT and clears the workspace's
    # status word and counters, and the call after it is correct
    L = ensure_built()
    g = wl.tiny().gemms[0]
    qa, sa = oracle.quant_act_1x128(g.A)
    qb, sb = oracle.quant_w_128x128(g.B)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    ops = [d(qa), d(sa), d(qb), d(sb)]
    M, K = qa.shape
    N = qb.shape[0]
    ws = fg.workspace_for(DEV, L.fgf8_gemm_workspace_bytes(M, N, K, 1))
    ws[256:1280].fill_(1)                            # counters as an aborted split could leave them
    assert L.fgf8_selftest_wait_timeout(fg._ptr(ws), 20000, fg._stream(ws.device)) == 0
    with pytest.raises(fg.FGF8Error, match="TIMEOUT"):
        fg.fp8_gemm_blockscaled(*ops, check=True)
    assert not bool(ws[:fg.WS_ZEROED_BYTES].any()), "status word and counters cleared"
    C = fg.fp8_gemm_blockscaled(*ops, check=True)
    Cr, S = oracle.gemm_blockscaled(qa, sa, qb, sb)
    assert_within_bound(bf16_out_to_f64(C), Cr, S)

