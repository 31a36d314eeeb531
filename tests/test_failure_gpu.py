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
