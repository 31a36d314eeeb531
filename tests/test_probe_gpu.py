"""Tensor-core accumulation probe ("dssusan.co.kr Q&A post 93378",
inner-dimension passage: FP8 GEMM accumulation on H800 keeps about 14 bits;
"jp-study.kr Q&A post 309256": Hopper aligns products to the largest
exponent before adding).  The probe chains tcgen05.mma instructions (K = 32
each) into one FP32 TMEM accumulator without promotion; these tests check it
on exactly representable sums and measure how many bits survive when one
large product is accumulated with many small ones."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import fine_grained_fp8_weight_b300 as fg
from tests.gpu_util import DEV, ensure_built

pytestmark = pytest.mark.gpu

INT_CODES = {v: c for c, v in [(0x00, 0), (0x38, 1), (0x40, 2), (0x44, 3), (0x48, 4), (0xB8, -1),
                               (0xC0, -2), (0xC4, -3), (0xC8, -4)]}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _codes(vals):
    return np.vectorize(lambda v: INT_CODES[int(v)])(vals).astype(np.uint8)


@pytest.mark.parametrize("N,K", [(16, 128), (32, 512), (128, 256), (256, 1024), (48, 128)])
def test_probe_exact_small_integers(N, K):
    rng = np.random.default_rng(N + K)
    av = rng.integers(-4, 5, size=(128, K))
    bv = rng.integers(-4, 5, size=(N, K))
    A, B = _codes(av), _codes(bv)
    D = fg.fgf8_mma_probe(torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV)).cpu().numpy()
    ref = (av @ bv.T).astype(np.float64)          # |sum| < 2^24: exact in FP32
    assert np.array_equal(D.astype(np.float64), ref)
    # the same against the oracle's exact dot product
    for m, n in [(0, 0), (127, N - 1), (64, N // 2)]:
        assert D[m, n] == oracle.dot_e4m3_exact(A[m], B[n]) / 2.0 ** 18


def _pow2_code(e):
    v = np.float32(2.0 ** e)
    return oracle.e4m3_encode(float(v))


def test_probe_accumulation_precision():
    """One product 2^8 plus n small products 2^(8-g), g = 0..26, either inside
    the same K=32 instruction as the large one or in later instructions.  A
    gap is kept when the result equals the binary32 rounding of the exact sum."""
    K, N = 128, 16
    A = np.zeros((128, K), np.uint8)
    B = np.zeros((N, K), np.uint8)
    ga = np.arange(128) % 14                       # A-side part of the gap
    for m in range(128):
        A[m, 0] = _pow2_code(4)
        A[m, 1:] = _pow2_code(4 - int(ga[m]))
    # columns: (instruction placement, B-side gap part)
    cols = {0: ("same", 0), 1: ("same", 13), 2: ("later", 0), 3: ("later", 13)}
    for n, (where, gb) in cols.items():
        B[n, 0] = _pow2_code(4)
        ks = range(1, 32) if where == "same" else range(32, 128)
        for k in ks:
            B[n, k] = _pow2_code(4 - gb)
    D = fg.fgf8_mma_probe(torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV)).cpu().numpy()
    table = {"same": {}, "later": {}}
    for m in range(14):
        for n, (where, gb) in cols.items():
            g = int(ga[m]) + gb
            exact = oracle.dot_e4m3_exact(A[m], B[n]) / 2.0 ** 18
            best = float(np.float32(exact))
            table[where][g] = {"got": float(D[m, n]), "exact": exact, "fp32": best,
                               "lost_fraction": (exact - float(D[m, n])) / (exact - 256.0)}
    kept = {w: max([g for g, r in t.items() if r["got"] == r["fp32"]] + [-1]) for w, t in table.items()}
    first_loss = {w: min([g for g, r in t.items() if r["got"] != r["fp32"]] + [99]) for w, t in table.items()}
    out = os.environ.get("FGF8_PROBE_OUT")
    if out:
        with open(out, "w") as f:
            json.dump({"kept_through_gap": kept, "first_gap_with_loss": first_loss, "table": table}, f, indent=1)
    print("accumulation probe: largest gap kept", kept, "first gap with loss", first_loss)
    # small gaps must always be exact: the products fit in a few bits
    assert all(table[w][g]["got"] == table[w][g]["fp32"] for w in table for g in range(0, 9))
