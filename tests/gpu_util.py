"""Helpers for the GPU parity tests: move the seeded host inputs to the
device, run the C-ABI path, and compare with the oracle."""
import numpy as np
import torch

import fine_grained_fp8_weight_b300 as fg
from fine_grained_fp8_weight_b300 import build as fgbuild
from fine_grained_fp8_weight_b300 import workloads as wl

DEV = "cuda:0"

# (label, max, mean, elements) of |C - C_ref| / S per full-size configuration,
# printed in the test session's summary
MARGINS = []


def report_margin(label: str, margin, n: int):
    MARGINS.append((label, margin[0], margin[1], int(n)))


def ensure_built():
    fgbuild.build()
    return fg.lib()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return wl.bf16_bits_to_torch(bits).to(DEV)


def host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def bf16_out_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_scales_equal(gpu_s: np.ndarray, ref_s: np.ndarray, used_cols: int):
    """Bit-exact comparison of the used part of a scale array."""
    g = np.ascontiguousarray(gpu_s[:, :used_cols]).view(np.uint32)
    r = np.ascontiguousarray(ref_s[:, :used_cols]).view(np.uint32)
    bad = np.argwhere(g != r)
    assert bad.size == 0, f"{len(bad)} scale mismatches, first at {bad[:5].tolist()}"


def assert_codes_equal(gpu_q: np.ndarray, ref_q: np.ndarray):
    bad = np.argwhere(gpu_q != ref_q)
    assert bad.size == 0, (f"{len(bad)} code mismatches, first at {bad[:5].tolist()}: "
                           f"gpu {[hex(gpu_q[tuple(i)]) for i in bad[:5]]} ref {[hex(ref_q[tuple(i)]) for i in bad[:5]]}")


def assert_within_bound(C_gpu: np.ndarray, C_ref: np.ndarray, S: np.ndarray, label: str = ""):
    """|C_gpu - C_ref| <= 2^-7 * S + 1e-6, elementwise (the GEMM's stated tolerance)."""
    err = np.abs(C_gpu - C_ref)
    bound = 2.0 ** -7 * S + 1e-6
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, (f"{label}: {len(bad)} elements outside the bound, first {bad[:5].tolist()}, "
                           f"err {err[tuple(bad[0])] if bad.size else 0}, bound {bound[tuple(bad[0])] if bad.size else 0}")
    with np.errstate(invalid="ignore", divide="ignore"):
        rel = np.where(S > 0, err / S, 0.0)
    return float(rel.max()), float(rel.mean())
