"""Independent E4M3 helpers for the oracle's pin tests.

The code -> value table comes from torch's ``float8_e4m3fn`` dtype (a library
implementation of the OCP E4M3 format) and is cross-checked against the
hand-written golden table; the nearest-code search is brute force over all
finite codes.  Nothing here is shared with the oracle or the CUDA library.
"""
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def code_table() -> np.ndarray:
    """Value of every one of the 256 codes, as float64 (NaN for the two NaN codes)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def golden_codes():
    out = []
    with open(os.path.join(GOLDEN, "e4m3_codes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            out.append((int(c, 16), float(v)))
    return out


_POS = None


def _positive_finite():
    global _POS
    if _POS is None:
        t = code_table()
        _POS = t[:0x7F].copy()          # codes 0x00..0x7E: 0 .. 448
    return _POS


def brute_force_encode(v: np.ndarray, chunk: int = 20000) -> np.ndarray:
    """Nearest finite E4M3 code to each binary32 value, ties to the code with
    an even mantissa (even code number), sign copied from the input.  Values
    beyond 448 have 448 as their nearest finite code, which is saturation."""
    v = np.asarray(v, np.float32).ravel()
    table = _positive_finite()
    out = np.empty(v.size, np.uint8)
    for i in range(0, v.size, chunk):
        # Above 448 every finite code keeps its distance order, so the
        # magnitude is capped where binary64 differences are still exact.
        a = np.minimum(np.abs(v[i:i + chunk].astype(np.float64)), 2.0 ** 20)
        d = np.abs(table[None, :] - a[:, None])
        c = np.argmin(d, axis=1)                      # lowest code among equals
        n = np.minimum(c + 1, table.size - 1)
        tie = (d[np.arange(c.size), n] == d[np.arange(c.size), c]) & (n != c)
        c = np.where(tie & (c % 2 == 1), n, c)
        sign = np.signbit(v[i:i + chunk]).astype(np.uint8) << 7
        out[i:i + chunk] = c.astype(np.uint8) | sign
    return out


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """BF16 bits of binary32 values that are exactly representable in BF16."""
    x = np.ascontiguousarray(x, np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not representable in BF16"
    return (u >> 16).astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint32) << 16).view(np.float32)
