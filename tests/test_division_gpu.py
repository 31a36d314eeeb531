"""The quantizers compute x / s with a correctly rounded reciprocal and one
fused correction step instead of CUDA's IEEE division; the quotient must be
the same binary32 value bit for bit, or the E4M3 codes would differ from the
oracle's.  Checked against CUDA's __fdiv_rn on the device over the inputs the
quantizers see (BF16 x, s = fl32(amax / 448) with amax >= |x|) and on generic
binary32 pairs, including subnormal and huge scales."""
import numpy as np
import pytest
import torch

import fine_grained_fp8_weight_b300 as fg
from fine_grained_fp8_weight_b300 import workloads as wl
from tests.gpu_util import DEV, ensure_built

pytestmark = pytest.mark.gpu


def _run(x, s):
    L = ensure_built()
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(DEV)
    sd = torch.from_numpy(np.ascontiguousarray(s, np.float32)).to(DEV)
    fast = torch.empty_like(xd)
    ieee = torch.empty_like(xd)
    assert L.fgf8_selftest_scaled_div(fg._ptr(xd), fg._ptr(sd), xd.numel(), fg._ptr(fast), fg._ptr(ieee),
                                      fg._stream(xd.device)) == 0
    torch.cuda.synchronize()
    return fast.cpu().numpy(), ieee.cpu().numpy()


def _assert_same_bits(fast, ieee, x, s):
    """Identical quotients wherever the bits can decide an E4M3 code.  The one
    exception the kernels allow: |x| < 2^-100 in a group with s >= 2^-90 has
    |x/s| < 2^-10, below every E4M3 rounding midpoint, so only the sign and
    the fact that it rounds to zero matter there."""
    tiny = (np.abs(x) < 2.0 ** -100) & (s >= 2.0 ** -90) & (s <= 2.0 ** 125)
    bad = np.nonzero((fast.view(np.uint32) != ieee.view(np.uint32)) & ~tiny)[0]
    assert bad.size == 0, f"{bad.size} differing quotients, e.g. x={x[bad[:3]]} s={s[bad[:3]]}"
    t = np.nonzero(tiny)[0]
    assert np.all(np.abs(fast[t]) <= 2.0 ** -10) and np.all(np.abs(ieee[t]) < 2.0 ** -10)
    assert np.array_equal(np.signbit(fast[t]), np.signbit(ieee[t]))
    codes_fast = torch.from_numpy(fast[t]).to(torch.float8_e4m3fn).view(torch.uint8)
    codes_ieee = torch.from_numpy(ieee[t]).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(codes_fast, codes_ieee)


def test_quantizer_domain_bf16():
    rng = np.random.default_rng(77)
    n = 1 << 24
    amax_bits = wl.to_bf16_bits((np.exp2(rng.uniform(-133, 127, n)) * rng.uniform(1, 2, n)).astype(np.float32))
    amax = (amax_bits.astype(np.uint32) << 16).view(np.float32)
    amax = np.where(np.isfinite(amax), amax, np.float32(1.0))
    s = (amax / np.float32(448.0)).astype(np.float32)
    frac = rng.uniform(-1, 1, n).astype(np.float32) * np.where(rng.random(n) < 0.1, np.float32(1), np.exp2(
        -rng.uniform(0, 30, n)).astype(np.float32))
    x = (wl.to_bf16_bits(amax * frac).astype(np.uint32) << 16).view(np.float32)
    x = np.where(np.abs(x) <= amax, x, amax)
    fast, ieee = _run(x, s)
    _assert_same_bits(fast, ieee, x, s)


def test_generic_binary32_pairs():
    rng = np.random.default_rng(78)
    n = 1 << 24
    s = (rng.integers(0x00000001, 0x7F000000, n, dtype=np.uint32)).view(np.float32)   # subnormal .. huge
    q = rng.uniform(-512, 512, n).astype(np.float32) * np.where(rng.random(n) < 0.5, np.float32(1),
                                                                 np.exp2(-rng.uniform(0, 40, n)).astype(np.float32))
    x = (q.astype(np.float64) * s.astype(np.float64)).astype(np.float32)
    x = np.where(np.isfinite(x), x, np.float32(0))
    fast, ieee = _run(x, s)
    _assert_same_bits(fast, ieee, x, s)


def test_midpoint_quotients():
    # quotients that land on or next to E4M3 rounding midpoints, where one
    # binary32 ulp decides the code
    rng = np.random.default_rng(79)
    mids = np.array([17, 19, 168, 336, 0.0009765625, 0.0029296875, 2.25, 440, 27, 52], np.float64)
    s = (np.exp2(rng.uniform(-100, 100, 1 << 20))).astype(np.float32)
    m = rng.choice(mids, size=s.size)
    x = (m * s.astype(np.float64)).astype(np.float32)
    x = np.concatenate([x, np.nextafter(x, np.float32(np.inf)), np.nextafter(x, np.float32(0))])
    s = np.concatenate([s, s, s])
    fast, ieee = _run(x, s)
    _assert_same_bits(fast, ieee, x, s)
