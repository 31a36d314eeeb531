"""Pins for the oracle's 1x128, 128x1 and 128x128 quantizers.

Expected values come from hand-worked tiles (tests/golden), tiles built from
exact E4M3 values times powers of two (whose scale and codes are known in
closed form), and invariants of the rule (max-abs element -> +-448, zero
groups, the half-ulp error bound, monotonicity of the block scale).
"""
import os

import numpy as np
import pytest

import oracle
from tests.e4m3_ref import GOLDEN, bf16_bits_from_f32, code_table, f32_from_bf16_bits


def _golden_tiles():
    tiles = []
    with open(os.path.join(GOLDEN, "quant_tile_worked.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, xs, s, cs = [p.strip() for p in line.split("|")]
            x = np.zeros(128, np.float32)
            for item in xs.split():
                i, v = item.split(":")
                x[int(i)] = np.float32(float(v))
            codes = np.zeros(128, np.uint8)
            for item in cs.split():
                i, c = item.split(":")
                codes[int(i)] = int(c, 16)
            tiles.append((name, x, np.float32(float(s)), codes))
    return tiles


@pytest.mark.parametrize("tile", _golden_tiles(), ids=lambda t: t[0])
def test_worked_tiles(tile):
    _, x, s, codes = tile
    bits = bf16_bits_from_f32(x)[None, :]
    q, sc = oracle.quant_act_1x128(bits)
    assert sc[0, 0] == s
    assert np.array_equal(q[0], codes)
    # the same tile as one token-direction tile and inside a weight block
    qT, sT = oracle.quant_act_128x1(np.ascontiguousarray(bits.T))
    assert sT[0, 0] == s and np.array_equal(qT[0], codes)
    blk = np.zeros((128, 128), np.uint16)
    blk[17] = bits[0]
    qw, sw = oracle.quant_w_128x128(blk)
    assert sw[0, 0] == s and np.array_equal(qw[17], codes)


def _random_bf16(rng, shape, sigma=1.0, p_out=0.01, mult=100.0):
    x = rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma)
    mask = rng.random(shape) < p_out
    x = np.where(mask, x * np.float32(mult), x)
    u = x.view(np.uint32)
    # round to nearest even BF16 by integer arithmetic (finite inputs)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def _exact_tensor(rng, rows, cols, group_rows, group_cols):
    """x = decode(c) * 2^j with one +-448 per group, so s = 2^j and q = c exactly."""
    t = code_table()
    finite = np.array([c for c in range(256) if not np.isnan(t[c])], np.uint8)
    c = rng.choice(finite, size=(rows, cols)).astype(np.uint8)
    gr = (rows + group_rows - 1) // group_rows
    gc = cols // group_cols
    j = rng.integers(-12, 12, size=(gr, gc))
    for a in range(gr):
        for b in range(gc):
            r0, r1 = a * group_rows, min(rows, (a + 1) * group_rows)
            c0 = b * group_cols
            rr = rng.integers(r0, r1)
            cc = rng.integers(c0, c0 + group_cols)
            c[rr, cc] = 0x7E if rng.random() < 0.5 else 0xFE
    scale = np.exp2(np.repeat(np.repeat(j, group_rows, 0)[:rows], group_cols, 1))
    x = (t[c] * scale).astype(np.float32)
    return bf16_bits_from_f32(x), c, j


@pytest.mark.parametrize("M", [1, 5, 128, 200])
def test_1x128_exact_construction(M):
    rng = np.random.default_rng(M)
    K = 384
    x, c, j = _exact_tensor(rng, M, K, 1, 128)
    q, s = oracle.quant_act_1x128(x)
    assert np.array_equal(q, c)
    assert s.shape == (K // 128, (M + 3) // 4 * 4)
    assert np.array_equal(s[:, :M], np.exp2(j.T).astype(np.float32))


@pytest.mark.parametrize("M", [128, 130, 255, 384])
def test_128x1_exact_construction(M):
    rng = np.random.default_rng(1000 + M)
    K = 136
    x, c, j = _exact_tensor(rng, M, K, 128, 1)     # token-major [M, K], groups of 128 tokens
    qT, sT = oracle.quant_act_128x1(x)
    assert np.array_equal(qT, np.ascontiguousarray(c.T))
    assert sT.shape == ((M + 127) // 128, K)
    assert np.array_equal(sT[:, :K], np.exp2(j).astype(np.float32))


@pytest.mark.parametrize("N", [128, 200, 256, 390])
def test_128x128_exact_construction(N):
    rng = np.random.default_rng(2000 + N)
    K = 384
    w, c, j = _exact_tensor(rng, N, K, 128, 128)
    q, s = oracle.quant_w_128x128(w)
    assert np.array_equal(q, c)
    nb = (N + 127) // 128
    assert s.shape == (K // 128, (nb + 3) // 4 * 4)
    assert np.array_equal(s[:, :nb], np.exp2(j.T).astype(np.float32))


def _check_invariants(x_groups_f32, q_groups, s_groups):
    """x, q: [G, n]; s: [G].  Max-abs -> +-448, zero group -> s=0, half-ulp bound."""
    t = code_table()
    for xg, qg, sg in zip(x_groups_f32, q_groups, s_groups):
        amax = np.max(np.abs(xg))
        if amax == 0:
            assert sg == 0 and np.all((qg & 0x7F) == 0)
            continue
        assert sg == np.float32(amax) / np.float32(448.0)
        i = np.argmax(np.abs(xg))
        assert qg[i] == (0xFE if xg[i] < 0 else 0x7E)
        y = np.abs(xg.astype(np.float64) / np.float64(sg))
        dq = np.abs(t[qg])
        # e4m3 spacing at |y|: 2^(max(floor(log2 y), -6) - 3); plus the binary32
        # rounding of x/s (relative 2^-24) that precedes the E4M3 rounding
        e = np.floor(np.log2(np.maximum(y, 2.0 ** -40)))
        ulp = np.exp2(np.maximum(e, -6) - 3)
        assert np.all(np.abs(dq - y) <= 0.5 * ulp + y * 2.0 ** -24 + 1e-300)
        assert np.all(np.isfinite(t[qg]))
        nz = xg != 0
        assert np.all(np.signbit(xg[nz]) == ((qg[nz] & 0x80) != 0))


def test_invariants_1x128_random_outliers():
    rng = np.random.default_rng(11)
    x = _random_bf16(rng, (64, 1024), 1.0, 0.01, 100.0)
    x[3, 128:256] = 0
    x[4, 0:128] = 0x8000        # a tile of negative zeros
    q, s = oracle.quant_act_1x128(x)
    xf = f32_from_bf16_bits(x)
    G = xf.reshape(64, 8, 128).reshape(-1, 128)
    Q = q.reshape(64, 8, 128).reshape(-1, 128)
    S = s[:, :64].T.reshape(-1)
    _check_invariants(G, Q, S)
    assert np.all(q[4, 0:128] == 0x80)


def test_invariants_128x1_random_ragged():
    rng = np.random.default_rng(12)
    M, K = 300, 256
    x = _random_bf16(rng, (M, K), 1.0, 0.001, 50.0)
    qT, sT = oracle.quant_act_128x1(x)
    xf = f32_from_bf16_bits(x)
    for tb in range(3):
        m0, m1 = tb * 128, min(M, tb * 128 + 128)
        _check_invariants(xf[m0:m1].T, qT[:, m0:m1], sT[tb, :K])


def test_invariants_128x128_random_ragged():
    rng = np.random.default_rng(13)
    N, K = 300, 384
    w = _random_bf16(rng, (N, K), 0.02, 0.0, 1.0)
    q, s = oracle.quant_w_128x128(w)
    wf = f32_from_bf16_bits(w)
    for nb in range(3):
        for kb in range(3):
            blk = wf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            qb = q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            _check_invariants(blk.reshape(1, -1), qb.reshape(1, -1), [s[kb, nb]])


def test_128x1_equals_1x128_of_transpose():
    rng = np.random.default_rng(14)
    x = _random_bf16(rng, (256, 384), 1.0, 0.01, 100.0)
    qT, sT = oracle.quant_act_128x1(x)
    q2, s2 = oracle.quant_act_1x128(np.ascontiguousarray(x.T))
    assert np.array_equal(qT, q2)
    assert np.array_equal(sT[:, :384], s2[:, :384])


def test_block_scale_is_max_of_row_scales():
    # s = fl(amax/448) is monotone in amax, so a block's scale is the largest
    # 1x128 scale of its rows (ragged last block included)
    rng = np.random.default_rng(15)
    w = _random_bf16(rng, (330, 256), 0.02, 0.001, 50.0)
    _, sw = oracle.quant_w_128x128(w)
    _, sr = oracle.quant_act_1x128(w)
    for nb in range(3):
        for kb in range(2):
            assert sw[kb, nb] == sr[kb, nb * 128:min(330, nb * 128 + 128)].max()


# --- the transposed weight operand of the data-gradient GEMM (dX = dY * W) ---


@pytest.mark.parametrize("N,K", [(256, 384), (384, 128), (128, 640)])
def test_transposed_weight_blocks_commute_with_transposition(N, K):
    # A 128x128 block of W^T holds the elements of one block of W: same amax,
    # same scale, same codes -- quantizing W^T must give the transpose of the
    # quantized W.  N != K so that a swapped index or leading dimension shows.
    rng = np.random.default_rng(N * 7 + K)
    w = _random_bf16(rng, (N, K), 0.02, 0.01, 50.0)
    q, s = oracle.quant_w_128x128(w)
    qT, sT = oracle.quant_w_128x128_t(w)
    assert qT.shape == (K, N)
    assert np.array_equal(qT, q.T)
    assert np.array_equal(sT[:, : K // 128], s[:, : N // 128].T)


def test_transposed_weight_block_closed_form():
    # blocks built from exact E4M3 values x 2^j: the scale of block (nb, kb) is
    # 2^j[nb, kb] and the codes are the construction's, read transposed
    rng = np.random.default_rng(11)
    bits, c, j = _exact_tensor(rng, 256, 384, 128, 128)
    qT, sT = oracle.quant_w_128x128_t(bits)
    assert np.array_equal(qT, c.T)
    for nb in range(2):
        for kb in range(3):
            assert sT[nb, kb] == np.float32(2.0 ** j[nb, kb])
