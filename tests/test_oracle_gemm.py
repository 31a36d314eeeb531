"""Pins for the oracle's block-scaled GEMM, grouped GEMM and exact dot product.

Expected values come from exact rational arithmetic (fractions), integer
matrix products (numpy int64 matmul) on cases where every dequantized product
is exact, and identity-like operands -- never from the oracle itself.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.e4m3_ref import code_table

T = code_table()
FINITE = np.array([c for c in range(256) if not np.isnan(T[c])], np.uint8)
# codes of the integers -8..8 (all exactly representable in E4M3)
INT_CODE = {int(T[c]): c for c in range(256) if not np.isnan(T[c]) and T[c] == int(T[c])
            and abs(T[c]) <= 8 and not (T[c] == 0 and c == 0x80)}


def _int_codes(rng, shape):
    vals = rng.integers(-8, 9, size=shape)
    codes = np.vectorize(lambda v: INT_CODE[int(v)])(vals).astype(np.uint8)
    return vals.astype(np.int64), codes


def _exact_reference(A, sa, B, sb, bkind):
    M, K = A.shape
    N = B.shape[0]
    C = [[Fraction(0)] * N for _ in range(M)]
    S = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            mag = Fraction(0)
            for k in range(K):
                kb = k // 128
                a = Fraction(float(T[A[m, k]])) * Fraction(float(sa[kb, m]))
                sbv = sb[kb, n // 128] if bkind == 0 else sb[kb, n]
                b = Fraction(float(T[B[n, k]])) * Fraction(float(sbv))
                acc += a * b
                mag += abs(a * b)
            C[m][n] = acc
            S[m][n] = mag
    return C, S


@pytest.mark.parametrize("K,bkind", [(128, 0), (512, 0), (256, 1)])
def test_gemm_exact_rational_small(K, bkind):
    rng = np.random.default_rng(K + bkind)
    M, N = 4, 4
    A = rng.choice(FINITE, size=(M, K))
    B = rng.choice(FINITE, size=(N, K))
    sa = np.exp(rng.uniform(-8, 4, size=(K // 128, M))).astype(np.float32)
    sb = np.exp(rng.uniform(-8, 4, size=(K // 128, 4 if bkind == 0 else N))).astype(np.float32)
    C, S = oracle.gemm_blockscaled(A, sa, B, sb, bkind)
    Ce, Se = _exact_reference(A, sa, B, sb, bkind)
    for m in range(M):
        for n in range(N):
            bound = 4 * K * 2.0 ** -53 * float(Se[m][n])
            assert abs(C[m, n] - float(Ce[m][n])) <= bound
            assert abs(S[m, n] - float(Se[m][n])) <= bound


def test_gemm_integer_case_is_int_matmul():
    rng = np.random.default_rng(21)
    M, N, K = 5, 7, 256
    av, A = _int_codes(rng, (M, K))
    bv, B = _int_codes(rng, (N, K))
    sa = np.ones((K // 128, 8), np.float32)
    sb = np.ones((K // 128, 4), np.float32)
    C, S = oracle.gemm_blockscaled(A, sa, B, sb, 0)
    assert np.array_equal(C, (av @ bv.T).astype(np.float64))
    assert np.array_equal(S, (np.abs(av) @ np.abs(bv).T).astype(np.float64))


@pytest.mark.parametrize("bkind", [0, 1])
def test_gemm_power_of_two_scales_index_pin(bkind):
    # distinct power-of-two scales per (K group, row) and per (K group, column
    # block or column): every product is exact, so the blocked integer matmul
    # below is exact and any wrong scale index, transposed operand or dropped
    # K group changes the result
    rng = np.random.default_rng(22 + bkind)
    M, N, K = 130, 260, 384
    av, A = _int_codes(rng, (M, K))
    bv, B = _int_codes(rng, (N, K))
    KB = K // 128
    ja = rng.integers(-6, 7, size=(KB, M))
    nb = (N + 127) // 128
    jb = rng.integers(-6, 7, size=(KB, nb if bkind == 0 else N))
    sa = np.zeros((KB, 132), np.float32)
    sa[:, :M] = np.exp2(ja)
    ldb = 4 if bkind == 0 else 260
    sb = np.zeros((KB, ldb), np.float32)
    sb[:, :jb.shape[1]] = np.exp2(jb)
    C, _ = oracle.gemm_blockscaled(A, sa, B, sb, bkind)
    ref = np.zeros((M, N))
    for kb in range(KB):
        part = (av[:, kb * 128:(kb + 1) * 128] @ bv[:, kb * 128:(kb + 1) * 128].T).astype(np.float64)
        colscale = np.exp2(np.repeat(jb[kb], 128)[:N]) if bkind == 0 else np.exp2(jb[kb])
        ref += part * np.exp2(ja[kb])[:, None] * colscale[None, :]
    assert np.array_equal(C, ref)


def test_gemm_identity_block_reproduces_dequantized_a():
    rng = np.random.default_rng(23)
    M, K = 6, 256
    A = rng.choice(FINITE, size=(M, K))
    sa = np.exp(rng.uniform(-4, 4, size=(K // 128, 8))).astype(np.float32)
    N = K
    B = np.zeros((N, K), np.uint8)
    B[np.arange(N), np.arange(N)] = 0x38          # 1.0
    sb = np.zeros((K // 128, 4), np.float32)
    sb[:, :2] = [[0.5, 1.0], [2.0, 4.0]]          # sb[kb][nb]: only kb == nb meets the diagonal
    C, _ = oracle.gemm_blockscaled(A, sa, B, sb, 0)
    ahat = T[A] * np.repeat(sa[:, :M].T, 128, axis=1).astype(np.float64)
    colscale = np.array([0.5] * 128 + [4.0] * 128)
    assert np.array_equal(C, ahat * colscale[None, :])


def test_gemm_row_subset_matches_full():
    rng = np.random.default_rng(24)
    A = rng.choice(FINITE, size=(40, 256))
    B = rng.choice(FINITE, size=(24, 256))
    sa = np.ones((2, 40), np.float32)
    sb = np.ones((2, 4), np.float32)
    av = T[A]; bv = T[B]
    rows = [39, 0, 17]
    C, _ = oracle.gemm_blockscaled(A, sa, B, sb, 0, rows=rows)
    # products of E4M3 values are exact in binary64 and the row sums of up to
    # 256 such products of at most 448^2 stay exact (multiples of 2^-18 below 2^53)
    assert np.array_equal(C, (av @ bv.T)[rows])


def test_grouped_gemm_integer_experts():
    rng = np.random.default_rng(25)
    E, N, K = 3, 136, 256
    counts = [130, 0, 70]
    m_idx = []
    for e, c in enumerate(counts):
        pad = (c + 127) // 128 * 128
        m_idx += [e] * c + [-1] * (pad - c)
    m_idx = np.array(m_idx, np.int32)
    M = len(m_idx)
    av, A = _int_codes(rng, (M, K))
    bv, B = _int_codes(rng, (E, N, K))
    ja = rng.integers(-3, 4, size=(K // 128, M))
    jb = rng.integers(-3, 4, size=(E, K // 128, 2))
    sa = np.exp2(ja).astype(np.float32)
    sb = np.zeros((E, K // 128, 4), np.float32)
    sb[:, :, :2] = np.exp2(jb)
    C, S = oracle.grouped_gemm_blockscaled(A, sa, B, sb, m_idx)
    for m in range(M):
        e = m_idx[m]
        if e < 0:
            assert np.all(np.isnan(C[m])) and np.all(S[m] == 0)
            continue
        ref = np.zeros(N)
        for kb in range(K // 128):
            part = (bv[e][:, kb * 128:(kb + 1) * 128] @ av[m, kb * 128:(kb + 1) * 128]).astype(np.float64)
            ref += part * 2.0 ** ja[kb, m] * np.exp2(np.repeat(jb[e, kb], 128)[:N])
        assert np.array_equal(C[m], ref)


def test_dot_exact_matches_fractions():
    rng = np.random.default_rng(26)
    for K in (32, 128, 1000):
        a = rng.choice(FINITE, size=K)
        b = rng.choice(FINITE, size=K)
        exact = sum(Fraction(float(T[x])) * Fraction(float(T[y])) for x, y in zip(a, b))
        assert Fraction(oracle.dot_e4m3_exact(a, b), 2 ** 18) == exact


def _masked_case(seed, E, cap, N, K, counts):
    rng = np.random.default_rng(seed)
    av, A = _int_codes(rng, (E, cap, K))
    bv, B = _int_codes(rng, (E, N, K))
    ja = rng.integers(-3, 4, size=(E, K // 128, cap))
    jb = rng.integers(-3, 4, size=(E, K // 128, (N + 127) // 128))
    sa = np.zeros((K // 128, E * cap + 4), np.float32)          # stacked slots, spare columns
    for e in range(E):
        sa[:, e * cap:(e + 1) * cap] = np.exp2(ja[e])
    sb = np.zeros((E, K // 128, ((N + 127) // 128 + 3) // 4 * 4), np.float32)
    sb[:, :, :jb.shape[2]] = np.exp2(jb)
    return av, A, bv, B, ja, jb, sa, sb


def test_masked_grouped_integer_experts():
    # exact: integer codes, power-of-two scales, sums far below 2^53
    E, cap, N, K = 3, 48, 144, 256
    counts = np.array([48, 0, 17], np.int32)      # cap 48: slots need not be powers of two
    av, A, bv, B, ja, jb, sa, sb = _masked_case(31, E, cap, N, K, counts)
    C, S = oracle.masked_grouped_gemm_blockscaled(A, sa, B, sb, counts)
    for e in range(E):
        for m in range(cap):
            if m >= counts[e]:
                assert np.all(np.isnan(C[e, m])) and np.all(S[e, m] == 0)
                continue
            ref = np.zeros(N)
            for kb in range(K // 128):
                part = (bv[e][:, kb * 128:(kb + 1) * 128] @ av[e, m, kb * 128:(kb + 1) * 128]).astype(np.float64)
                ref += part * 2.0 ** ja[e, kb, m] * np.exp2(np.repeat(jb[e, kb], 128)[:N])
            assert np.array_equal(C[e, m], ref)


def test_masked_grouped_equals_contiguous_grouped():
    # the masked slots, packed into the contiguous padded layout, must give the
    # contiguous-layout routine's result row for row (a separate code path)
    E, cap, N, K = 4, 64, 256, 384
    counts = np.array([64, 5, 0, 33], np.int32)
    _, A, _, B, _, _, sa, sb = _masked_case(32, E, cap, N, K, counts)
    Cm, Sm = oracle.masked_grouped_gemm_blockscaled(A, sa, B, sb, counts)
    rows, m_idx, sa_c = [], [], []
    for e in range(E):
        pad = (int(counts[e]) + 127) // 128 * 128
        for r in range(pad):
            rows.append(A[e, r] if r < counts[e] else np.zeros(K, np.uint8))
            m_idx.append(e if r < counts[e] else -1)
            sa_c.append(sa[:, e * cap + r] if r < counts[e] else np.zeros(K // 128, np.float32))
    Ac = np.stack(rows)
    sac = np.zeros((K // 128, (len(rows) + 3) // 4 * 4), np.float32)
    sac[:, :len(rows)] = np.stack(sa_c, axis=1)
    Cc, Sc = oracle.grouped_gemm_blockscaled(Ac, sac, B, sb, np.array(m_idx, np.int32))
    i = 0
    for e in range(E):
        pad = (int(counts[e]) + 127) // 128 * 128
        for r in range(int(counts[e])):
            assert np.array_equal(Cm[e, r], Cc[i + r]) and np.array_equal(Sm[e, r], Sc[i + r])
        i += pad


def test_masked_counts_outside_the_slot_are_clamped():
    # a count past the slot stands for the whole slot and a negative count for
    # none (the masked GEMM's argument rule); exact sums as above
    E, cap, N, K = 3, 32, 128, 256
    counts = np.array([cap + 7, -2, 5], np.int32)
    used = [cap, 0, 5]
    av, A, bv, B, ja, jb, sa, sb = _masked_case(33, E, cap, N, K, counts)
    C, S = oracle.masked_grouped_gemm_blockscaled(A, sa, B, sb, counts)
    for e in range(E):
        for m in range(cap):
            if m >= used[e]:
                assert np.all(np.isnan(C[e, m])) and np.all(S[e, m] == 0)
                continue
            ref = np.zeros(N)
            for kb in range(K // 128):
                part = (bv[e][:, kb * 128:(kb + 1) * 128] @ av[e, m, kb * 128:(kb + 1) * 128]).astype(np.float64)
                ref += part * 2.0 ** ja[e, kb, m] * np.exp2(np.repeat(jb[e, kb], 128)[:N])
            assert np.array_equal(C[e, m], ref)
