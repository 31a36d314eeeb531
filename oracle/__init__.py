"""CPU parity oracle for fine-grained FP8 quantization and block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; the product path never imports it.
It wraps ``oracle.c`` (plain C, binary64 GEMM) through ctypes and shares no
code with the CUDA library.  Every function cites the passage it follows in
``oracle.c``.

Arrays are numpy arrays; BF16 tensors are passed as their ``uint16`` bit
patterns so that no library conversion sits between the test inputs and the
oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# No -ffast-math and no FMA contraction: the binary32 divisions and binary64
# sums must be the plain IEEE operations written in the source.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    """The oracle library.  ``FGF8_ORACLE_LIB`` names another build of the
    oracle source to load instead (the mutation test uses it to run the pins
    against copies of the oracle with planted mistakes)."""
    global _lib
    if _lib is None:
        path = os.environ.get("FGF8_ORACLE_LIB")
        if not path:
            path = build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode_array.argtypes = [P, I64, P]
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_decode.restype = ctypes.c_double
        L.oracle_quant_act_1x128.argtypes = [P, I64, I64, I64, P, P, I64]
        L.oracle_quant_act_128x1.argtypes = [P, I64, I64, I64, P, P, I64]
        L.oracle_quant_w_128x128.argtypes = [P, I64, I64, I64, P, P, I64]
        L.oracle_gemm_blockscaled.argtypes = [P, P, I64, P, P, I64, ctypes.c_int,
                                              I64, I64, I64, P, I64, P, P]
        L.oracle_grouped_gemm_blockscaled.argtypes = [P, P, I64, P, P, I64, P, ctypes.c_int32,
                                                      I64, I64, I64, P, I64, P, P]
        L.oracle_dot_e4m3_exact.argtypes = [P, P, I64]
        L.oracle_dot_e4m3_exact.restype = ctypes.c_int64
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, "BF16 inputs are passed as uint16 bit patterns"
    return x


def round_up(v: int, m: int) -> int:
    return (v + m - 1) // m * m


def e4m3_encode(v: float) -> int:
    """E4M3 code of one binary32 value, RNE with saturation."""
    return int(lib().oracle_e4m3_encode(ctypes.c_float(v)))


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    """Element-wise E4M3 codes of a binary32 array."""
    v = np.ascontiguousarray(v, np.float32)
    out = np.zeros(v.shape, np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode(c: int) -> float:
    """Exact value of one E4M3 code."""
    return float(lib().oracle_e4m3_decode(ctypes.c_uint8(c)))


def e4m3_decode_array(q: np.ndarray) -> np.ndarray:
    table = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[q]


def quant_act_1x128(x_bits: np.ndarray):
    """1x128 tiles along K.  Returns (q [M,K] uint8, s [K/128, round_up(M,4)] float32)."""
    x = _bits16(x_bits)
    M, K = x.shape
    lds = round_up(M, 4)
    q = np.zeros((M, K), np.uint8)
    s = np.zeros((K // 128, lds), np.float32)
    lib().oracle_quant_act_1x128(_ptr(x), M, K, K, _ptr(q), _ptr(s), lds)
    return q, s


def quant_act_128x1(x_bits: np.ndarray):
    """128x1 tiles along M, transposed output.

    Returns (qT [K,M] uint8, sT [ceil(M/128), round_up(K,4)] float32)."""
    x = _bits16(x_bits)
    M, K = x.shape
    ldsT = round_up(K, 4)
    qT = np.zeros((K, M), np.uint8)
    sT = np.zeros(((M + 127) // 128, ldsT), np.float32)
    lib().oracle_quant_act_128x1(_ptr(x), M, K, K, _ptr(qT), _ptr(sT), ldsT)
    return qT, sT


def quant_w_128x128(w_bits: np.ndarray):
    """128x128 blocks.  Returns (q [N,K] uint8, s [K/128, round_up(ceil(N/128),4)] float32)."""
    w = _bits16(w_bits)
    N, K = w.shape
    lds = round_up((N + 127) // 128, 4)
    q = np.zeros((N, K), np.uint8)
    s = np.zeros((K // 128, lds), np.float32)
    lib().oracle_quant_w_128x128(_ptr(w), N, K, K, _ptr(q), _ptr(s), lds)
    return q, s


def quant_w_128x128_t(w_bits: np.ndarray):
    """The 128x128 block quantization of W^T (W: BF16 bits [N, K]), i.e. the B
    operand of the data-gradient GEMM dX = dY * W, whose inner dimension is N.
    It is the 128x128 rule applied to the transposed matrix, literally.
    Returns (qT [K, N] uint8, sT [N/128, round_up(K/128, 4)] float32) with
    sT[nb, kb] the scale of the block of rows nb*128.. and columns kb*128.. of W."""
    return quant_w_128x128(np.ascontiguousarray(np.asarray(w_bits, np.uint16).T))


def gemm_blockscaled(A, sa, B, sb, bkind: int = 0, rows=None):
    """Binary64 reference of C = A_hat * B_hat^T and the magnitude sum S.

    A [M,K] codes with sa [K/128, lda_s]; B [N,K] codes with sb [K/128, ldb_s]
    (bkind 0: 128x128 block scales indexed by n/128; bkind 1: per-row scales
    indexed by n).  ``rows``: optional list of A rows to evaluate."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32)
    sb = np.ascontiguousarray(sb, np.float32)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K and K % 128 == 0
    if rows is None:
        nr, rp = M, None
    else:
        rows = np.ascontiguousarray(rows, np.int64)
        nr, rp = len(rows), rows
    C = np.zeros((nr, N), np.float64)
    S = np.zeros((nr, N), np.float64)
    lib().oracle_gemm_blockscaled(_ptr(A), _ptr(sa), sa.shape[1], _ptr(B), _ptr(sb), sb.shape[1],
                                  bkind, M, N, K, _ptr(rp) if rp is not None else None, nr,
                                  _ptr(C), _ptr(S))
    return C, S


def grouped_gemm_blockscaled(A, sa, B, sb, m_indices, rows=None):
    """Grouped contiguous-layout reference.  B [E,N,K], sb [E,K/128,ldb_s];
    padding rows (m_indices < 0) come back as NaN with S = 0."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32)
    sb = np.ascontiguousarray(sb, np.float32)
    mi = np.ascontiguousarray(m_indices, np.int32)
    M, K = A.shape
    E, N, _ = B.shape
    if rows is None:
        nr, rp = M, None
    else:
        rows = np.ascontiguousarray(rows, np.int64)
        nr, rp = len(rows), rows
    C = np.zeros((nr, N), np.float64)
    S = np.zeros((nr, N), np.float64)
    lib().oracle_grouped_gemm_blockscaled(_ptr(A), _ptr(sa), sa.shape[1], _ptr(B), _ptr(sb),
                                          sb.shape[2], _ptr(mi), E, M, N, K,
                                          _ptr(rp) if rp is not None else None, nr,
                                          _ptr(C), _ptr(S))
    return C, S


def masked_grouped_gemm_blockscaled(A, sa, B, sb, counts, rows_per_expert=None):
    """Masked-layout grouped reference (decode MoE): expert e owns a slot of
    `cap` token rows, of which the first counts[e] are real.
    A [E, cap, K] codes with sa [K/128, lda_s] the scales of the stacked slots
    (expert e's token m in column e*cap + m, as a 1x128 quantization of the
    [E*cap, K] buffer writes them); B [E, N, K], sb [E, K/128, ldb_s].
    Returns C, S of shape [E, cap, N]: for every expert the dense block-scaled
    GEMM of its real rows with its own weights; rows past the count are NaN
    (S = 0).  ``rows_per_expert``: optional list of row indices to evaluate
    within each expert's real rows."""
    A = np.ascontiguousarray(A, np.uint8)
    E, cap, K = A.shape
    N = B.shape[1]
    C = np.full((E, cap, N), np.nan)
    S = np.zeros((E, cap, N))
    for e in range(E):
        c = int(min(max(int(counts[e]), 0), cap))
        if c == 0:
            continue
        rows = None
        if rows_per_expert is not None:
            rows = [r for r in rows_per_expert if r < c]
            if not rows:
                continue
        sa_e = np.ascontiguousarray(np.asarray(sa, np.float32)[:, e * cap:(e + 1) * cap])
        Ce, Se = gemm_blockscaled(A[e, :c], sa_e, B[e], sb[e], 0, rows=rows)
        idx = rows if rows is not None else slice(0, c)
        C[e, idx] = Ce
        S[e, idx] = Se
    return C, S


def dot_e4m3_exact(a_codes, b_codes) -> int:
    """Exact dot product of two E4M3 code vectors, in units of 2^-18."""
    a = np.ascontiguousarray(a_codes, np.uint8)
    b = np.ascontiguousarray(b_codes, np.uint8)
    assert a.shape == b.shape
    return int(lib().oracle_dot_e4m3_exact(_ptr(a), _ptr(b), a.size))
