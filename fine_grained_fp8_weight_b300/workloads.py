"""Seeded synthetic inputs for the fine-grained FP8 path.

This module only draws random numbers: it holds none of the quantization or
GEMM arithmetic, and both the CUDA path's tests and the CPU oracle read the
same host arrays it returns.  Every tensor is returned as the ``uint16`` bit
pattern of a BF16 array (numpy), so that the oracle and the device path see
bit-identical inputs.

Recipe (stated once, used everywhere): ``numpy.random.default_rng(seed)``;
each tensor is drawn as binary32 ``standard_normal * sigma``; where the
workload has outliers, a Bernoulli(p) mask is drawn next
(``rng.random(shape) < p``) and the masked entries are multiplied by
``mult``; the result is rounded once to BF16 (round-to-nearest-even).  Draws
happen in the order each workload function lists them.  The shapes and
distributions are those of the five workloads: a tiny reference GEMM, a
prefill projection pair, decode-size GEMMs, a grouped MoE expert GEMM and a
weight-gradient GEMM.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

ROW_BLOCK = 128     # tokens per group in the contiguous grouped layout


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 to BF16 (nearest even) and return the uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_normal(rng: np.random.Generator, shape, sigma: float = 1.0,
                p_out: float = 0.0, mult: float = 1.0, chunk_rows: int = 2048) -> np.ndarray:
    """BF16 bits of sigma * N(0,1), with a fraction p_out of entries times mult.

    Drawn in row chunks (normal draws of a chunk, then its mask) so that large
    tensors never hold more than one binary32 chunk."""
    shape = tuple(int(s) for s in shape)
    rows = shape[0]
    rest = shape[1:]
    out = np.empty(shape, np.uint16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = rng.standard_normal((r1 - r0, *rest), dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        if p_out > 0.0:
            mask = rng.random((r1 - r0, *rest)) < p_out
            x[mask] *= np.float32(mult)
        out[r0:r1] = to_bf16_bits(x)
    return out


def bf16_bits_to_torch(bits: np.ndarray) -> torch.Tensor:
    """A CPU torch.bfloat16 tensor sharing the bits (no rounding)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


# ----------------------------------------------------------------- shapes --

@dataclass
class Dense:
    """One dense GEMM C[M,N] = A[M,K] * B[N,K]^T with BF16 inputs."""
    name: str
    A: np.ndarray
    B: np.ndarray
    out: str = "bf16"


@dataclass
class Grouped:
    """Grouped contiguous-layout GEMM: rows of A belong to experts."""
    name: str
    A: np.ndarray                 # [M_pad, K], padding rows are zero
    B: np.ndarray                 # [E, N, K]
    m_indices: np.ndarray         # [M_pad] int32, -1 for padding
    counts: np.ndarray            # [E] real tokens per expert
    out: str = "bf16"


@dataclass
class Wgrad:
    """dW[N,K] = dY[T,N]^T * X[T,K], both operands quantized along T."""
    name: str
    dY: np.ndarray
    X: np.ndarray
    out: str = "fp32"


@dataclass
class Dgrad:
    """dX[T,K] = dY[T,N] * W[N,K]: dY quantized 1x128 along N, W as W^T in
    128x128 blocks (the GEMM's B operand [K,N])."""
    name: str
    dY: np.ndarray
    W: np.ndarray
    out: str = "bf16"


@dataclass
class Masked:
    """Masked-layout grouped GEMM (decode MoE): A [E, cap, K] token slots of
    which the first counts[e] rows are real, B [E, N, K]."""
    name: str
    A: np.ndarray                 # [E, cap, K], rows past the count are zero
    B: np.ndarray                 # [E, N, K]
    counts: np.ndarray            # [E] int32
    out: str = "bf16"


@dataclass
class Workload:
    name: str
    gemms: list = field(default_factory=list)


def tiny(seed: int = 0) -> Workload:
    """Tiny reference GEMM: A [128,512] N(0,1) with 1% outliers x100,
    B [256,512] N(0,0.02); bf16 output."""
    rng = np.random.default_rng(seed)
    A = bf16_normal(rng, (128, 512), 1.0, 0.01, 100.0)
    B = bf16_normal(rng, (256, 512), 0.02)
    return Workload("tiny_128x256x512", [Dense("tiny", A, B)])


def prefill_pair(seed: int = 1, M: int = 4096, H: int = 7168, F: int = 18432) -> Workload:
    """Prefill projection pair: A1 [M,H] N(0,1), 0.1% outliers x50; B1 [F,H]
    N(0,0.02); A2 [M,F] likewise; B2 [H,F]; bf16 outputs."""
    rng = np.random.default_rng(seed)
    A1 = bf16_normal(rng, (M, H), 1.0, 0.001, 50.0)
    B1 = bf16_normal(rng, (F, H), 0.02)
    A2 = bf16_normal(rng, (M, F), 1.0, 0.001, 50.0)
    B2 = bf16_normal(rng, (H, F), 0.02)
    return Workload(f"prefill_pair_{M}x{F}x{H}",
                    [Dense("up", A1, B1), Dense("down", A2, B2)])


def decode(seed: int = 2, Ms=(16, 64, 128, 256), H: int = 7168, F: int = 4096,
           K2: int = 2048, N2: int = 7168) -> Workload:
    """Decode-size GEMMs: for each M, A [M,H] and A' [M,K2] N(0,1); then the
    shared weights B1 [F,H] and B2 [N2,K2] N(0,0.02); bf16 outputs."""
    rng = np.random.default_rng(seed)
    acts = []
    for M in Ms:
        acts.append((M, bf16_normal(rng, (M, H)), bf16_normal(rng, (M, K2))))
    B1 = bf16_normal(rng, (F, H), 0.02)
    B2 = bf16_normal(rng, (N2, K2), 0.02)
    gemms = []
    for M, A, A2 in acts:
        gemms.append(Dense(f"decode_m{M}_a", A, B1))
        gemms.append(Dense(f"decode_m{M}_b", A2, B2))
    return Workload("decode", gemms)


def moe_grouped(seed: int = 3, E: int = 32, tokens: int = 32768, N: int = 4096,
                K: int = 7168) -> Workload:
    """Grouped MoE GEMM: expert shares ~ Dirichlet(1), counts ~ multinomial;
    A [tokens,K] N(0,1) laid out per expert with each group padded to 128
    rows; B_e [N,K] N(0,0.02) for e = 0..E-1; bf16 output."""
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(E))
    counts = rng.multinomial(tokens, p)
    A_real = bf16_normal(rng, (tokens, K))
    B = np.empty((E, N, K), np.uint16)
    for e in range(E):
        B[e] = bf16_normal(rng, (N, K), 0.02)
    return _grouped_layout(f"moe_{E}x{tokens}x{N}x{K}", A_real, B, counts)


def _grouped_layout(name, A_real, B, counts) -> Workload:
    padded = [(int(c) + ROW_BLOCK - 1) // ROW_BLOCK * ROW_BLOCK for c in counts]
    M_pad = int(sum(padded))
    K = A_real.shape[1]
    A = np.zeros((M_pad, K), np.uint16)
    m_idx = np.full(M_pad, -1, np.int32)
    src = dst = 0
    for e, (c, pc) in enumerate(zip(counts, padded)):
        A[dst:dst + c] = A_real[src:src + c]
        m_idx[dst:dst + c] = e
        src += c
        dst += pc
    return Workload(name, [Grouped(name, A, B, m_idx, np.asarray(counts))])


def grouped_small(seed: int, counts, N: int, K: int) -> Workload:
    """A small grouped case with given token counts per expert (tests)."""
    rng = np.random.default_rng(seed)
    A_real = bf16_normal(rng, (int(sum(counts)), K))
    B = np.stack([bf16_normal(rng, (N, K), 0.02) for _ in counts])
    return _grouped_layout("grouped_small", A_real, B, np.asarray(counts))


def wgrad(seed: int = 4, T: int = 8192, N: int = 7168, K: int = 2048) -> Workload:
    """Weight gradient: dY [T,N] and X [T,K] N(0,1), 0.1% outliers x50 each;
    dW = dY^T X in fp32."""
    rng = np.random.default_rng(seed)
    dY = bf16_normal(rng, (T, N), 1.0, 0.001, 50.0)
    X = bf16_normal(rng, (T, K), 1.0, 0.001, 50.0)
    return Workload(f"wgrad_{N}x{K}x{T}", [Wgrad("wgrad", dY, X)])


def dgrad(seed: int = 5, T: int = 4096, N: int = 18432, K: int = 7168) -> Workload:
    """Data gradient through the prefill up-projection: dY [T,N] N(0,1) with
    0.1% outliers x50, W [N,K] N(0,0.02); dX = dY W in bf16."""
    rng = np.random.default_rng(seed)
    dY = bf16_normal(rng, (T, N), 1.0, 0.001, 50.0)
    W = bf16_normal(rng, (N, K), 0.02)
    return Workload(f"dgrad_{T}x{K}x{N}", [Dgrad("dgrad", dY, W)])


def masked_small(seed, counts, cap, N, K):
    """Small masked-layout case for parity tests: slots [E, cap, K] N(0,1)
    (rows past each count zero), B [E, N, K] N(0,0.02)."""
    rng = np.random.default_rng(seed)
    counts = np.asarray(counts, np.int32)
    E = len(counts)
    A = np.zeros((E, cap, K), np.uint16)
    for e in range(E):
        if counts[e]:
            A[e, :counts[e]] = bf16_normal(rng, (int(counts[e]), K), 1.0, 0.001, 50.0)
    B = np.stack([bf16_normal(rng, (N, K), 0.02) for _ in range(E)])
    return Workload(f"masked_{E}x{cap}x{N}x{K}", [Masked("masked", A, B, counts)])


def moe_decode(seed: int = 6, E: int = 32, cap: int = 256, tokens: int = 2048, N: int = 4096, K: int = 7168) -> Workload:
    """Decode-time MoE in the masked layout: `tokens` routed tokens spread over
    E experts by a Dirichlet(1) share and a multinomial draw, each expert's
    count capped at its slot size `cap`; slots [E, cap, K] N(0,1) with 0.1%
    outliers x50 (rows past the count zero), expert weights [E, N, K] N(0,0.02)."""
    rng = np.random.default_rng(seed)
    share = rng.dirichlet(np.ones(E))
    counts = np.minimum(rng.multinomial(tokens, share), cap).astype(np.int32)
    A = np.zeros((E, cap, K), np.uint16)
    for e in range(E):
        if counts[e]:
            A[e, :counts[e]] = bf16_normal(rng, (int(counts[e]), K), 1.0, 0.001, 50.0)
    B = np.stack([bf16_normal(rng, (N, K), 0.02) for _ in range(E)])
    return Workload(f"moe_decode_{E}x{cap}x{N}x{K}", [Masked("masked", A, B, counts)])
