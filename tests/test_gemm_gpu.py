"""GPU parity of the block-scaled FP8 GEMM (dense, per-row B scales, grouped):
every output element within |C - C_ref| <= 2^-7 * sum|a_hat*b_hat| + 1e-6 of
the oracle's binary64 result, through the C ABI, on seeded inputs.  The
quantized operands come from the oracle, so the GEMM is tested on its own."""
import numpy as np
import pytest
import torch

import oracle
import fine_grained_fp8_weight_b300 as fg
from fine_grained_fp8_weight_b300 import workloads as wl
from tests.gpu_util import DEV, assert_within_bound, bf16_out_to_f64, dev_bf16, ensure_built, report_margin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _d(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _sample_rows(M, n, seed):
    return np.sort(np.random.default_rng(seed).choice(M, size=min(n, M), replace=False))


def _rows_per_block(M, n, seed):
    """n random rows of every 128-row block (all rows of a shorter last block)."""
    rng = np.random.default_rng(seed)
    return np.concatenate([np.sort(rng.choice(np.arange(m0, min(m0 + 128, M)), size=min(n, M - m0), replace=False))
                           for m0 in range(0, M, 128)])


def _run_dense(Abits, Bbits, out_dtype, rows=None, bkind=0, workspace=None):
    qa, sa = oracle.quant_act_1x128(Abits)
    if bkind == 0:
        qb, sb = oracle.quant_w_128x128(Bbits)
    else:
        qb, sb = oracle.quant_act_1x128(Bbits)          # per-row (1x128) B scales
    C = fg.fp8_gemm_blockscaled(_d(qa), _d(sa), _d(qb), _d(sb), bkind=bkind, out_dtype=out_dtype,
                                workspace=workspace, check=True)
    torch.cuda.synchronize()
    Cg = bf16_out_to_f64(C) if out_dtype == torch.bfloat16 else C.cpu().numpy().astype(np.float64)
    Cr, S = oracle.gemm_blockscaled(qa, sa, qb, sb, bkind, rows=rows)
    if rows is not None:
        Cg = Cg[rows]
    return Cg, Cr, S


def test_tiny_workload():
    g = wl.tiny().gemms[0]
    Cg, Cr, S = _run_dense(g.A, g.B, torch.bfloat16)
    mx, mean = assert_within_bound(Cg, Cr, S, "tiny")
    assert mx < 2.0 ** -7
    report_margin("C1 tiny 128x256x512", (mx, mean), Cg.size)


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (1, 16, 128), (77, 144, 256), (300, 400, 512),
                                   (256, 256, 1024), (129, 272, 384), (1000, 48, 128)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_dense_shapes(M, N, K, out):
    rng = np.random.default_rng(M * 31 + N * 7 + K)
    A = wl.bf16_normal(rng, (M, K), 1.0, 0.01, 100.0)
    B = wl.bf16_normal(rng, (N, K), 0.02)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    Cg, Cr, S = _run_dense(A, B, dt)
    assert_within_bound(Cg, Cr, S, f"{M}x{N}x{K}")


# Larger M: several M blocks per N block, a ragged last M block, odd and even
# K-group counts, and N past the last tile column.
@pytest.mark.parametrize("M,N,K", [(256, 128, 128), (257, 144, 384), (600, 400, 512), (1024, 16, 256),
                                   (768, 256, 640)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_dense_large_m(M, N, K, out):
    rng = np.random.default_rng(M * 13 + N * 5 + K)
    A = wl.bf16_normal(rng, (M, K), 1.0, 0.01, 100.0)
    B = wl.bf16_normal(rng, (N, K), 0.02)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    Cg, Cr, S = _run_dense(A, B, dt)
    assert_within_bound(Cg, Cr, S, f"{M}x{N}x{K}")


# Last-wave split: tiles left over after the whole waves are cut along K and
# the last piece of each adds the FP32 partials.  Cases: no whole wave (every
# tile split), one and two whole waves, both tile widths, both B-scale kinds,
# both output types.  The same GEMM with the least workspace runs whole tiles
# only; both schedules must meet the bound.  The oracle takes sampled rows of
# every 128-row block (two, one on the largest shapes), so every output tile
# is checked.
_split_cases = {}


def _split_case(M, N, K, bkind):
    """Quantized operands, sampled rows and the oracle's result, once per shape
    (the oracle is the slow part; both output types and schedules reuse it)."""
    key = (M, N, K, bkind)
    if key not in _split_cases:
        rng = np.random.default_rng(M * 3 + N + K + bkind)
        A = wl.bf16_normal(rng, (M, K), 1.0, 0.01, 100.0)
        B = wl.bf16_normal(rng, (N, K), 0.02)
        qa, sa = oracle.quant_act_1x128(A)
        qb, sb = oracle.quant_w_128x128(B) if bkind == 0 else oracle.quant_act_1x128(B)
        rows = _rows_per_block(M, 1 if M * K > 4_000_000 else 2, M + K)
        Cr, S = oracle.gemm_blockscaled(qa, sa, qb, sb, bkind, rows=rows)
        _split_cases[key] = ([_d(t) for t in (qa, sa, qb, sb)], rows, Cr, S)
    return _split_cases[key]


@pytest.mark.parametrize("M,N,K,bkind,bn", [(384, 3072, 1792, 0, 128), (1280, 4096, 2048, 0, 128),
                                            (2560, 4096, 4096, 0, 256), (1280, 4096, 2048, 1, 128),
                                            (2560, 4096, 4096, 1, 256)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_last_wave_split(M, N, K, bkind, bn, out):
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    sch = fg.fgf8_testing_gemm_schedule(M, N, K, bkind, num_sms=sm)
    assert sch["pair"] == 0 and sch["bn"] == bn and sch["tail_s"] > 1, sch
    ops, rows, Cr, S = _split_case(M, N, K, bkind)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    ws_min = torch.zeros(fg.lib().fgf8_gemm_workspace_min_bytes(M, N, K, 1), dtype=torch.uint8, device=DEV)
    assert fg.fgf8_testing_gemm_schedule(M, N, K, bkind, ws_bytes=ws_min.numel(), num_sms=sm)["tail_s"] == 1
    for label, ws in (("split", None), ("whole tiles", ws_min)):
        C = fg.fp8_gemm_blockscaled(*ops, bkind=bkind, out_dtype=dt, workspace=ws)
        torch.cuda.synchronize()
        Cg = bf16_out_to_f64(C) if dt == torch.bfloat16 else C.cpu().numpy().astype(np.float64)
        assert_within_bound(Cg[rows], Cr, S, f"{label} {M}x{N}x{K}")


# CTA-pair kernel (256 x 128 tiles on two SMs whose tensor cores run as one;
# off by default, switched on by the test hook): M blocks go in pairs, so the
# last pair's second CTA may hold a few rows past M or none at all; N may end
# inside a tile or be narrower than one; one 128-row block past the first
# (M = 129) with many weight tiles; odd K-group counts (the even and odd
# promotion warps get different numbers of groups).
@pytest.fixture
def pair_on():
    assert fg.lib().fgf8_testing_set_pair(1) == 0
    try:
        yield
    finally:
        assert fg.lib().fgf8_testing_set_pair(0) == 0


@pytest.mark.parametrize("M,N,K", [(512, 256, 128), (384, 272, 512), (129, 18432, 256), (640, 48, 384),
                                   (1000, 1040, 1152), (2048, 4096, 2048)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_pair_shapes(M, N, K, out, pair_on):
    assert fg.fgf8_testing_gemm_schedule(M, N, K)["pair"] == 1
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A = wl.bf16_normal(rng, (M, K), 1.0, 0.01, 100.0)
    B = wl.bf16_normal(rng, (N, K), 0.02)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    rows = _rows_per_block(M, 4, M + 1) if M * N * K > 2 ** 31 else None
    Cg, Cr, S = _run_dense(A, B, dt, rows=rows)
    assert_within_bound(Cg, Cr, S, f"pair {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(512, 2048, 2048), (1280, 4096, 2048), (768, 4096, 2048)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_pair_last_wave_split(M, N, K, out, pair_on):
    # the planner with the pairs this device runs at once: some tiles are cut
    # into K pieces; the same GEMM with the least workspace runs whole tiles
    sm = 2 * fg.lib().fgf8_testing_pair_clusters()
    sch = fg.fgf8_testing_gemm_schedule(M, N, K, 0, num_sms=sm)
    assert sch["pair"] == 1 and sch["tail_s"] > 1, sch
    ops, rows, Cr, S = _split_case(M, N, K, 0)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    ws_min = torch.zeros(fg.lib().fgf8_gemm_workspace_min_bytes(M, N, K, 1), dtype=torch.uint8, device=DEV)
    for label, ws in (("split", None), ("whole tiles", ws_min)):
        C = fg.fp8_gemm_blockscaled(*ops, out_dtype=dt, workspace=ws)
        torch.cuda.synchronize()
        Cg = bf16_out_to_f64(C) if dt == torch.bfloat16 else C.cpu().numpy().astype(np.float64)
        assert_within_bound(Cg[rows], Cr, S, f"pair {label} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,out", [(2048, 4096, 4096, "bf16"), (1280, 4096, 2048, "fp32"),
                                       (3072, 1792, 2048, "bf16")])
def test_pair_repeated_launches_bitwise_identical(M, N, K, out, pair_on):
    _repeat_check(M, N, K, 0, out)


def test_pair_output_row_stride_and_untouched_padding(pair_on):
    # rows past M and columns past N of a larger output buffer stay as they were
    rng = np.random.default_rng(16)
    A = wl.bf16_normal(rng, (300, 256))
    B = wl.bf16_normal(rng, (272, 256), 0.02)
    qa, sa = oracle.quant_act_1x128(A)
    qb, sb = oracle.quant_w_128x128(B)
    big = torch.full((512, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = big[:300, :272]
    assert fg.fgf8_testing_gemm_schedule(300, 272, 256)["pair"] == 1
    fg.fp8_gemm_blockscaled(_d(qa), _d(sa), _d(qb), _d(sb), out=out)
    torch.cuda.synchronize()
    assert torch.isnan(big[:, 272:]).all() and torch.isnan(big[300:]).all(), "elements past M or N were written"
    Cr, S = oracle.gemm_blockscaled(qa, sa, qb, sb)
    assert_within_bound(bf16_out_to_f64(out), Cr, S)


# M <= 128 takes the small-M path (weights on the MMA's M side, the K groups
# of each weight tile split over the CTAs of a thread-block cluster, which add
# their partials in split order through distributed shared memory): every
# token width 16..128, a ragged last weight tile, 1 to 8 splits, both output
# types; 129..256 tokens (large tiles with the last-wave split) as well.
@pytest.mark.parametrize("M,N,K", [(16, 4096, 7168), (5, 144, 2048), (33, 512, 1024), (64, 7168, 2048),
                                   (100, 400, 640), (200, 1024, 3072), (256, 2048, 512), (250, 16, 128)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_small_m(M, N, K, out):
    rng = np.random.default_rng(M * 17 + N + K)
    A = wl.bf16_normal(rng, (M, K), 1.0, 0.01, 100.0)
    B = wl.bf16_normal(rng, (N, K), 0.02)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    rows = _sample_rows(M, 40, M) if M * N * K > 2 ** 31 else None
    Cg, Cr, S = _run_dense(A, B, dt, rows=rows)
    assert_within_bound(Cg, Cr, S, f"small {M}x{N}x{K}")


def test_small_m_repeated_calls_same_workspace():
    # the same split on every call: bit-identical outputs
    rng = np.random.default_rng(77)
    A = wl.bf16_normal(rng, (48, 1024))
    B = wl.bf16_normal(rng, (1024, 1024), 0.02)
    qa, sa = oracle.quant_act_1x128(A)
    qb, sb = oracle.quant_w_128x128(B)
    ws = torch.zeros(fg.lib().fgf8_gemm_workspace_bytes(48, 1024, 1024, 1) + 4096, dtype=torch.uint8, device=DEV)
    outs = [fg.fp8_gemm_blockscaled(_d(qa), _d(sa), _d(qb), _d(sb), workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    Cr, S = oracle.gemm_blockscaled(qa, sa, qb, sb)
    for o in outs:
        assert_within_bound(bf16_out_to_f64(o), Cr, S)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2]), "split order must be deterministic"
    assert fg.fgf8_read_status(ws) == (0, 0)


@pytest.fixture
def small_splits():
    yield lambda s: fg.lib().fgf8_testing_set_small_splits(s)
    fg.lib().fgf8_testing_set_small_splits(0)


# Every cluster size the small-M kernel can take (1..8 CTAs per weight tile,
# odd sizes included), forced through the testing hook: each within the bound
# against the oracle and bit-identical over repeated launches.
@pytest.mark.parametrize("M,N,K", [(48, 1024, 2048), (100, 400, 1024)])
def test_small_m_every_split_count(M, N, K, small_splits):
    rng = np.random.default_rng(M + N + K)
    A = wl.bf16_normal(rng, (M, K), 1.0, 0.01, 100.0)
    B = wl.bf16_normal(rng, (N, K), 0.02)
    qa, sa = oracle.quant_act_1x128(A)
    qb, sb = oracle.quant_w_128x128(B)
    Cr, S = oracle.gemm_blockscaled(qa, sa, qb, sb)
    ops = [_d(qa), _d(sa), _d(qb), _d(sb)]
    for splits in range(1, 9):
        assert small_splits(splits) == 0
        assert fg.fgf8_testing_gemm_schedule(M, N, K)["tail_s"] == min(splits, K // 128)
        outs = [fg.fp8_gemm_blockscaled(*ops, check=True) for _ in range(2)]
        assert torch.equal(outs[0], outs[1]), f"{splits} splits: repeated launches differ"
        assert_within_bound(bf16_out_to_f64(outs[0]), Cr, S, f"{M}x{N}x{K} with {splits} splits")
    assert small_splits(9) == 1                       # FGF8_ERR_INVALID_ARG


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (200, 256, 512), (256, 144, 384), (512, 256, 1024)])
def test_row_scaled_b(M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = wl.bf16_normal(rng, (M, K), 1.0, 0.001, 50.0)
    B = wl.bf16_normal(rng, (N, K), 1.0, 0.001, 50.0)
    Cg, Cr, S = _run_dense(A, B, torch.float32, bkind=1)
    assert_within_bound(Cg, Cr, S, "row-scaled")


def test_fp32_fp32_accumulation_is_tight():
    # with FP32 output the error comes only from the tensor-core partial sums
    # and the FP32 promotion: far below the stated bound
    rng = np.random.default_rng(3)
    A = wl.bf16_normal(rng, (256, 2048), 1.0, 0.01, 100.0)
    B = wl.bf16_normal(rng, (256, 2048), 0.02)
    Cg, Cr, S = _run_dense(A, B, torch.float32)
    mx, _ = assert_within_bound(Cg, Cr, S)
    assert mx < 2.0 ** -16


def test_zero_operand_gives_zero():
    A = np.zeros((128, 256), np.uint16)
    B = wl.bf16_normal(np.random.default_rng(4), (128, 256), 0.02)
    Cg, Cr, S = _run_dense(A, B, torch.bfloat16)
    assert np.all(Cg == 0)


def test_output_row_stride_and_untouched_padding():
    rng = np.random.default_rng(6)
    A = wl.bf16_normal(rng, (130, 256))
    B = wl.bf16_normal(rng, (48, 256), 0.02)
    qa, sa = oracle.quant_act_1x128(A)
    qb, sb = oracle.quant_w_128x128(B)
    big = torch.full((130, 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = big[:, :48]
    fg.fp8_gemm_blockscaled(_d(qa), _d(sa), _d(qb), _d(sb), out=out)
    torch.cuda.synchronize()
    assert torch.isnan(big[:, 48:]).all(), "columns past N were written"
    Cr, S = oracle.gemm_blockscaled(qa, sa, qb, sb)
    assert_within_bound(bf16_out_to_f64(out), Cr, S)


def _grouped_case(seed, counts, N, K, rows=None):
    w = wl.grouped_small(seed, counts, N, K).gemms[0]
    qa, sa = oracle.quant_act_1x128(w.A)
    E = w.B.shape[0]
    qbs, sbs = zip(*[oracle.quant_w_128x128(w.B[e]) for e in range(E)])
    qb = np.stack(qbs)
    sb = np.stack(sbs)
    out = torch.full((w.A.shape[0], N), float("nan"), dtype=torch.bfloat16, device=DEV)
    fg.fp8_grouped_gemm_blockscaled(_d(qa), _d(sa), _d(qb), _d(sb), _d(w.m_indices), out=out, check=True)
    torch.cuda.synchronize()
    Cr, S = oracle.grouped_gemm_blockscaled(qa, sa, qb, sb, w.m_indices, rows=rows)
    Cg = bf16_out_to_f64(out)
    if rows is not None:
        Cg = Cg[rows]
    return w, Cg, Cr, S


@pytest.mark.parametrize("counts", [[130, 0, 70, 256], [1], [0, 0, 300], [128, 128]])
def test_grouped_small(counts):
    w, Cg, Cr, S = _grouped_case(sum(counts) + len(counts), counts, 144, 256)
    real = w.m_indices >= 0
    assert_within_bound(Cg[real], Cr[real], S[real], "grouped")
    assert np.all(np.isnan(Cg[~real])), "padding rows were written"


# Grouped contiguous layout at full size (32 experts, 32 768 tokens padded to
# 34 944 rows, N = 4096, K = 7168): both operands quantized on the GPU by the
# package's quantizers and checked bit for bit against the oracle's codes and
# scales (every weight byte, every activation row), then the grouped GEMM
# against the oracle's binary64 result on rows of every expert -- its first
# and last real rows, two rows between, and the first row after each padding
# boundary -- with every padding row left unwritten.  At this size each CTA
# walks ~15 tiles of the m-outer schedule, so expert changes inside one CTA's
# walk and padding blocks between them are covered.
def test_full_size_moe_grouped():
    w = wl.moe_grouped().gemms[0]
    E, N, K = w.B.shape
    Mp = w.A.shape[0]
    A = dev_bf16(w.A)
    qa, sa, _, _ = fg.fp8_quant_act_1x128(A)
    del A
    Bd = wl.bf16_bits_to_torch(w.B).to(DEV)
    qb, sb = fg.fp8_quant_w_128x128_grouped(Bd)
    del Bd
    mi = torch.from_numpy(w.m_indices).to(DEV)
    out = torch.full((Mp, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    fg.fp8_grouped_gemm_blockscaled(qa, sa, qb, sb, mi, out=out, check=True)
    torch.cuda.synchronize()
    rqa, rsa = oracle.quant_act_1x128(w.A)
    assert np.array_equal(qa.cpu().numpy(), rqa), "activation codes differ from the oracle"
    assert np.array_equal(sa.cpu().numpy()[:, :Mp].view(np.uint32), rsa[:, :Mp].view(np.uint32))
    qbh, sbh = qb.cpu().numpy(), sb.cpu().numpy()
    rqb = np.empty_like(qbh)
    rsb = np.empty_like(sbh)
    for e in range(E):
        rqb[e], rsb[e] = oracle.quant_w_128x128(w.B[e])
        assert np.array_equal(qbh[e], rqb[e]), f"weight codes of expert {e} differ from the oracle"
        assert np.array_equal(sbh[e, :, :N // 128].view(np.uint32), rsb[e, :, :N // 128].view(np.uint32))
    starts = np.concatenate([[0], np.cumsum((w.counts + 127) // 128 * 128)[:-1]])
    rng = np.random.default_rng(31)
    rows = []
    for e, (r0, c) in enumerate(zip(starts, w.counts)):
        if c == 0:
            continue
        rows += [r0, r0 + c - 1] + [int(r0 + x) for x in rng.integers(0, c, 2)]
    rows = np.unique(np.array(rows, np.int64))
    Cr, S = oracle.grouped_gemm_blockscaled(rqa, rsa, rqb, rsb, w.m_indices, rows=rows)
    report_margin("C4 MoE grouped (sampled rows)",
                  assert_within_bound(bf16_out_to_f64(out[torch.from_numpy(rows).to(DEV)]), Cr, S, "moe grouped"),
                  Cr.size)
    pad = torch.from_numpy(w.m_indices < 0).to(DEV)
    assert bool(torch.isnan(out[pad]).all()), "padding rows were written"


# --- full-size workloads, sampled rows ---


def test_full_size_prefill_pair_sampled():
    for g, seed in zip(wl.prefill_pair().gemms, (11, 12)):
        rows = _sample_rows(g.A.shape[0], 3, seed)
        Cg, Cr, S = _run_dense(g.A, g.B, torch.bfloat16, rows=rows)
        report_margin(f"C2 {g.name} (sampled rows)", assert_within_bound(Cg, Cr, S, g.name), Cg.size)


def test_full_size_decode():
    for g in wl.decode().gemms:
        rows = _sample_rows(g.A.shape[0], 8, 13)
        Cg, Cr, S = _run_dense(g.A, g.B, torch.bfloat16, rows=rows)
        report_margin(f"C3 {g.name} (sampled rows)", assert_within_bound(Cg, Cr, S, g.name), Cg.size)


def test_full_size_wgrad_sampled():
    g = wl.wgrad().gemms[0]
    dYt, sdY = oracle.quant_act_128x1(g.dY)       # [N, T], [T/128, N]
    Xt, sX = oracle.quant_act_128x1(g.X)          # [K, T], [T/128, K]
    C = fg.fp8_gemm_blockscaled(_d(dYt), _d(sdY), _d(Xt), _d(sX), bkind=fg.BSCALE_ROW1x128,
                                out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = _sample_rows(dYt.shape[0], 3, 14)
    Cr, S = oracle.gemm_blockscaled(dYt, sdY, Xt, sX, 1, rows=rows)
    report_margin("C5 wgrad (sampled rows)",
                  assert_within_bound(C.cpu().numpy().astype(np.float64)[rows], Cr, S, "wgrad"), Cr.size)


# Every path adds in a fixed order (small-M adds its K splits in split order
# too): repeated launches on the same operands must agree bit for bit over the
# whole output.  A race between the tensor-memory loads, the scale ring and its
# TMA refills, or the output stores shows up here as a differing element long
# before a sampled comparison with the oracle sees it.  The shapes give every
# CTA several tiles (the scale ring then runs into the next tile), on both
# tile widths, both B-scale kinds and both output types, plus small M.
@pytest.mark.parametrize("M,N,K,bkind,out", [(2048, 4096, 4096, 0, "bf16"), (4096, 2048, 4096, 1, "fp32"),
                                             (4096, 2048, 4096, 1, "bf16"), (4096, 4096, 2048, 0, "fp32"),
                                             (3072, 1792, 2048, 1, "fp32"), (3072, 1792, 2048, 0, "bf16"),
                                             (64, 7168, 4096, 0, "bf16"), (200, 2048, 4096, 0, "fp32"),
                                             (2560, 4096, 4096, 0, "bf16"), (1280, 4096, 2048, 1, "fp32")])
def test_repeated_launches_bitwise_identical(M, N, K, bkind, out):
    _repeat_check(M, N, K, bkind, out)


def _repeat_check(M, N, K, bkind, out):
    g = torch.Generator(device="cpu").manual_seed(M + N + K + bkind)
    qa = torch.randint(0, 256, (M, K), dtype=torch.uint8, generator=g)
    qa[(qa & 0x7F) == 0x7F] = 0x3C                  # no NaN codes
    qb = torch.randint(0, 256, (N, K), dtype=torch.uint8, generator=g)
    qb[(qb & 0x7F) == 0x7F] = 0x3C
    sa = torch.rand((K // 128, M), generator=g) + 0.5
    if bkind == 0:
        sb = torch.rand((K // 128, ((N + 127) // 128 + 3) // 4 * 4), generator=g) + 0.5   # row stride % 4 == 0
    else:
        sb = torch.rand((K // 128, N), generator=g) + 0.5
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    args = [t.to(DEV) for t in (qa, sa, qb, sb)]
    outs = [fg.fp8_gemm_blockscaled(*args, bkind=bkind, out_dtype=dt) for _ in range(6)]
    torch.cuda.synchronize()
    for i, o in enumerate(outs[1:], 1):
        bad = (o.view(torch.int16 if dt == torch.bfloat16 else torch.int32)
               != outs[0].view(torch.int16 if dt == torch.bfloat16 else torch.int32))
        assert not bool(bad.any()), f"launch {i} differs at {bad.nonzero()[:4].tolist()}"


# Multicast clusters (off by default, switched on by the test hook): two CTAs
# on vertically adjacent 128 x 256 tiles, each loading its own A panel and half
# of the B panel they share, multicast into both.  Odd 128-row block counts
# leave the last cluster's second CTA past M (M = 384, 640, 129, 300, 1408,
# 3200); N narrower than the shared half (48) or ending inside either half.
@pytest.fixture
def multicast_on():
    assert fg.lib().fgf8_testing_set_pair(2) == 0
    try:
        yield
    finally:
        assert fg.lib().fgf8_testing_set_pair(0) == 0


@pytest.mark.parametrize("M,N,K", [(512, 256, 128), (384, 272, 512), (129, 18432, 256), (640, 48, 384),
                                   (1000, 1040, 1152), (2048, 4096, 2048)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_multicast_shapes(M, N, K, out, multicast_on):
    assert fg.fgf8_testing_gemm_schedule(M, N, K)["pair"] == 2
    rng = np.random.default_rng(M * 5 + N * 3 + K)
    A = wl.bf16_normal(rng, (M, K), 1.0, 0.01, 100.0)
    B = wl.bf16_normal(rng, (N, K), 0.02)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    rows = _rows_per_block(M, 4, M + 1) if M * N * K > 2 ** 31 else None
    Cg, Cr, S = _run_dense(A, B, dt, rows=rows)
    assert_within_bound(Cg, Cr, S, f"multicast {M}x{N}x{K}")


# Whole tiles (the least workspace: no K split) on multicast clusters compute
# every element with the same MMAs and promotion as single CTAs with 256-column
# tiles: equal bit for bit.
@pytest.mark.parametrize("M,N,K", [(1408, 2304, 1024), (3200, 1024, 1024), (4096, 4096, 1024), (2048, 4096, 2048)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_multicast_whole_tiles_equal_single_cta(M, N, K, out):
    g = torch.Generator(device="cpu").manual_seed(M + 3 * N + K)
    qa = torch.randint(0, 256, (M, K), dtype=torch.uint8, generator=g)
    qa[(qa & 0x7F) == 0x7F] = 0x3C                  # no NaN codes
    qb = torch.randint(0, 256, (N, K), dtype=torch.uint8, generator=g)
    qb[(qb & 0x7F) == 0x7F] = 0x3C
    sa = torch.rand((K // 128, M), generator=g) + 0.5
    sb = torch.rand((K // 128, ((N + 127) // 128 + 3) // 4 * 4), generator=g) + 0.5
    args = [t.to(DEV) for t in (qa, sa, qb, sb)]
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    ws = torch.zeros(fg.lib().fgf8_gemm_workspace_min_bytes(M, N, K, 1), dtype=torch.uint8, device=DEV)
    single = fg.fgf8_testing_gemm_schedule(M, N, K, ws_bytes=ws.numel())
    assert single["bn"] == 256 and single["tail_s"] == 1 and single["pair"] == 0, single
    ref = fg.fp8_gemm_blockscaled(*args, out_dtype=dt, workspace=ws, check=True)
    assert fg.lib().fgf8_testing_set_pair(2) == 0
    try:
        assert fg.fgf8_testing_gemm_schedule(M, N, K, ws_bytes=ws.numel())["pair"] == 2
        mc = fg.fp8_gemm_blockscaled(*args, out_dtype=dt, workspace=ws, check=True)
        torch.cuda.synchronize()
    finally:
        assert fg.lib().fgf8_testing_set_pair(0) == 0
    iv = torch.int16 if dt == torch.bfloat16 else torch.int32
    bad = mc.view(iv) != ref.view(iv)
    assert not bool(bad.any()), f"multicast differs from single CTAs at {bad.nonzero()[:4].tolist()}"


@pytest.mark.parametrize("M,N,K", [(1280, 4096, 2048), (2560, 4096, 4096), (512, 2048, 2048), (3072, 1792, 2048)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_multicast_last_wave_split(M, N, K, out, multicast_on):
    # the planner with the clusters this device runs at once: some cluster
    # tiles are cut into K pieces; with the least workspace, whole tiles
    sm = 2 * fg.lib().fgf8_testing_multicast_clusters()
    sch = fg.fgf8_testing_gemm_schedule(M, N, K, 0, num_sms=sm)
    assert sch["pair"] == 2 and sch["tail_s"] > 1, sch
    ops, rows, Cr, S = _split_case(M, N, K, 0)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    ws_min = torch.zeros(fg.lib().fgf8_gemm_workspace_min_bytes(M, N, K, 1), dtype=torch.uint8, device=DEV)
    for label, ws in (("split", None), ("whole tiles", ws_min)):
        C = fg.fp8_gemm_blockscaled(*ops, out_dtype=dt, workspace=ws, check=True)
        torch.cuda.synchronize()
        Cg = bf16_out_to_f64(C) if dt == torch.bfloat16 else C.cpu().numpy().astype(np.float64)
        assert_within_bound(Cg[rows], Cr, S, f"multicast {label} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,out", [(2048, 4096, 4096, "bf16"), (1280, 4096, 2048, "fp32"),
                                       (3072, 1792, 2048, "bf16")])
def test_multicast_repeated_launches_bitwise_identical(M, N, K, out, multicast_on):
    _repeat_check(M, N, K, 0, out)


def test_multicast_output_row_stride_and_untouched_padding(multicast_on):
    # rows past M and columns past N of a larger output buffer stay as they
    # were; 3 row blocks: the second CTA of the last cluster is past M
    rng = np.random.default_rng(17)
    A = wl.bf16_normal(rng, (300, 256))
    B = wl.bf16_normal(rng, (272, 256), 0.02)
    qa, sa = oracle.quant_act_1x128(A)
    qb, sb = oracle.quant_w_128x128(B)
    big = torch.full((512, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = big[:300, :272]
    assert fg.fgf8_testing_gemm_schedule(300, 272, 256)["pair"] == 2
    fg.fp8_gemm_blockscaled(_d(qa), _d(sa), _d(qb), _d(sb), out=out, check=True)
    torch.cuda.synchronize()
    assert torch.isnan(big[:, 272:]).all() and torch.isnan(big[300:]).all(), "elements past M or N were written"
    Cr, S = oracle.gemm_blockscaled(qa, sa, qb, sb)
    assert_within_bound(bf16_out_to_f64(out), Cr, S)


def test_full_size_prefill_multicast_sampled(multicast_on):
    # one row of every 128-row block: both CTAs of every cluster row
    for g, seed in zip(wl.prefill_pair().gemms, (21, 22)):
        (M, K), N = g.A.shape, g.B.shape[0]
        assert fg.fgf8_testing_gemm_schedule(M, N, K)["pair"] == 2
        rows = _rows_per_block(M, 1, seed)
        Cg, Cr, S = _run_dense(g.A, g.B, torch.bfloat16, rows=rows)
        report_margin(f"C2 {g.name} multicast (sampled rows)", assert_within_bound(Cg, Cr, S, g.name), Cg.size)


# The grouped layout repeated: m-outer tile walk with several tiles per CTA,
# expert changes inside a CTA's walk, padding blocks between experts and an
# empty expert; the whole output (padding rows left NaN) must match bit for bit.
@pytest.mark.parametrize("counts,N,K", [([700, 300, 0, 1000, 130, 2000, 50, 640], 4096, 1024),
                                        ([129, 1, 255, 3000, 77], 2048, 2048)])
def test_grouped_repeated_launches_bitwise_identical(counts, N, K):
    g = torch.Generator(device="cpu").manual_seed(sum(counts) + N + K)
    E = len(counts)
    padded = [(c + 127) // 128 * 128 for c in counts]
    Mp = sum(padded)
    mi = np.full(Mp, -1, np.int32)
    r = 0
    for e, (c, pc) in enumerate(zip(counts, padded)):
        mi[r:r + c] = e
        r += pc
    qa = torch.randint(0, 256, (Mp, K), dtype=torch.uint8, generator=g)
    qa[(qa & 0x7F) == 0x7F] = 0x3C
    qb = torch.randint(0, 256, (E, N, K), dtype=torch.uint8, generator=g)
    qb[(qb & 0x7F) == 0x7F] = 0x3C
    sa = torch.rand((K // 128, Mp), generator=g) + 0.5
    sb = torch.rand((E, K // 128, ((N + 127) // 128 + 3) // 4 * 4), generator=g) + 0.5
    args = [t.to(DEV) for t in (qa, sa, qb, sb)] + [torch.from_numpy(mi).to(DEV)]
    outs = []
    for _ in range(5):
        o = torch.full((Mp, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        fg.fp8_grouped_gemm_blockscaled(*args, out=o)
        outs.append(o)
    torch.cuda.synchronize()
    ref = outs[0].view(torch.int16)
    for i, o in enumerate(outs[1:], 1):
        bad = o.view(torch.int16) != ref
        assert not bool(bad.any()), f"launch {i} differs at {bad.nonzero()[:4].tolist()}"
    assert bool(torch.isnan(outs[0][torch.from_numpy(mi < 0).to(DEV)]).all())


# --- data gradient dX = dY * W: A = dY (1x128 along N), B = W^T (128x128) ---


@pytest.mark.parametrize("T,N,K", [(200, 384, 256), (256, 1024, 512), (1000, 256, 384)])
def test_dgrad_small(T, N, K):
    rng = np.random.default_rng(T + N * 3 + K)
    dY = wl.bf16_normal(rng, (T, N), 1.0, 0.001, 50.0)
    W = wl.bf16_normal(rng, (N, K), 0.02)
    qa, sa = oracle.quant_act_1x128(dY)
    qT, sT = fg.fp8_quant_w_128x128_t(dev_bf16(W))
    C = fg.fp8_gemm_blockscaled(_d(qa), _d(sa), qT, sT, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rqT, rsT = oracle.quant_w_128x128_t(W)
    Cr, S = oracle.gemm_blockscaled(qa, sa, rqT, rsT)
    assert_within_bound(C.cpu().numpy().astype(np.float64), Cr, S, "dgrad")


def test_full_size_dgrad_sampled():
    g = wl.dgrad().gemms[0]
    qa, sa = oracle.quant_act_1x128(g.dY)
    rqT, rsT = oracle.quant_w_128x128_t(g.W)
    C = fg.fp8_gemm_blockscaled(_d(qa), _d(sa), _d(rqT), _d(rsT))
    torch.cuda.synchronize()
    rows = _sample_rows(g.dY.shape[0], 3, 15)
    Cr, S = oracle.gemm_blockscaled(qa, sa, rqT, rsT, rows=rows)
    report_margin("dgrad 4096x7168x18432 (sampled rows)",
                  assert_within_bound(bf16_out_to_f64(C)[rows], Cr, S, "dgrad"), Cr.size)


# --- masked-layout grouped GEMM (decode MoE): per-expert token slots + counts ---


def _masked_inputs(w):
    g = w.gemms[0]
    E, cap, K = g.A.shape
    qa, sa = oracle.quant_act_1x128(g.A.reshape(E * cap, K))          # stacked slots
    qbs, sbs = zip(*[oracle.quant_w_128x128(g.B[e]) for e in range(E)])
    return g, qa.reshape(E, cap, K), sa, np.stack(qbs), np.stack(sbs)


def _run_masked(w, dt, rows=None, workspace=None):
    g, qa, sa, qb, sb = _masked_inputs(w)
    E, cap, K = qa.shape
    N = qb.shape[1]
    out = torch.full((E, cap, N), float("nan"), dtype=dt, device=DEV)
    counts = torch.from_numpy(g.counts).to(DEV)
    fg.fp8_masked_grouped_gemm_blockscaled(_d(qa), _d(sa), _d(qb), _d(sb), counts, out=out, workspace=workspace,
                                           check=True)
    torch.cuda.synchronize()
    Cr, S = oracle.masked_grouped_gemm_blockscaled(qa, sa, qb, sb, g.counts, rows_per_expert=rows)
    Cg = out.float().cpu().numpy().astype(np.float64) if dt == torch.float32 else bf16_out_to_f64(out.reshape(E * cap, N)).reshape(E, cap, N)
    return g, Cg, Cr, S


# E x weight tiles below the SM count -> K split over a cluster per (expert,
# weight tile); 40 x 4 tiles -> one split, direct stores; token widths 16, 64, 256.
# A slot batches as many K groups as its expert's count allows: counts of 80,
# 48, 112 in 256-row slots give 3, 4, 2 groups per batch at odd token offsets,
# and 11 or 9 K groups leave ragged last batches.
@pytest.mark.parametrize("counts,cap,N,K", [([64, 5, 0, 33], 64, 256, 512), ([16, 1], 16, 128, 256),
                                            ([256, 0, 200, 17, 1, 128, 255, 64], 256, 512, 1024),
                                            ([80, 48, 112, 96, 176, 16], 256, 256, 1408),
                                            ([128, 40, 72, 0, 100], 128, 384, 1152),
                                            ([int(c) for c in np.random.default_rng(5).integers(0, 33, 40)], 32, 512, 512)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_masked_grouped(counts, cap, N, K, out):
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    w = wl.masked_small(len(counts) * 7 + cap + N, counts, cap, N, K)
    g, Cg, Cr, S = _run_masked(w, dt)
    for e, c in enumerate(g.counts):
        if c:
            assert_within_bound(Cg[e, :c], Cr[e, :c], S[e, :c], f"masked expert {e}")
        assert np.all(np.isnan(Cg[e, c:])), f"rows past the count of expert {e} were written"


def test_masked_grouped_repeated_calls_same_workspace():
    w = wl.masked_small(3, [40, 0, 7, 64], 64, 256, 1024)
    g, qa, sa, qb, sb = _masked_inputs(w)
    ws = torch.zeros(fg.lib().fgf8_masked_gemm_workspace_bytes(4, 64, 256, 1024) + 4096, dtype=torch.uint8, device=DEV)
    counts = torch.from_numpy(g.counts).to(DEV)
    outs = [fg.fp8_masked_grouped_gemm_blockscaled(_d(qa), _d(sa), _d(qb), _d(sb), counts, workspace=ws)
            for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        for e, c in enumerate(g.counts):
            assert torch.equal(o[e, :c], outs[0][e, :c]), "split order must be deterministic"
    assert fg.fgf8_read_status(ws) == (0, 0)


def test_full_size_moe_decode_sampled():
    w = wl.moe_decode()
    g, Cg, Cr, S = _run_masked(w, torch.bfloat16, rows=[0, 1, 63, 130, 255])
    for e, c in enumerate(g.counts):
        for r in (0, 1, 63, 130, 255):
            if r < c:
                assert_within_bound(Cg[e, r:r + 1], Cr[e, r:r + 1], S[e, r:r + 1], f"moe decode expert {e} row {r}")


# --- token operand given as BF16, quantized inside the GEMM (decode M <= 256) ---


@pytest.mark.parametrize("M,N,K", [(16, 4096, 7168), (5, 144, 2048), (33, 512, 1024), (64, 7168, 2048),
                                   (64, 256, 128), (1, 16, 256), (128, 4096, 7168), (100, 512, 1024),
                                   (256, 7168, 2048), (200, 1024, 640)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_bf16a_equals_quantize_then_gemm(M, N, K, out):
    # same rule and arithmetic as the quantization kernel: up to 128 tokens
    # (where the two-step GEMM runs the small-M kernel too) the fused GEMM
    # must equal quantize + GEMM bit for bit; beyond, the two-step GEMM runs
    # large tiles (the same sum grouped differently), so both are held to the
    # bound against the oracle
    rng = np.random.default_rng(M * 11 + N + K)
    X = wl.bf16_normal(rng, (M, K), 1.0, 0.01, 100.0)
    W = wl.bf16_normal(rng, (N, K), 0.02)
    qb, sb = fg.fp8_quant_w_128x128(dev_bf16(W))
    x = dev_bf16(X)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    fused = fg.fp8_gemm_bf16a_blockscaled(x, qb, sb, out_dtype=dt, check=True)
    qa, sa, _, _ = fg.fp8_quant_act_1x128(x)
    twostep = fg.fp8_gemm_blockscaled(qa, sa, qb, sb, out_dtype=dt)
    torch.cuda.synchronize()
    iv = torch.int16 if dt == torch.bfloat16 else torch.int32
    if M <= 128:
        assert torch.equal(fused.view(iv), twostep.view(iv)), "fused quantization differs from the two-step path"
    rqa, rsa = oracle.quant_act_1x128(X)
    rqb, rsb = oracle.quant_w_128x128(W)
    rows = _sample_rows(M, 16, M)
    Cr, S = oracle.gemm_blockscaled(rqa, rsa, rqb, rsb, rows=rows)
    for C, what in ((fused, "bf16a"), (twostep, "two-step")):
        Cg = bf16_out_to_f64(C) if dt == torch.bfloat16 else C.cpu().numpy().astype(np.float64)
        assert_within_bound(Cg[rows], Cr, S, f"{what} {M}x{N}x{K}")


def test_bf16a_row_stride_and_rejects_large_m():
    rng = np.random.default_rng(8)
    X = wl.bf16_normal(rng, (32, 1024))
    W = wl.bf16_normal(rng, (256, 512), 0.02)
    big = dev_bf16(X)[:, :512]                       # ldx = 1024 > K = 512
    qb, sb = fg.fp8_quant_w_128x128(dev_bf16(W))
    fused = fg.fp8_gemm_bf16a_blockscaled(big, qb, sb)
    qa, sa, _, _ = fg.fp8_quant_act_1x128(big.contiguous())
    twostep = fg.fp8_gemm_blockscaled(qa, sa, qb, sb)
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int16), twostep.view(torch.int16))
    with pytest.raises(fg.FGF8Error, match="UNSUPPORTED_SHAPE"):
        fg.fp8_gemm_bf16a_blockscaled(dev_bf16(wl.bf16_normal(rng, (257, 512))), qb, sb)


# One workspace serves every GEMM kernel in turn: a small-M split-K call and a
# masked call (both reduced within their clusters) and a last-wave split call
# (arrival counters in their own region, no partial sums written there) leave
# the counters at zero.  Each result is checked against the oracle.
def test_one_workspace_serves_every_kernel():
    L = fg.lib()
    need = max(L.fgf8_gemm_workspace_bytes(16, 1024, 2048, 1), L.fgf8_gemm_workspace_bytes(384, 3072, 1792, 1),
               L.fgf8_masked_gemm_workspace_bytes(4, 64, 256, 1024))
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    rng = np.random.default_rng(77)
    small = (wl.bf16_normal(rng, (16, 2048), 1.0, 0.01, 100.0), wl.bf16_normal(rng, (1024, 2048), 0.02))
    split = (wl.bf16_normal(rng, (384, 1792), 1.0, 0.01, 100.0), wl.bf16_normal(rng, (3072, 1792), 0.02))
    w = wl.masked_small(9, [40, 0, 7, 64], 64, 256, 1024)
    assert fg.fgf8_testing_gemm_schedule(16, 1024, 2048)["small_m"] == 1
    assert fg.fgf8_testing_gemm_schedule(384, 3072, 1792)["tail_s"] > 1
    for round_ in range(2):
        for A, B in (small, split):
            rows = _rows_per_block(A.shape[0], 2, round_)
            Cg, Cr, S = _run_dense(A, B, torch.float32, rows=rows, workspace=ws)
            assert_within_bound(Cg, Cr, S, f"{A.shape[0]}x{B.shape[0]} pass {round_}")
        g, Cg, Cr, S = _run_masked(w, torch.float32, workspace=ws)
        for e, c in enumerate(g.counts):
            if c:
                assert_within_bound(Cg[e, :c], Cr[e, :c], S[e, :c], f"masked expert {e} pass {round_}")
    assert not bool(ws[256:1280].any()), "arrival counters left non-zero"
