"""GPU parity of the quantization kernels: E4M3 codes and scales bit-exact
against the oracle, through the C ABI, on seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import fine_grained_fp8_weight_b300 as fg
from fine_grained_fp8_weight_b300 import workloads as wl
from tests.gpu_util import DEV, assert_codes_equal, assert_scales_equal, dev_bf16, ensure_built, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _check_rows(bits):
    M, K = bits.shape
    q, s, _, _ = fg.fp8_quant_act_1x128(dev_bf16(bits))
    rq, rs = oracle.quant_act_1x128(bits)
    assert_codes_equal(host(q), rq)
    assert_scales_equal(host(s), rs, M)


def _check_transposed(bits, rows_too):
    M, K = bits.shape
    q, s, qT, sT = fg.fp8_quant_act_1x128(dev_bf16(bits), rows=rows_too, transposed=True)
    rqT, rsT = oracle.quant_act_128x1(bits)
    assert_codes_equal(host(qT), rqT)
    assert_scales_equal(host(sT), rsT, K)
    if rows_too:
        rq, rs = oracle.quant_act_1x128(bits)
        assert_codes_equal(host(q), rq)
        assert_scales_equal(host(s), rs, M)


def _check_weights(bits):
    N, K = bits.shape
    q, s = fg.fp8_quant_w_128x128(dev_bf16(bits))
    rq, rs = oracle.quant_w_128x128(bits)
    assert_codes_equal(host(q), rq)
    assert_scales_equal(host(s), rs, (N + 127) // 128)


@pytest.mark.parametrize("M,K", [(1, 128), (5, 384), (64, 512), (130, 1024), (1000, 640), (2053, 256)])
def test_act_rows_random(M, K):
    rng = np.random.default_rng(M * 7 + K)
    _check_rows(wl.bf16_normal(rng, (M, K), 1.0, 0.01, 100.0))


@pytest.mark.parametrize("M,K,rows_too", [(128, 128, False), (144, 256, True), (256, 384, False),
                                          (400, 128, True), (16, 512, True), (1024, 1024, True)])
def test_act_transposed_random(M, K, rows_too):
    rng = np.random.default_rng(M + K)
    _check_transposed(wl.bf16_normal(rng, (M, K), 1.0, 0.001, 50.0), rows_too)


@pytest.mark.parametrize("N,K", [(128, 128), (200, 384), (256, 512), (1000, 256), (16, 128)])
def test_weights_random(N, K):
    rng = np.random.default_rng(N * 3 + K)
    _check_weights(wl.bf16_normal(rng, (N, K), 0.02))


def _edge_tensor(rows, K):
    """Tiles that exercise the rule's corners: zero and negative-zero tiles,
    subnormal and huge max-abs, values on E4M3 rounding midpoints, the
    divide-vs-reciprocal and double-rounding cases."""
    rng = np.random.default_rng(99)
    x = (rng.standard_normal((rows, K)) * np.exp2(rng.integers(-20, 20, (rows, 1)))).astype(np.float32)
    x[0, 0:128] = 0.0
    x[1, 0:128] = -0.0
    x[2, 0:128] = rng.standard_normal(128).astype(np.float32) * np.float32(1e-39)   # BF16 subnormals
    x[3, 0:128] = rng.standard_normal(128).astype(np.float32) * np.float32(1e37)
    mids = np.array([17.0, 19.0, 0.0009765625, -0.0029296875, 168.0, 336.0, 1.5, -2.25], np.float32)
    x[4, 0:128] = 0.0
    x[4, 0] = 448.0
    x[4, 1:1 + len(mids)] = mids
    x[5, 0:128] = 0.0
    x[5, 0], x[5, 1] = 3.875, 1.453125
    x[6, 0:128] = 0.0
    x[6, 0], x[6, 1] = 11.25, 8.4375
    x[7, 0:128] = np.float32(2.0 ** -133)        # smallest BF16 subnormal everywhere
    return wl.to_bf16_bits(x)


def test_act_rows_edge_cases():
    _check_rows(_edge_tensor(16, 256))


def test_act_transposed_edge_cases():
    # the edge tiles laid along the token direction: channel c, tokens 0..127
    # hold edge row c of the row-direction case
    x = _edge_tensor(16, 256)
    xt = np.zeros((256, 128), np.uint16)
    xt[:, :16] = x.T
    _check_transposed(xt, rows_too=True)


def test_weights_edge_cases():
    x = _edge_tensor(256, 256)
    _check_weights(x)
    z = np.zeros((130, 128), np.uint16)
    _check_weights(z)


def test_empty_input_is_a_noop():
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device=DEV)
    q, s, _, _ = fg.fp8_quant_act_1x128(x)
    assert q.shape == (0, 256)


def test_row_stride_larger_than_k():
    rng = np.random.default_rng(5)
    bits = wl.bf16_normal(rng, (50, 512), 1.0, 0.01, 100.0)
    full = dev_bf16(bits)
    view = full[:, :384]
    q, s, _, _ = fg.fp8_quant_act_1x128(view)
    rq, rs = oracle.quant_act_1x128(np.ascontiguousarray(bits[:, :384]))
    assert_codes_equal(host(q), rq)
    assert_scales_equal(host(s), rs, 50)


def test_e4m3_pair_byte_order():
    # one tile whose codes are all distinct positions: lane packing must keep
    # element i at byte i
    vals = np.zeros((1, 128), np.float32)
    vals[0, :16] = [448, 1, 2, 3, 4, 5, 6, 7, -1, -2, -3, -4, -5, -6, -7, -8]
    _check_rows(wl.to_bf16_bits(vals))


# --- full-size tensors of the five workloads, sampled rows / block rows ---

def _sampled_rows_check(bits, nrows, seed):
    M, K = bits.shape
    q, s, _, _ = fg.fp8_quant_act_1x128(dev_bf16(bits))
    rows = np.random.default_rng(seed).choice(M, size=min(nrows, M), replace=False)
    rq, rs = oracle.quant_act_1x128(np.ascontiguousarray(bits[rows]))
    qh = host(q)
    sh = host(s)
    assert_codes_equal(qh[rows], rq)
    assert np.array_equal(sh[:, rows].view(np.uint32), rs[:, :len(rows)].view(np.uint32))


def _sampled_blocks_check(bits, nblocks, seed):
    N, K = bits.shape
    q, s = fg.fp8_quant_w_128x128(dev_bf16(bits))
    nb_total = (N + 127) // 128
    blocks = np.random.default_rng(seed).choice(nb_total, size=min(nblocks, nb_total), replace=False)
    qh, sh = host(q), host(s)
    for nb in blocks:
        r0, r1 = nb * 128, min(N, nb * 128 + 128)
        rq, rs = oracle.quant_w_128x128(np.ascontiguousarray(bits[r0:r1]))
        assert_codes_equal(qh[r0:r1], rq)
        assert np.array_equal(sh[:, nb].view(np.uint32), rs[:, 0].view(np.uint32))


def test_full_size_prefill_tensors():
    w = wl.prefill_pair()
    up, down = w.gemms
    _sampled_rows_check(up.A, 64, 1)
    _sampled_blocks_check(up.B, 6, 2)
    _sampled_rows_check(down.A, 32, 3)
    _sampled_blocks_check(down.B, 4, 4)


def test_full_size_wgrad_transposed():
    # one channel of every 128-channel group, its position in the group
    # cycling through 0..127 (the kernel maps its warps to 8-channel x
    # 4-token octets, so every octet position of the mapping is visited)
    w = wl.wgrad().gemms[0]
    for x in (w.dY, w.X):
        T, C = x.shape
        _, _, qT, sT = fg.fp8_quant_act_1x128(dev_bf16(x), rows=False, transposed=True)
        chans = np.array([g * 128 + (g * 37 + 5) % 128 for g in range(C // 128)])
        rqT, rsT = oracle.quant_act_128x1(np.ascontiguousarray(x[:, chans]))
        assert_codes_equal(host(qT)[chans], rqT)
        assert np.array_equal(host(sT)[:, chans].view(np.uint32), rsT[:, :len(chans)].view(np.uint32))


def test_full_size_decode_and_tiny():
    for g in wl.tiny().gemms + wl.decode().gemms[:2]:
        _check_rows(g.A)
    _check_weights(wl.tiny().gemms[0].B)


# --- W^T for the data-gradient GEMM (128x128 blocks written transposed) ---


def _check_weights_t(bits, forward):
    N, K = bits.shape
    out = fg.fp8_quant_w_128x128_t(dev_bf16(bits), forward=forward)
    rqT, rsT = oracle.quant_w_128x128_t(bits)
    assert_codes_equal(host(out[0]), rqT)
    assert_scales_equal(host(out[1]), rsT, K // 128)
    if forward:
        rq, rs = oracle.quant_w_128x128(bits)
        assert_codes_equal(host(out[2]), rq)
        assert_scales_equal(host(out[3]), rs, N // 128)


@pytest.mark.parametrize("N,K,forward", [(128, 128, False), (256, 384, True), (384, 128, False),
                                         (1024, 640, True), (128, 2048, False)])
def test_weights_transposed_random(N, K, forward):
    rng = np.random.default_rng(N * 5 + K)
    _check_weights_t(wl.bf16_normal(rng, (N, K), 0.02, 0.001, 50.0), forward)


def test_weights_transposed_edge_cases():
    _check_weights_t(_edge_tensor(256, 256), forward=True)
    _check_weights_t(np.zeros((128, 256), np.uint16), forward=True)


def test_weights_transposed_rejects_ragged_n():
    w = torch.zeros((200, 256), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fg.FGF8Error, match="UNSUPPORTED_SHAPE"):
        fg.fp8_quant_w_128x128_t(w)


def test_full_size_dgrad_weight():
    g = wl.dgrad().gemms[0]
    qT, sT = fg.fp8_quant_w_128x128_t(dev_bf16(g.W))
    torch.cuda.synchronize()
    # sampled 128-column blocks of W (= 128-row blocks of W^T), checked whole
    rng = np.random.default_rng(21)
    for kb in rng.choice(g.W.shape[1] // 128, size=3, replace=False):
        cols = slice(int(kb) * 128, int(kb) * 128 + 128)
        rqT, rsT = oracle.quant_w_128x128_t(np.ascontiguousarray(g.W[:, cols]))
        assert_codes_equal(host(qT[cols]), rqT)
        assert_scales_equal(host(sT[:, int(kb):int(kb) + 1]), rsT, 1)
