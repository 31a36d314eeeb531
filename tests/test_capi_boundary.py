"""The C-ABI library loads, exports every function the headers declare, and
rejects bad arguments on the host with the documented status codes (these
checks run before any device call, so no GPU is needed)."""
import ctypes
import os
import re

import pytest

import fine_grained_fp8_weight_b300 as fg
from fine_grained_fp8_weight_b300 import build as fgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    fgbuild.build()
    return fg.lib()


def _declared():
    names = set()
    for h in ("fgf8.h", "fgf8_testing.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b((?:fp8|fgf8)_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(L):
    declared = _declared()
    assert declared == set(fg.EXPORTED)
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings(L):
    for code in range(8):
        assert L.fgf8_status_string(code)
    assert L.fgf8_version().startswith(b"fgf8")


# fake, never-dereferenced device addresses
A16 = ctypes.c_void_p(0x10000)
MIS = ctypes.c_void_p(0x10008)


def test_quant_act_rejects(L):
    f = L.fp8_quant_act_1x128
    assert f(None, 4, 128, 128, A16, A16, 4, None, None, 0, None) == 1         # null x
    assert f(A16, 4, 128, 128, None, None, 0, None, None, 0, None) == 1      # no output
    assert f(A16, 4, 128, 128, A16, None, 4, None, None, 0, None) == 1       # q without s
    assert f(A16, 4, 100, 100, A16, A16, 4, None, None, 0, None) == 3        # K % 128
    assert f(A16, 4, 128, 128, A16, A16, 2, None, None, 0, None) == 1        # lds < M
    assert f(A16, 4, 128, 128, A16, A16, 6, None, None, 0, None) == 1        # lds % 4
    assert f(MIS, 4, 128, 128, A16, A16, 4, None, None, 0, None) == 2        # x misaligned
    assert f(A16, 4, 128, 132, A16, A16, 4, None, None, 0, None) == 2        # ldx % 8
    assert f(A16, 20, 128, 128, None, None, 0, A16, A16, 128, None) == 3     # qT needs M % 16
    assert f(A16, 16, 128, 128, None, None, 0, A16, A16, 126, None) == 1     # ldsT < K


def test_quant_w_rejects(L):
    f = L.fp8_quant_w_128x128
    assert f(None, 128, 128, 128, A16, A16, 4, None) == 1
    assert f(A16, 128, 200, 200, A16, A16, 4, None) == 3
    assert f(A16, 300, 128, 128, A16, A16, 2, None) == 1                     # lds < ceil(N/128)
    assert f(A16, 128, 128, 128, MIS, A16, 4, None) == 2


def test_gemm_rejects(L):
    f = L.fp8_gemm_blockscaled
    ok = dict(A=A16, sa=A16, ldsa=4, B=A16, sb=A16, ldsb=4, bk=0, C=A16, ldc=128, cdt=0,
              M=4, N=128, K=128, ws=A16, wsb=1 << 20, st=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["A"], a["sa"], a["ldsa"], a["B"], a["sb"], a["ldsb"], a["bk"], a["C"], a["ldc"], a["cdt"],
                 a["M"], a["N"], a["K"], a["ws"], a["wsb"], a["st"])

    assert call(A=None) == 1
    assert call(ws=None) == 1
    assert call(M=0) == 1
    assert call(bk=5) == 1
    assert call(cdt=3) == 1
    assert call(K=200) == 3
    assert call(N=120, ldc=120) == 3
    assert call(ldsa=2) == 1
    assert call(bk=1, ldsb=64) == 1          # per-row scales need ldsb >= N
    assert call(ldc=100) == 1
    assert call(B=MIS) == 2
    assert call(ldc=132) == 2                # 264-byte rows are not 16-byte multiples
    assert call(ws=ctypes.c_void_p(0x10010)) == 2
    assert call(wsb=16) == 5


def test_grouped_rejects(L):
    f = L.fp8_grouped_gemm_blockscaled
    base = [A16, A16, 256, A16, A16, 4, A16, 2, A16, 128, 0, 256, 128, 128, A16, 1 << 20, None]
    bad = list(base); bad[6] = None
    assert f(*bad) == 1                      # no m_indices
    bad = list(base); bad[11] = 200
    assert f(*bad) == 3                      # M_total % 128
    bad = list(base); bad[7] = 0
    assert f(*bad) == 1                      # no experts


def test_quant_w_grouped_and_transposed_reject(L):
    g = L.fp8_quant_w_128x128_grouped
    assert g(A16, -1, 256, 128, 128, A16, A16, 4, None) == 1          # negative expert count
    assert g(A16, 2, 256, 200, 200, A16, A16, 4, None) == 3           # K % 128
    assert g(A16, 0, 256, 128, 128, None, None, 0, None) == 0          # no experts: nothing touched
    assert g(None, 2, 256, 128, 128, A16, A16, 4, None) == 1
    assert g(A16, 2, 256, 128, 100, A16, A16, 4, None) == 1           # ldw < K
    assert g(A16, 2, 256, 128, 128, A16, A16, 6, None) == 1           # lds % 4
    assert g(A16, 2, 256, 128, 128, MIS, A16, 4, None) == 2
    t = L.fp8_quant_w_128x128_t
    assert t(A16, 200, 128, 128, A16, A16, 4, None, None, 0, None) == 3   # N % 128 (W^T's K groups)
    assert t(A16, 256, 200, 200, A16, A16, 4, None, None, 0, None) == 3   # K % 128
    assert t(A16, 0, 128, 128, None, None, 0, None, None, 0, None) == 0   # empty: nothing touched
    assert t(A16, 256, 128, 128, None, A16, 4, None, None, 0, None) == 1  # no qT
    assert t(A16, 256, 384, 384, A16, A16, 2, None, None, 0, None) == 1   # ldsT < K/128
    assert t(A16, 256, 128, 128, A16, A16, 4, A16, None, 4, None) == 1    # q without s
    assert t(A16, 256, 128, 128, A16, A16, 4, A16, A16, 1, None) == 1     # lds < N/128
    assert t(A16, 256, 128, 132, A16, A16, 4, None, None, 0, None) == 2   # ldw % 8
    assert t(A16, 256, 128, 128, A16, A16, 4, MIS, A16, 4, None) == 2     # q misaligned


def test_masked_rejects(L):
    f = L.fp8_masked_grouped_gemm_blockscaled
    ok = dict(A=A16, sa=A16, ldsa=128, B=A16, sb=A16, ldsb=4, cnt=A16, E=2, cap=64, C=A16, ldc=256, cdt=0,
              N=256, K=512, ws=A16, wsb=1 << 26, st=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["A"], a["sa"], a["ldsa"], a["B"], a["sb"], a["ldsb"], a["cnt"], a["E"], a["cap"], a["C"],
                 a["ldc"], a["cdt"], a["N"], a["K"], a["ws"], a["wsb"], a["st"])

    assert call(E=0, A=None, cnt=None) == 0      # no experts: nothing touched
    assert call(E=-1) == 1
    assert call(cnt=None) == 1
    assert call(cdt=2) == 1
    assert call(cap=72) == 3                     # cap % 16
    assert call(cap=272, ldsa=544) == 3          # cap > 256
    assert call(N=250, ldc=256) == 3             # N % 16
    assert call(ldsa=100) == 1                   # ldsa < E * cap
    assert call(ldsb=1, N=256) == 1              # ldsb < ceil(N/128)... and % 4
    assert call(ldc=200) == 1
    assert call(cnt=ctypes.c_void_p(0x10002)) == 2   # counts not 4-byte aligned
    assert call(ws=ctypes.c_void_p(0x10010)) == 2    # workspace not 256-byte aligned
    need = L.fgf8_masked_gemm_workspace_bytes(2, 64, 256, 512)
    assert need == 256                           # the status header: the split reduces within its cluster
    assert call(wsb=need - 1) == 5


def test_bf16a_rejects(L):
    f = L.fp8_gemm_bf16a_blockscaled
    ok = dict(x=A16, ldx=512, B=A16, sb=A16, ldsb=4, C=A16, ldc=256, cdt=0, M=16, N=256, K=512,
              ws=A16, wsb=1 << 26, st=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["x"], a["ldx"], a["B"], a["sb"], a["ldsb"], a["C"], a["ldc"], a["cdt"], a["M"], a["N"],
                 a["K"], a["ws"], a["wsb"], a["st"])

    assert call(M=0, x=None) == 0                # empty output: nothing touched
    assert call(x=None) == 1
    assert call(M=257) == 3                      # at most 256 tokens
    assert call(K=200, ldx=200) == 3
    assert call(N=250, ldc=256) == 3
    assert call(ldx=256) == 1                    # ldx < K
    assert call(ldsb=2) == 1
    assert call(x=MIS) == 2
    assert call(ldx=516) == 2                    # BF16 rows must be 16-byte multiples
    assert call(wsb=16) == 5


def test_probe_rejects(L):
    f = L.fgf8_mma_probe
    assert f(A16, A16, A16, 24, 128, A16, None) == 3
    assert f(A16, A16, A16, 512, 128, A16, None) == 3
    assert f(A16, A16, A16, 32, 100, A16, None) == 3
    assert f(None, A16, A16, 32, 128, A16, None) == 1


def test_workspace_size(L):
    assert L.fgf8_gemm_workspace_bytes(4096, 18432, 7168, 1) >= 256
    assert L.fgf8_gemm_workspace_min_bytes(4096, 18432, 7168, 1) >= 256
    # the recommended size holds the last-wave split, the least does not need to
    for shape in [(4096, 18432, 7168), (4096, 7168, 18432), (16, 4096, 7168), (384, 3072, 1792)]:
        assert L.fgf8_gemm_workspace_bytes(*shape, 1) >= L.fgf8_gemm_workspace_min_bytes(*shape, 1)
    assert L.fgf8_gemm_workspace_min_bytes(4096, 7168, 18432, 1) <= 1 << 20


# --- schedule choice (host only) ---

def _tiles(M, N, sch):
    rows = 256 if sch["pair"] else 128          # a CTA pair covers two 128-row blocks
    return -(-M // rows) * -(-N // sch["bn"])


@pytest.fixture
def pair_on(L):
    """The CTA-pair kernel switched on for one test (process-wide switch)."""
    assert L.fgf8_testing_set_pair(1) == 0
    try:
        yield
    finally:
        assert L.fgf8_testing_set_pair(0) == 0


def _check_split_invariants(sms, bkind, pair):
    seen_split = 0
    for M in (257, 384, 1000, 1280, 2560, 4096, 7168):
        for N in (512, 1792, 3072, 4096, 7168, 18432):
            for K in (128, 1024, 2048, 7168, 18432):
                sch = fg.fgf8_testing_gemm_schedule(M, N, K, bkind, num_sms=sms)
                if sch["small_m"]:
                    continue
                assert sch["pair"] == pair
                G = sms // 2 if sch["pair"] else min(sms, 148)
                tiles = _tiles(M, N, sch)
                if sch["tail_s"] == 1:
                    assert sch["dp_tiles"] == tiles
                    continue
                seen_split += 1
                R = tiles - sch["dp_tiles"]
                assert sch["dp_tiles"] % G == 0 and 0 < R < G
                assert 2 <= sch["tail_s"] <= K // 128 and R * sch["tail_s"] <= G
                # with the least workspace the same GEMM runs whole tiles only
                wmin = fg.lib().fgf8_gemm_workspace_min_bytes(M, N, K, 1)
                plain = fg.fgf8_testing_gemm_schedule(M, N, K, bkind, ws_bytes=wmin, num_sms=sms)
                assert plain["tail_s"] == 1 and plain["dp_tiles"] == _tiles(M, N, plain)
    assert seen_split > 10


@pytest.mark.parametrize("sms", [148, 132, 64])
@pytest.mark.parametrize("bkind", [0, 1])
def test_last_wave_split_invariants(L, sms, bkind):
    """Whole tiles fill whole waves over min(SMs, 148) CTAs; the rest (fewer
    than that) are cut into s <= K/128 pieces that fit one more wave."""
    _check_split_invariants(sms, bkind, 0)


@pytest.mark.parametrize("sms", [148, 132])
def test_pair_last_wave_split_invariants(L, pair_on, sms):
    """The same for the CTA-pair kernel: SMs / 2 pairs, 256 x 128 tiles."""
    _check_split_invariants(sms, 0, 1)
    assert fg.fgf8_testing_gemm_schedule(4096, 18432, 7168, 1)["pair"] == 0   # per-row B scales: single SMs


def test_schedule_of_the_prefill_pair_and_wgrad(L):
    # 4096 x 7168 x 18432: 896 tiles of 128 x 256 = 6 waves + 8; the 8 run as
    # 8 K pieces each (18 K groups per piece) next to the 6 whole waves
    assert fg.fgf8_testing_gemm_schedule(4096, 7168, 18432) == {"small_m": 0, "bn": 256, "dp_tiles": 888,
                                                                "tail_s": 8, "pair": 0}
    # 4096 x 18432 x 7168: 2304 tiles = 15 waves + 84; splitting 84 tiles
    # cannot fill a wave better than whole tiles do
    assert fg.fgf8_testing_gemm_schedule(4096, 18432, 7168)["tail_s"] == 1
    # weight gradient 7168 x 2048 x 8192 (per-row B scales): 448 tiles = 3 waves + 4
    sch = fg.fgf8_testing_gemm_schedule(7168, 2048, 8192, 1)
    assert sch["bn"] == 256 and sch["dp_tiles"] == 444 and sch["tail_s"] > 1
    assert fg.fgf8_testing_gemm_schedule(16, 4096, 7168)["small_m"] == 1
    # decode: up to 128 tokens on the small-M kernel (K over 4 CTAs per weight
    # tile for N = 4096); 256 tokens on 64 large tiles of 128 x 128 cut into
    # 2 K pieces (128 CTAs)
    assert fg.fgf8_testing_gemm_schedule(128, 4096, 7168) == {"small_m": 1, "bn": 0, "dp_tiles": 0,
                                                              "tail_s": 4, "pair": 0}
    assert fg.fgf8_testing_gemm_schedule(256, 4096, 7168) == {"small_m": 0, "bn": 128, "dp_tiles": 0,
                                                              "tail_s": 2, "pair": 0}


def test_pair_schedule_of_the_prefill_pair(L, pair_on):
    # 4096 x 18432 x 7168 on 74 pairs: 16 x 144 = 2304 tiles of 256 x 128 = 31
    # waves + 10; the 10 run as 4 K pieces each
    assert fg.fgf8_testing_gemm_schedule(4096, 18432, 7168) == {"small_m": 0, "bn": 128, "dp_tiles": 2294,
                                                                "tail_s": 4, "pair": 1}
    # one 128-row block: single-SM tiles
    assert fg.fgf8_testing_gemm_schedule(128, 18432, 7168)["pair"] == 0


def test_set_pair_rejects(L):
    assert L.fgf8_testing_set_pair(3) == 1
    assert L.fgf8_testing_set_pair(-1) == 1


@pytest.fixture
def multicast_on(L):
    """Clusters of two 128 x 256 tiles sharing B by TMA multicast, for one test."""
    assert L.fgf8_testing_set_pair(2) == 0
    try:
        yield
    finally:
        assert L.fgf8_testing_set_pair(0) == 0


@pytest.mark.parametrize("sms", [148, 132])
def test_multicast_last_wave_split_invariants(L, multicast_on, sms):
    """The same for multicast clusters: SMs / 2 clusters, cluster tiles of
    two 128-row blocks x 256 columns."""
    _check_split_invariants(sms, 0, 2)
    assert fg.fgf8_testing_gemm_schedule(4096, 18432, 7168, 1)["pair"] == 0   # per-row B scales: single CTAs


def test_multicast_schedule_of_the_prefill_pair(L, multicast_on):
    # 4096 x 18432 x 7168 on 74 clusters: 16 x 72 = 1152 cluster tiles = 15
    # waves + 42, run whole as on single CTAs (no split beats them);
    # 4096 x 7168 x 18432: 448 = 6 waves + 4, cut into 8 K pieces each
    assert fg.fgf8_testing_gemm_schedule(4096, 18432, 7168) == {"small_m": 0, "bn": 256, "dp_tiles": 1152,
                                                                "tail_s": 1, "pair": 2}
    assert fg.fgf8_testing_gemm_schedule(4096, 7168, 18432) == {"small_m": 0, "bn": 256, "dp_tiles": 444,
                                                                "tail_s": 8, "pair": 2}
    assert fg.fgf8_testing_gemm_schedule(128, 18432, 7168)["pair"] == 0   # one 128-row block
    assert fg.fgf8_testing_gemm_schedule(64, 4096, 7168)["small_m"] == 1


def test_schedule_rejects(L):
    out = (ctypes.c_int32 * 5)()
    f = L.fgf8_testing_gemm_schedule
    assert f(0, 128, 128, 0, 1 << 20, 148, out) == 1
    assert f(128, 128, 100, 0, 1 << 20, 148, out) == 1
    assert f(128, 128, 128, 2, 1 << 20, 148, out) == 1
    assert f(128, 128, 128, 0, 1 << 20, 0, out) == 1
    assert f(128, 128, 128, 0, 1 << 20, 148, None) == 1


def test_small_m_cluster_sizes(L):
    """The small-M kernel's K split is one thread-block cluster per weight tile:
    at most 8 CTAs (the portable cluster size), at most K/128, and all
    clusters fit one wave of the SMs."""
    seen = set()
    for M in (1, 16, 33, 64, 128):
        for N in (16, 128, 256, 1024, 2048, 4096, 7168, 9472):
            for K in (128, 256, 512, 2048, 7168, 18432):
                sch = fg.fgf8_testing_gemm_schedule(M, N, K)
                if not sch["small_m"]:
                    assert N > 74 * 128
                    continue
                S = sch["tail_s"]
                tiles = (N + 127) // 128
                assert 1 <= S <= min(8, K // 128), (M, N, K, S)
                assert tiles * S <= 148, (M, N, K, S)
                seen.add(S)
    assert seen >= {1, 2, 4, 8}
