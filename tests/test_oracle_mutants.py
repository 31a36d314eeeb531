"""The oracle's pins are sensitive: each plausible mistake planted in a copy
of the oracle source (a wrong constant, rounding rule, sign, index, dropped
term or transposed operand) makes at least one pin test fail.

Each C mutant is compiled with the oracle's own flags and the pin tests run
against it in a child process; the planted mistakes all stay within the
buffers' bounds.  The oracle's Python layer (the masked layout's slot
arithmetic, the W^T wrapper) gets the same treatment: a mutated copy of the
package runs the pins in a scratch directory.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_e4m3.py", "tests/test_oracle_quant.py", "tests/test_oracle_gemm.py"]

MUTANTS = {
    "scale_constant": ("float s = amax / ORACLE_E4M3_MAX;", "float s = amax / 447.0f;"),
    "round_half_up": ("return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "return fl + 1.0;"),
    "no_subnormal_range": ("if (E < -6) E = -6;", ";"),
    "reciprocal_multiply": ("float y = vals[i] / s;", "float y = vals[i] * (1.0f / s);"),
    "late_saturation": ("if (a >= 448.0) return (uint8_t)(sign | 0x7E);",
                        "if (a >= 480.0) return (uint8_t)(sign | 0x7E);"),
    "decode_drops_sign": ("return neg ? -mag : mag;", "return mag;"),
    "amax_signed": ("if (a > amax) amax = a;", "if (vals[i] > amax) amax = vals[i];"),
    "zero_tile_sign": ("codes[i] = signbit(vals[i]) ? 0x80 : 0x00;", "codes[i] = 0x00;"),
    "act_scale_layout": ("s[kb * lds + m] = quant_group(vals, 128, codes);",
                         "s[m * (K / 128) + kb] = quant_group(vals, 128, codes);"),
    "transposed_output_index": ("qT[k * M + m0 + i] = codes[i];", "qT[(m0 + i) * K + k] = codes[i];"),
    "block_amax_one_row": ("s[kb * lds + nb] = quant_group(vals, rows * 128, codes);",
                           "s[kb * lds + nb] = quant_group(vals, 128, codes);"),
    "gemm_transposed_b": ("oracle_e4m3_decode(B[n * K + k])", "oracle_e4m3_decode(B[k * N + n])"),
    "gemm_sa_index": ("* (double)sa[(k / 128) * lda_s + m];", "* (double)sa[(k / 128) * lda_s];"),
    "gemm_sb_kgroup": ("int64_t sidx = (k / 128) * ldb_s + (bkind == 0 ? n / 128 : n);",
                       "int64_t sidx = (bkind == 0 ? n / 128 : n);"),
    "gemm_dropped_term": ("acc += p;", "acc += (k == K - 1) ? 0.0 : p;"),
    "grouped_expert_scales": ("sb + (int64_t)e * KB * ldb_s, ldb_s, 0,", "sb, ldb_s, 0,"),
}


# Mistakes planted in the Python layer of the oracle (oracle/__init__.py).
PY_MUTANTS = {
    "masked_slot_column": ("[:, e * cap:(e + 1) * cap]", "[:, e:e + cap]"),
    "masked_shared_expert_scales": ("B[e], sb[e], 0, rows=rows)", "B[e], sb[0], 0, rows=rows)"),
    "masked_count_unclamped": ("c = int(min(max(int(counts[e]), 0), cap))", "c = int(counts[e])"),
    "wt_not_transposed": ("np.ascontiguousarray(np.asarray(w_bits, np.uint16).T)",
                          "np.ascontiguousarray(np.asarray(w_bits, np.uint16))"),
}


def _run_py_mutant(name, tmpdir):
    before, after = PY_MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert src.count(before) == 1, f"{name}: pattern must occur exactly once"
    work = os.path.join(tmpdir, name)
    os.makedirs(os.path.join(work, "oracle"))
    with open(os.path.join(work, "oracle", "__init__.py"), "w") as f:
        f.write(src.replace(before, after))
    shutil.copy(os.path.join(ROOT, "oracle", "oracle.c"), os.path.join(work, "oracle"))
    shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(work, "tests"),
                    ignore=shutil.ignore_patterns("__pycache__"))
    env = dict(os.environ, FGF8_ORACLE_LIB=oracle.build())
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                       cwd=work, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def _run_mutant(name, tmpdir):
    before, after = MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert src.count(before) == 1, f"{name}: pattern must occur exactly once"
    c = os.path.join(tmpdir, f"{name}.c")
    so = os.path.join(tmpdir, f"{name}.so")
    with open(c, "w") as f:
        f.write(src.replace(before, after))
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-o", so, c, "-lm"])
    env = dict(os.environ, FGF8_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def test_every_planted_mistake_is_caught(tmp_path):
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda n: _run_mutant(n, str(tmp_path)), MUTANTS))
    survivors = [(n, out) for n, rc, out in results if rc != 1]
    assert not survivors, f"mutants not caught (or crashed): {survivors}"


def test_every_planted_python_mistake_is_caught(tmp_path):
    with ThreadPoolExecutor(max_workers=min(4, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda n: _run_py_mutant(n, str(tmp_path)), PY_MUTANTS))
    survivors = [(n, out) for n, rc, out in results if rc != 1]
    assert not survivors, f"mutants not caught (or crashed): {survivors}"


def test_python_mutant_harness_passes_the_unmutated_oracle(tmp_path):
    # the scratch-directory copy itself must not fail the pins
    PY_MUTANTS["_identity"] = ("def round_up(v: int, m: int) -> int:", "def round_up(v: int, m: int) -> int:")
    try:
        name, rc, out = _run_py_mutant("_identity", str(tmp_path))
    finally:
        del PY_MUTANTS["_identity"]
    assert rc == 0, out
