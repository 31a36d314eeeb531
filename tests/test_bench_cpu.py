"""bench.py on the host: the reference arm (the oracle, no GPU) runs end to end
and prints one JSON line with the contract's keys."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0


def test_oracle_sample_covers_every_gemm_kind():
    # the host-side oracle timing of bench.py's workloads key runs on every
    # GEMM layout of the path (small shapes of each) and counts its work
    sys.path.insert(0, ROOT)
    import bench
    from fine_grained_fp8_weight_b300 import workloads as wl
    works = [wl.tiny(), wl.grouped_small(1, [130, 0, 7], 256, 256), wl.wgrad(2, T=256, N=256, K=128),
             wl.dgrad(3, T=128, N=256, K=256), wl.masked_small(4, [5, 0, 16], 16, 256, 256)]
    for w in works:
        flops, secs, full = bench.oracle_sample(w, 3, 2, seed=0)
        assert flops > 0 and secs > 0 and full >= secs * 0.5, w.name


def test_measured_traffic_names_this_build():
    # the roofline line's DRAM traffic is keyed by the library's version
    # string; a build that changes a kernel changes the string, and the
    # prefill GEMMs' ncu totals must be recorded for it (else the bench
    # line would carry traffic: null)
    sys.path.insert(0, ROOT)
    import bench
    import fine_grained_fp8_weight_b300 as fg
    version = fg.lib().fgf8_version().decode()
    entry = bench.MEASURED_TRAFFIC.get(version)
    assert entry is not None, f"no DRAM traffic recorded for {version}"
    for op in ("up.gemm", "down.gemm"):
        assert entry.get(f"prefill_pair_4096x18432x7168/{op}", 0) > 0, op
