"""Benchmark of the fine-grained FP8 hot path on B300.

One step = the whole path over the prefill projection pair (GEMM1 4096 x
18432 x 7168, GEMM2 4096 x 7168 x 18432, BF16 output):

    quantize A1 (1x128) -> quantize W1 (128x128) -> block-scaled GEMM1 ->
    quantize A2 (1x128) -> quantize W2 (128x128) -> block-scaled GEMM2

``value`` is the step's GEMM FLOPs (2*M*N*K summed over both GEMMs) divided by
the device time of the step, with all inputs resident in HBM (BF16 inputs of
738 MB per step, larger than the 126 MB L2, so no flush is needed between
steps).  The step is captured once as a CUDA graph and replayed, so that the
timed region holds device work only; per-kernel times replay each op's own
graph with an L2 flush between replays.  The JSON line also carries the roofline of the dominant kernel (the
GEMM), per-kernel times, quantize bandwidth, an end-to-end figure through the
public API with pinned host buffers, and the CPU oracle timed on a bounded
sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload prefill|decode|moe|wgrad|tiny] [--profile-gemm]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "block-scaled FP8 GEMM TFLOP/s (% of FP8 peak); quantize GB/s (% of HBM)"
FP8_PER_BF16 = 2.0          # nominal dense FP8 : BF16 tensor rate on Blackwell
FUSED_A_MAX_M = 256         # token count up to which fp8_gemm_bf16a_blockscaled takes BF16 tokens

# DRAM bytes (read + write) of one launch, from an ncu capture of that exact
# kernel build (profiles/ holds the summaries).  Keyed by the library version
# string, which changes whenever a kernel changes, so a stale figure is never
# reported: a kernel without a capture of its current build reports null.
MEASURED_TRAFFIC = {
    "fgf8 0.13 sm_103a": {                                   # profiles/gemm_blockscaled_prefill_traffic.md
        "prefill_pair_4096x18432x7168/up.gemm": 166400000 + 126772480,
        "prefill_pair_4096x18432x7168/down.gemm": 520134400 + 51309312,
    },
    # 0.12 changed the masked-layout small-M launch only: the prefill GEMMs run the 0.10 kernel
    "fgf8 0.12 sm_103a": {                                   # profiles/gemm_blockscaled_prefill_traffic.md
        "prefill_pair_4096x18432x7168/up.gemm": 167797760 + 126922240,
        "prefill_pair_4096x18432x7168/down.gemm": 522013696 + 51453184,
    },
    # 0.11 changed the per-row-B promotion only: the prefill GEMMs (block B scales) run the
    # 0.10 kernel unchanged
    "fgf8 0.11 sm_103a": {                                   # profiles/gemm_blockscaled_prefill_traffic.md
        "prefill_pair_4096x18432x7168/up.gemm": 167797760 + 126922240,
        "prefill_pair_4096x18432x7168/down.gemm": 522013696 + 51453184,
    },
    "fgf8 0.10 sm_103a": {                                   # profiles/gemm_blockscaled_prefill_traffic.md
        "prefill_pair_4096x18432x7168/up.gemm": 167797760 + 126922240,
        "prefill_pair_4096x18432x7168/down.gemm": 522013696 + 51453184,
    },
    "fgf8 0.9 sm_103a": {                                    # profiles/gemm_blockscaled_prefill_traffic.md
        "prefill_pair_4096x18432x7168/up.gemm": 166803456 + 126609152,
        "prefill_pair_4096x18432x7168/down.gemm": 521767168 + 51166720,
    },
    "fgf8 0.8 sm_103a": {                                    # profiles/gemm_blockscaled_prefill_traffic.md
        "prefill_pair_4096x18432x7168/up.gemm": 166761216 + 127433216,
        "prefill_pair_4096x18432x7168/down.gemm": 625504256 + 51429632,
    },
    # captured on 0.5; 0.6 changed only the E4M3 encode step (quantizers and the in-GEMM token
    # quantizer), not gemm_blockscaled_kernel
    "fgf8 0.6 sm_103a": {                                    # profiles/gemm_blockscaled_prefill_up.md
        "prefill_pair_4096x18432x7168/up.gemm": 167170048 + 127274240,
        "prefill_pair_4096x18432x7168/down.gemm": 627054848 + 51585280,
    },
}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """SM clock, power and clock-event reasons of the GPU, sampled through the
    driver's NVML library (ctypes) in a background thread every millisecond
    while the timed region runs, so that a region of a few tens of
    milliseconds still gets samples; read-only queries, no setting of the GPU
    is touched.  Falls back to nvidia-smi polling when NVML cannot be loaded."""

    # NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period_s: float = 0.001):
        self.index = index
        self.period = period_s
        self.samples = []          # (sm_mhz, power_w, reason bits)
        self.sm_max = None
        self._stop = threading.Event()
        self.thread = None
        self.nvml = None
        self.proc = None
        self.lines = []
        self.nvml_error = None

    def start(self):
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")      # the driver's NVML, read-only queries only
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit_v2 failed")
            self.nvml = nv
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
                raise RuntimeError("nvmlDeviceGetHandleByIndex_v2 failed")
            NVML_CLOCK_SM = 1
            mx, sm, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
            if nv.nvmlDeviceGetMaxClockInfo(h, NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.sm_max = float(mx.value)
            reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons

            def loop():
                while not self._stop.is_set():
                    if (nv.nvmlDeviceGetClockInfo(h, NVML_CLOCK_SM, ctypes.byref(sm)) == 0 and
                            nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 and
                            reasons(h, ctypes.byref(rs)) == 0):
                        self.samples.append((float(sm.value), pw.value / 1000.0, int(rs.value)))
                    time.sleep(self.period)

            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            t = time.time()
            while not self.samples and time.time() - t < 2.0:     # running before timing starts
                time.sleep(0.001)
            self.samples.clear()
        except Exception as e:  # noqa: BLE001
            self.nvml = None
            self.nvml_error = f"{type(e).__name__}: {e}"[:200]
            self._start_smi()

    def _start_smi(self):
        fields = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={fields}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=lambda: [self.lines.append(l.strip()) for l in self.proc.stdout],
                                           daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def stop(self):
        if self.nvml is not None:
            self._stop.set()
            self.thread.join(timeout=2.0)
            self.nvml.nvmlShutdown()
        elif self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            bits = {v: k for k, v in self.REASONS.items()}
            for line in self.lines:
                parts = [x.strip() for x in line.split(",")]
                try:
                    self.sm_max = float(parts[1])
                    rs = sum(bits[n] for n, v in zip(names, parts[3:7]) if v.lower() == "active")
                    self.samples.append((float(parts[0]), float(parts[2]), rs))
                except (ValueError, IndexError):
                    continue
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"], "samples": 0}
        sm = [x[0] for x in self.samples]
        reasons = sorted({name for _, _, rs in self.samples for bit, name in self.REASONS.items() if rs & bit})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.sm_max, "reasons": reasons,
                "samples": len(sm), "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": round(max(x[1] for x in self.samples), 1) if self.samples else None,
                "source": "nvml" if self.nvml is not None else f"nvidia-smi ({self.nvml_error})"}


# --------------------------------------------------------------- workloads --

def make_workload(name):
    from fine_grained_fp8_weight_b300 import workloads as wl
    if name == "prefill":
        return wl.prefill_pair()
    if name == "decode":
        return wl.decode()
    if name == "moe":
        return wl.moe_grouped()
    if name == "wgrad":
        return wl.wgrad()
    if name == "dgrad":
        return wl.dgrad()
    if name == "moe_decode":
        return wl.moe_decode()
    if name == "tiny":
        return wl.tiny()
    raise SystemExit(f"unknown workload {name}")


def gemm_flops(g):
    from fine_grained_fp8_weight_b300.workloads import Dense, Dgrad, Grouped, Masked, Wgrad
    if isinstance(g, Masked):
        return 2.0 * float(g.counts.sum()) * g.B.shape[1] * g.A.shape[2]
    if isinstance(g, Dense):
        return 2.0 * g.A.shape[0] * g.B.shape[0] * g.A.shape[1]
    if isinstance(g, Dgrad):
        return 2.0 * g.dY.shape[0] * g.W.shape[1] * g.dY.shape[1]
    if isinstance(g, Grouped):
        return 2.0 * float(g.counts.sum()) * g.B.shape[1] * g.A.shape[1]
    if isinstance(g, Wgrad):
        return 2.0 * g.dY.shape[1] * g.X.shape[1] * g.dY.shape[0]
    raise TypeError(g)


def gemm_bytes(g):
    """Algorithmic DRAM bytes of one GEMM launch: E4M3 operands, FP32 scales, output."""
    from fine_grained_fp8_weight_b300.workloads import Dense, Dgrad, Grouped, Masked, Wgrad
    if isinstance(g, Masked):
        E, cap, K = g.A.shape
        N = g.B.shape[1]
        live = int((g.counts > 0).sum())      # idle experts' weights are not read
        return (int(g.counts.sum()) * K + live * N * K + 4 * (E * cap * K // 128 + live * ((N + 127) // 128) * (K // 128))
                + 2 * int(g.counts.sum()) * N)
    if isinstance(g, Dense):
        M, K = g.A.shape
        N = g.B.shape[0]
        return M * K + N * K + 4 * (M * K // 128 + ((N + 127) // 128) * (K // 128)) + 2 * M * N
    if isinstance(g, Dgrad):
        T, N = g.dY.shape
        K = g.W.shape[1]
        return T * N + K * N + 4 * (T * N // 128 + (N // 128) * (K // 128)) + 2 * T * K
    if isinstance(g, Grouped):
        M, K = g.A.shape
        E, N, _ = g.B.shape
        return M * K + E * N * K + 4 * (M * K // 128 + E * ((N + 127) // 128) * (K // 128)) + 2 * M * N
    if isinstance(g, Wgrad):
        T, N = g.dY.shape
        K = g.X.shape[1]
        return T * N + T * K + 4 * (T // 128) * (N + K) + 4 * N * K
    raise TypeError(g)


def max_over_ranks(ms_total, dist=None, device=None):
    """The job's time: the slowest rank's (replicas run the same step on their
    own data; `value` is all ranks' work over this time)."""
    if dist is None:
        return ms_total
    import torch
    t = torch.tensor([ms_total], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step, world, ms_step):
    """Whole-job throughput: every rank's FLOPs of one step over the step time."""
    return flops_per_rank_step * world / (ms_step * 1e-3) / 1e12


class DevicePath:
    """The step on device buffers: every op is one C-ABI call on one stream."""

    def __init__(self, work, dev, fused_a=False, least_workspace=False):
        import torch
        import fine_grained_fp8_weight_b300 as fg
        from fine_grained_fp8_weight_b300 import workloads as wl
        from fine_grained_fp8_weight_b300.workloads import Dense, Dgrad, Grouped, Masked, Wgrad
        self.fg, self.torch, self.dev = fg, torch, dev
        self.ops = []          # (kind, name, callable, bytes or flops)
        self.workspaces = []   # GEMM workspaces allocated here (the rest are the library's cached ones)
        self.kernel_of = {}    # GEMM op name -> the kernel that runs it

        def gemm_ws(M, N, K):
            # None: the library's recommended workspace (every schedule); else a
            # workspace of the least accepted size (whole output tiles only)
            if not least_workspace:
                return None
            ws = torch.zeros(max(fg.lib().fgf8_gemm_workspace_min_bytes(M, N, K, 1), 4096), dtype=torch.uint8,
                             device=dev)
            self.workspaces.append(ws)
            return ws

        def dense_kernel(M, N, K, bkind=0):
            sch = fg.fgf8_testing_gemm_schedule(M, N, K, bkind)
            return "gemm_smallm_kernel" if sch["small_m"] else "gemm_blockscaled_kernel"

        self.inputs = []       # (host numpy bits, device tensor) for the end-to-end leg
        self.outputs = []
        self.groups = []       # per GEMM: (its input indices, its op indices, its output index)
        for g in work.gemms:
            n_in, n_ops = len(self.inputs), len(self.ops)
            if isinstance(g, Dense):
                A = wl.bf16_bits_to_torch(g.A).to(dev)
                B = wl.bf16_bits_to_torch(g.B).to(dev)
                self.inputs += [(g.A, A), (g.B, B)]
                M, K = A.shape
                N = B.shape[0]
                st = {}
                C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                self.outputs.append(C)
                qbytes = lambda r, c, sc: r * c * 3 + sc * 4
                self.kernel_of[f"{g.name}.gemm"] = dense_kernel(M, N, K)
                if fused_a and M <= FUSED_A_MAX_M:
                    # tokens quantized inside the GEMM: no activation-quantize launch
                    self.ops.append(("quant", f"{g.name}.quant_w_128x128",
                                     lambda B=B, st=st: st.update(b=fg.fp8_quant_w_128x128(B)),
                                     qbytes(N, K, (N // 128 + 1) * K // 128)))
                    self.ops.append(("gemm", f"{g.name}.gemm",
                                     lambda A=A, st=st, C=C: fg.fp8_gemm_bf16a_blockscaled(A, st["b"][0], st["b"][1],
                                                                                          out=C),
                                     gemm_flops(g)))
                else:
                    self.ops.append(("quant", f"{g.name}.quant_act_1x128",
                                     lambda A=A, st=st: st.update(a=fg.fp8_quant_act_1x128(A)),
                                     qbytes(M, K, M * K // 128)))
                    self.ops.append(("quant", f"{g.name}.quant_w_128x128",
                                     lambda B=B, st=st: st.update(b=fg.fp8_quant_w_128x128(B)),
                                     qbytes(N, K, (N // 128 + 1) * K // 128)))
                    self.ops.append(("gemm", f"{g.name}.gemm",
                                     lambda st=st, C=C, ws=gemm_ws(M, N, K): fg.fp8_gemm_blockscaled(
                                         st["a"][0], st["a"][1], st["b"][0], st["b"][1], out=C, workspace=ws),
                                     gemm_flops(g)))
            elif isinstance(g, Grouped):
                A = wl.bf16_bits_to_torch(g.A).to(dev)
                B = wl.bf16_bits_to_torch(g.B).to(dev)
                mi = torch.from_numpy(g.m_indices).to(dev)
                self.inputs += [(g.A, A), (g.B, B)]
                M, K = A.shape
                E, N, _ = B.shape
                st = {}
                C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                self.outputs.append(C)
                self.ops.append(("quant", f"{g.name}.quant_act_1x128",
                                 lambda A=A, st=st: st.update(a=fg.fp8_quant_act_1x128(A)), M * K * 3 + M * K // 32))
                self.ops.append(("quant", f"{g.name}.quant_w_128x128_grouped",
                                 lambda B=B, st=st: st.update(b=fg.fp8_quant_w_128x128_grouped(B)), E * N * K * 3))
                self.kernel_of[f"{g.name}.grouped_gemm"] = "gemm_blockscaled_kernel (grouped)"
                self.ops.append(("gemm", f"{g.name}.grouped_gemm",
                                 lambda st=st, C=C, mi=mi: fg.fp8_grouped_gemm_blockscaled(
                                     st["a"][0], st["a"][1], st["b"][0], st["b"][1], mi, out=C),
                                 gemm_flops(g)))
            elif isinstance(g, Masked):
                E, cap, K = g.A.shape
                N = g.B.shape[1]
                A = wl.bf16_bits_to_torch(g.A.reshape(E * cap, K)).to(dev)
                B = wl.bf16_bits_to_torch(g.B).to(dev)
                cnt = torch.from_numpy(g.counts).to(dev)
                self.inputs += [(g.A.reshape(E * cap, K), A), (g.B, B)]
                st = {}
                C = torch.empty((E, cap, N), dtype=torch.bfloat16, device=dev)
                self.outputs.append(C)
                self.ops.append(("quant", f"{g.name}.quant_act_1x128",
                                 lambda A=A, st=st: st.update(a=fg.fp8_quant_act_1x128(A)),
                                 E * cap * K * 3 + E * cap * K // 32))
                self.ops.append(("quant", f"{g.name}.quant_w_128x128_grouped",
                                 lambda B=B, st=st: st.update(b=fg.fp8_quant_w_128x128_grouped(B)), E * N * K * 3))
                self.kernel_of[f"{g.name}.gemm"] = "gemm_smallm_kernel (masked)"
                self.ops.append(("gemm", f"{g.name}.gemm",
                                 lambda st=st, C=C, cnt=cnt, E=E, cap=cap, K=K: fg.fp8_masked_grouped_gemm_blockscaled(
                                     st["a"][0].view(E, cap, K), st["a"][1], st["b"][0], st["b"][1], cnt, out=C),
                                 gemm_flops(g)))
            elif isinstance(g, Dgrad):
                dY = wl.bf16_bits_to_torch(g.dY).to(dev)
                W = wl.bf16_bits_to_torch(g.W).to(dev)
                self.inputs += [(g.dY, dY), (g.W, W)]
                T, N = dY.shape
                K = W.shape[1]
                st = {}
                C = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
                self.outputs.append(C)
                self.ops.append(("quant", f"{g.name}.quant_dY_1x128",
                                 lambda dY=dY, st=st: st.update(a=fg.fp8_quant_act_1x128(dY)),
                                 T * N * 3 + T * N // 32))
                self.ops.append(("quant", f"{g.name}.quant_wT_128x128",
                                 lambda W=W, st=st: st.update(b=fg.fp8_quant_w_128x128_t(W)),
                                 N * K * 3 + (N // 128) * (K // 128) * 4))
                self.kernel_of[f"{g.name}.gemm"] = dense_kernel(T, K, N)
                self.ops.append(("gemm", f"{g.name}.gemm",
                                 lambda st=st, C=C, ws=gemm_ws(T, K, N): fg.fp8_gemm_blockscaled(
                                     st["a"][0], st["a"][1], st["b"][0], st["b"][1], out=C, workspace=ws),
                                 gemm_flops(g)))
            elif isinstance(g, Wgrad):
                dY = wl.bf16_bits_to_torch(g.dY).to(dev)
                X = wl.bf16_bits_to_torch(g.X).to(dev)
                self.inputs += [(g.dY, dY), (g.X, X)]
                T, N = dY.shape
                K = X.shape[1]
                st = {}
                C = torch.empty((N, K), dtype=torch.float32, device=dev)
                self.outputs.append(C)
                self.ops.append(("quant", f"{g.name}.quant_dY_128x1",
                                 lambda dY=dY, st=st: st.update(a=fg.fp8_quant_act_1x128(dY, rows=False, transposed=True)),
                                 T * N * 3 + T * N // 32))
                self.ops.append(("quant", f"{g.name}.quant_X_128x1",
                                 lambda X=X, st=st: st.update(b=fg.fp8_quant_act_1x128(X, rows=False, transposed=True)),
                                 T * K * 3 + T * K // 32))
                self.kernel_of[f"{g.name}.gemm"] = "gemm_blockscaled_kernel (per-row B scales)"
                self.ops.append(("gemm", f"{g.name}.gemm",
                                 lambda st=st, C=C, ws=gemm_ws(N, K, T): fg.fp8_gemm_blockscaled(
                                     st["a"][2], st["a"][3], st["b"][2], st["b"][3], bkind=fg.BSCALE_ROW1x128,
                                     out=C, workspace=ws),
                                 gemm_flops(g)))
            self.groups.append((list(range(n_in, len(self.inputs))), list(range(n_ops, len(self.ops))),
                                len(self.outputs) - 1))
        self.gemm_flops = sum(w for k, _, _, w in self.ops if k == "gemm")
        self.gemm_bytes = {f"{g.name}.{'grouped_gemm' if isinstance(g, Grouped) else 'gemm'}": gemm_bytes(g)
                           for g in work.gemms}

    def step(self, events=None):
        for i, (_, _, fn, _) in enumerate(self.ops):
            if events is not None:
                events[i][0].record()
            fn()
            if events is not None:
                events[i][1].record()


# -------------------------------------------------------------------- main --

def run_device(args, rank, world, local_rank):
    import torch
    import fine_grained_fp8_weight_b300 as fg  # noqa: F401  (fails loudly if the library is missing)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    work = make_workload(args.workload)
    path = DevicePath(work, dev, fused_a=args.fused_a, least_workspace=args.workspace == "least")
    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_PER_BF16

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        path.step()
    barrier()

    # The step is captured once into a CUDA graph and replayed, so that host
    # launch overhead does not enter the device-timed region.
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        path.step()                                  # allocations settle outside the capture
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(step_graph, stream=stream):
            path.step()
    torch.cuda.current_stream(dev).wait_stream(stream)
    for _ in range(args.warmup):
        step_graph.replay()
    barrier()

    # Each kernel timed alone (its own graph, L2 flushed between replays)
    # before the long step loop, which on a 1.1 kW part can run into the
    # power cap and lower the clocks that follow it.
    per_op = time_ops(path, dev, stream, max(3, min(args.op_reps, args.steps)), fp8_peak, peaks)
    barrier()

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    clocks.start()
    barrier()
    t0.record()
    for _ in range(args.steps):
        step_graph.replay()
    t1.record()
    barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1), dist, dev)
    ms_step = ms_total / args.steps

    n_ops = len(path.ops)
    value = job_tflops(path.gemm_flops, world, ms_step)
    version = fg.lib().fgf8_version().decode()
    roof = roofline_of(path, per_op, work.name, fp8_peak, peaks, version)
    q_bytes = sum(w for k, _, _, w in path.ops if k == "quant")
    q_ms = sum(e["ms"] for e in per_op.values() if e["kind"] == "quant")
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate)",
        "data": "synthetic (seeded numpy normals, bf16)",
        "config": {"workload": work.name,
                   "gemms": [n for k, n, _, _ in path.ops if k == "gemm"],
                   "l2": "no flush: each step reads inputs larger than the 126 MB L2",
                   "gemm_workspace": args.workspace,
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "quantize": {"GB/s": round(q_bytes / (q_ms * 1e-3) / 1e9, 1), "peak_hbm_gbs": peaks["hbm_gbs"],
                     "frac": round(q_bytes / (q_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
        "kernels": per_op,
        "clocks": clk,
        "gpu_launches": n_ops * args.steps,
    }
    if not args.no_e2e:
        result["e2e"] = run_e2e(path, args, torch)
    problems = device_status(fg, path)
    del path
    if rank == 0 and not args.no_workloads:
        result["workloads"] = run_workloads(args, dev, stream, fp8_peak, peaks, version)
        problems += device_status(fg, None)
    if problems:
        # a device-side wait expired somewhere: the kernels that gave up ran
        # short, so no throughput of this run is reported
        result["value"] = None
        result["error"] = "device-side wait expired: " + "; ".join(problems)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(work, args)
    if dist is not None:
        dist.destroy_process_group()
    return result


class L2Flush:
    """Untimed L2 flush between replays: a write of a buffer twice the 126 MB
    L2, so that no op finds inputs left in L2 by its previous replay, then a
    read of a second such buffer, so that the L2 holds clean lines and the
    timed op does not pay for writing the first buffer's dirty lines back to
    HBM (2 us of a 20 us quantization otherwise)."""

    def __init__(self, torch, dev):
        n = 2 * 126 * 2 ** 20 // 4 + 2 ** 20
        self.dirty = torch.empty(n, dtype=torch.float32, device=dev)
        self.clean = torch.ones(n, dtype=torch.float32, device=dev)

    def __call__(self):
        self.dirty.fill_(1.0)
        self.clean.sum()


def time_ops(path, dev, stream, reps, fp8_peak, peaks):
    """Per-kernel device time: each op captured alone into a CUDA graph and
    replayed, one event pair per replay (the median is reported), with an
    untimed L2 flush (L2Flush) in between.  A short device-side sleep before
    the first event keeps the GPU busy while the host submits the event and
    the replay, so the interval holds the op alone and not the host's
    submission latency."""
    import torch
    flush = L2Flush(torch, dev)
    per_op = {}
    for kind, name, fn, work_units in path.ops:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(g, stream=stream):
                fn()
        torch.cuda.current_stream(dev).wait_stream(stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        g.replay()
        for e0, e1 in ev:
            flush()
            torch.cuda._sleep(SLEEP_CYCLES)
            e0.record()
            g.replay()
            e1.record()
        torch.cuda.synchronize(dev)
        avg = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
        entry = {"kind": kind, "ms": round(avg, 4), "timing": f"median of {reps} replays"}
        if kind == "gemm":
            entry["TFLOP/s"] = round(work_units / (avg * 1e-3) / 1e12, 1)
            entry["frac_fp8_peak"] = round(entry["TFLOP/s"] / fp8_peak, 4)
            entry["GB/s"] = round(path.gemm_bytes[name] / (avg * 1e-3) / 1e9, 1)
            entry["frac_hbm"] = round(entry["GB/s"] / peaks["hbm_gbs"], 4)
        else:
            entry["GB/s"] = round(work_units / (avg * 1e-3) / 1e9, 1)
            entry["frac_hbm"] = round(entry["GB/s"] / peaks["hbm_gbs"], 4)
        per_op[name] = entry
    return per_op


def time_ops_rotating(paths, dev, stream, reps, fp8_peak, peaks):
    """Per-kernel device time for workloads whose operands fit in L2: the
    same op of len(paths) independent copies of the workload (their operand
    sets together larger than twice the 126 MB L2) captured back to back,
    ROTATE_ROUNDS times over, into one CUDA graph, so that no launch finds its
    inputs in L2 and the start of a replay is spread over many kernels; the L2
    is flushed before each timed replay.  Reports the mean time per launch."""
    import torch
    flush = L2Flush(torch, dev)
    R = len(paths)
    per_op = {}
    for j, (kind, name, _, work_units) in enumerate(paths[0].ops):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for pth in paths:
                pth.ops[j][2]()
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(g, stream=stream):
                for _ in range(ROTATE_ROUNDS):
                    for pth in paths:
                        pth.ops[j][2]()
        torch.cuda.current_stream(dev).wait_stream(stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        g.replay()
        for e0, e1 in ev:
            flush()
            torch.cuda._sleep(SLEEP_CYCLES)
            e0.record()
            g.replay()
            e1.record()
        torch.cuda.synchronize(dev)
        avg = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev) / (R * ROTATE_ROUNDS)
        entry = {"kind": kind, "ms": round(avg, 5),
                 "timing": f"median of {reps} replays of {R * ROTATE_ROUNDS} back-to-back launches on {R} "
                           f"separate operand copies"}
        if kind == "gemm":
            entry["TFLOP/s"] = round(work_units / (avg * 1e-3) / 1e12, 1)
            entry["frac_fp8_peak"] = round(entry["TFLOP/s"] / fp8_peak, 4)
            entry["GB/s"] = round(paths[0].gemm_bytes[name] / (avg * 1e-3) / 1e9, 1)
            entry["frac_hbm"] = round(entry["GB/s"] / peaks["hbm_gbs"], 4)
        else:
            entry["GB/s"] = round(work_units / (avg * 1e-3) / 1e9, 1)
            entry["frac_hbm"] = round(entry["GB/s"] / peaks["hbm_gbs"], 4)
        per_op[name] = entry
    return per_op


def roofline_of(path, per_op, work_name, fp8_peak, peaks, version):
    """Roofline of the dominant kernel: the GEMM launch that takes longest.
    Below the ridge point (peak FLOP/s over peak bytes/s) a launch is bound by
    HBM, above it by the FP8 tensor rate."""
    gemm_ops = [(per_op[name]["ms"], name, w) for kind, name, _, w in path.ops if kind == "gemm"]
    dom_ms, dom_name, dom_flops = max(gemm_ops)
    dom_bytes = path.gemm_bytes[dom_name]
    hbm_bound = dom_flops / dom_bytes < fp8_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    traffic = MEASURED_TRAFFIC.get(version, {}).get(f"{work_name}/{dom_name}")
    kernel = path.kernel_of.get(dom_name, "gemm_blockscaled_kernel")
    if hbm_bound:
        return {"bound": "hbm", "achieved": per_op[dom_name]["GB/s"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": per_op[dom_name]["frac_hbm"], "traffic": traffic,
                "kernel": f"{kernel} ({dom_name}, {version})", "algorithmic_bytes_per_launch": dom_bytes,
                "peak_note": f"{peaks['source']} HBM copy bandwidth"}
    ach = dom_flops / (dom_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(ach, 1), "peak": round(fp8_peak, 1),
            "unit": "TFLOP/s", "frac": round(ach / fp8_peak, 4), "traffic": traffic,
            "kernel": f"{kernel} ({dom_name}, {version})", "algorithmic_flops_per_launch": dom_flops,
            "peak_note": f"fp8 = {FP8_PER_BF16:g} x {peaks['source']} bf16 burst "
                         f"{peaks['bf16_tflops']} TFLOP/s (sustained bf16 {peaks['bf16_tflops_sustained']})"}


def device_status(fg, path):
    """Read (and clear) the device status word of every GEMM workspace the run
    used: the library's cached workspaces and any the path allocated itself.
    Returns the problems found (an expired device-side wait), if any."""
    wss = list(fg._workspaces.values()) + (list(path.workspaces) if path is not None else [])
    problems = []
    for ws in wss:
        st, site = fg.fgf8_read_status(ws)
        if st != 0:
            problems.append(f"status {st} at wait site {site}")
    return problems


# Workloads measured in the line's "workloads" key besides the headline one:
# the other configurations of the path (tiny GEMM, decode GEMMs, grouped MoE,
# weight gradient) and the data gradient.
EXTRA_WORKLOADS = ["tiny", "decode", "moe", "wgrad", "dgrad"]
# Workloads whose GEMMs each take less BF16 input than this (the decode and
# tiny GEMMs, whose operands would otherwise come from L2) are timed on
# ROTATE_COPIES copies back to back (time_ops_rotating); 8 copies of the decode
# workload's operands take ~2.8 GB, far more than twice L2.
ROTATE_BELOW_BYTES = 126 << 20
ROTATE_COPIES = 8
ROTATE_ROUNDS = 4
# A device-side sleep before each timed replay (about 1 ms at 2 GHz) keeps the
# GPU busy while the host submits the event and the replay, so that the timed
# interval holds the kernels alone and not the submission of the graph.
SLEEP_CYCLES = 2_000_000


def run_workloads(args, dev, stream, fp8_peak, peaks, version):
    """Per-kernel device times, throughput and roofline fractions of every
    workload in EXTRA_WORKLOADS (and the decode GEMMs with the tokens quantized
    inside the GEMM, for comparison), each op replayed with an L2 flush in
    between."""
    import torch
    out = {}
    names = [w for w in EXTRA_WORKLOADS if w != args.workload] + ["decode:fused_a"]
    if args.moe_decode:
        names.append("moe_decode")
    reps = max(3, min(args.op_reps, 20))
    for name in names:
        base, _, variant = name.partition(":")
        work = make_workload(base)
        path = DevicePath(work, dev, fused_a=variant == "fused_a")
        with torch.cuda.stream(stream):
            path.step()
        torch.cuda.synchronize(dev)
        footprint = max(sum(path.inputs[i][1].numel() * path.inputs[i][1].element_size() for i in ins)
                        for ins, _, _ in path.groups)
        if footprint < ROTATE_BELOW_BYTES:
            # operands that fit in L2: copies of the workload timed back to back
            copies = [path] + [DevicePath(work, dev, fused_a=variant == "fused_a") for _ in range(ROTATE_COPIES - 1)]
            with torch.cuda.stream(stream):
                for pth in copies[1:]:
                    pth.step()
            torch.cuda.synchronize(dev)
            per_op = time_ops_rotating(copies, dev, stream, reps, fp8_peak, peaks)
            del copies
        else:
            per_op = time_ops(path, dev, stream, reps, fp8_peak, peaks)
        key = work.name + (" (tokens quantized in the GEMM)" if variant else "")
        gflop = path.gemm_flops / 1e9
        ms = sum(e["ms"] for e in per_op.values())
        out[key] = {"kernels": per_op, "ms_sum_of_kernels": round(ms, 4),
                    "gemm_GFLOP": round(gflop, 3), "TFLOP/s_over_kernels": round(gflop / ms, 1),
                    "roofline": roofline_of(path, per_op, work.name, fp8_peak, peaks, version)}
        if not args.no_cpu_baseline and not variant:
            out[key]["oracle"] = workload_oracle(work, args)
        del path, work
        torch.cuda.empty_cache()
    return out


def run_e2e(path, args, torch):
    """Same metric through the public API from pinned host memory: every step
    copies its BF16 inputs host->device, runs the path, and reads the outputs
    back (device->host), all inside the timed region.  Host-to-device copies,
    compute and device-to-host copies run on three streams, ordered by
    events only where data flows: a GEMM's quantize and GEMM calls wait for
    its own inputs; its output goes back as soon as it has finished; the next
    step's copy into an input buffer waits until this step's calls that read
    it are done, and its GEMM into an output buffer until the previous read-
    back of it is.  So one GEMM's copies overlap another's compute, copies in
    the two directions overlap each other (PCIe is full duplex), and
    consecutive steps overlap; the timed region ends when every copy of the
    last step has landed in host memory."""
    from fine_grained_fp8_weight_b300 import workloads as wl
    dev = path.dev
    host_in = [wl.bf16_bits_to_torch(bits).pin_memory() for bits, _ in path.inputs]
    host_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in path.outputs]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    main = torch.cuda.current_stream(dev)
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    ngroups = len(path.groups)
    computed = [None] * ngroups                 # per GEMM group: its calls of the previous step done
    read_back = [None] * ngroups                # per GEMM group: its output's previous read-back done

    def e2e_step():
        arrived = []
        with torch.cuda.stream(up):
            for g, (ins, _, _) in enumerate(path.groups):
                if computed[g] is not None:
                    up.wait_event(computed[g])
                for i in ins:
                    path.inputs[i][1].copy_(host_in[i], non_blocking=True)
                arrived.append(torch.cuda.Event())
                arrived[-1].record(up)
        for g, (ins, ops, _) in enumerate(path.groups):
            main.wait_event(arrived[g])
            if read_back[g] is not None:
                main.wait_event(read_back[g])
            for j in ops:
                path.ops[j][2]()
            computed[g] = torch.cuda.Event()
            computed[g].record(main)
        with torch.cuda.stream(down):
            for g, (_, _, o) in enumerate(path.groups):
                down.wait_event(computed[g])
                host_out[o].copy_(path.outputs[o], non_blocking=True)
                read_back[g] = torch.cuda.Event()
                read_back[g].record(down)

    def drain():
        for st in (up, main, down):
            st.synchronize()

    steps = max(1, min(args.steps, 5))
    e2e_step()
    drain()
    t = time.perf_counter()
    for _ in range(steps):
        e2e_step()
    drain()
    dt = (time.perf_counter() - t) / steps
    return {"value": round(path.gemm_flops / dt / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(dt * 1e3, 3),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "note": "host-to-device, compute and device-to-host on three streams, ordered by data dependences; "
                    "copies overlap compute, each other and the neighbouring steps"}


def _quant_slices(pool, fn, x, threads, axis):
    """fn over slices of x along `axis` (multiples of 128 rows or columns), in
    parallel; returns the list of (codes, scales) per slice and the slices."""
    n = x.shape[axis]
    step = 128 * max(1, (n // 128) // (4 * threads))
    cuts = [(c, min(n, c + step)) for c in range(0, n, step)]
    take = (lambda c: np.ascontiguousarray(x[c[0]:c[1]])) if axis == 0 else (
        lambda c: np.ascontiguousarray(x[:, c[0]:c[1]]))
    return list(pool.map(lambda c: fn(take(c)), cuts)), cuts


def oracle_sample(work, rows, threads, seed=0):
    """The oracle as it stands (plain C in binary64, called through ctypes,
    which releases the GIL, so `threads` host threads run it side by side) on
    each GEMM of the workload: every operand quantized in full (in slices of
    128 rows or columns spread over the threads) as the device path quantizes
    it (A 1x128 and B 128x128; W^T for dgrad; both operands 128x1 along the
    tokens for wgrad; per expert for the grouped and masked layouts), and
    `rows` seeded output rows against all N columns (grouped: a quarter of
    that, at least one, of every expert with tokens; masked: that many rows
    of every live expert),
    the rows split over the threads.  Returns (GEMM FLOPs of the sample,
    measured seconds, seconds of the whole workload extrapolated from it: the
    GEMM part scaled by the real output rows / the sampled rows)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    from fine_grained_fp8_weight_b300.workloads import Dense, Dgrad, Grouped, Masked, Wgrad
    oracle.lib()                                 # built and loaded before the threads start
    flops = secs = full = 0.0
    rng = np.random.default_rng(seed)

    def quant_rows(pool, fn, x, axis=0):
        # fn over 128-row (axis 0) or 128-column (axis 1) slices; codes and scales reassembled
        parts, cuts = _quant_slices(pool, fn, x, threads, axis)
        return parts, cuts

    def act_1x128(pool, A):
        M, K = A.shape
        parts, cuts = quant_rows(pool, oracle.quant_act_1x128, A)
        sa = np.zeros((K // 128, (M + 3) // 4 * 4), np.float32)
        for (r0, r1), (_, s_) in zip(cuts, parts):
            sa[:, r0:r1] = s_[:, :r1 - r0]
        return np.concatenate([q for q, _ in parts]), sa

    def w_128x128(pool, Bw):
        N, K = Bw.shape
        parts, cuts = quant_rows(pool, oracle.quant_w_128x128, Bw)
        sb = np.zeros((K // 128, ((N + 127) // 128 + 3) // 4 * 4), np.float32)
        for (b0, b1), (_, s_) in zip(cuts, parts):
            sb[:, b0 // 128:(b1 + 127) // 128] = s_[:, :(b1 - b0 + 127) // 128]
        return np.concatenate([q for q, _ in parts]), sb

    def act_128x1(pool, X):
        # transposed output of 128x1 tiles along the tokens: qT [K, T], per-row
        # scales of qT as the GEMM reads them, sb[t/128][k]
        T, K = X.shape
        parts, cuts = quant_rows(pool, oracle.quant_act_128x1, X)
        qT = np.concatenate([q for q, _ in parts], axis=1)
        sT = np.concatenate([s_ for _, s_ in parts], axis=0)
        return qT, np.ascontiguousarray(sT[:, :(K + 3) // 4 * 4])

    with ThreadPoolExecutor(max_workers=threads) as pool:
        for g in work.gemms:
            t0 = time.perf_counter()
            if isinstance(g, (Dense, Dgrad)):
                A = g.A if isinstance(g, Dense) else g.dY
                qa, sa = act_1x128(pool, A)
                if isinstance(g, Dense):
                    qb, sb = w_128x128(pool, g.B)
                else:                            # B = W^T: slices of W's columns are rows of W^T
                    Bw = g.W
                    N = Bw.shape[1]
                    parts, cuts = quant_rows(pool, oracle.quant_w_128x128_t, Bw, axis=1)
                    sb = np.zeros((A.shape[1] // 128, (N // 128 + 3) // 4 * 4), np.float32)
                    for (c0, c1), (_, s_) in zip(cuts, parts):
                        sb[:, c0 // 128:c1 // 128] = s_[:, :(c1 - c0) // 128]
                    qb = np.concatenate([q for q, _ in parts])
                t1 = time.perf_counter()
                M, K = qa.shape
                N = qb.shape[0]
                r = np.sort(rng.choice(M, size=min(rows, M), replace=False))
                chunks = [c for c in np.array_split(r, threads) if len(c)]
                list(pool.map(lambda c: oracle.gemm_blockscaled(qa, sa, qb, sb, 0, rows=c), chunks))
                real_rows = M
            elif isinstance(g, Wgrad):
                qa, sa = act_128x1(pool, g.dY)   # dY^T [N, T], scales per (token group, row)
                qb, sb = act_128x1(pool, g.X)    # X^T [K, T]
                t1 = time.perf_counter()
                M, K = qa.shape
                N = qb.shape[0]
                r = np.sort(rng.choice(M, size=min(rows, M), replace=False))
                chunks = [c for c in np.array_split(r, threads) if len(c)]
                list(pool.map(lambda c: oracle.gemm_blockscaled(qa, sa, qb, sb, 1, rows=c), chunks))
                real_rows = M
            elif isinstance(g, Grouped):
                qa, sa = act_1x128(pool, g.A)
                E, N, K = g.B.shape
                qs = list(pool.map(oracle.quant_w_128x128, [g.B[e] for e in range(E)]))
                qb = np.stack([q for q, _ in qs])
                sb = np.stack([s_ for _, s_ in qs])
                t1 = time.perf_counter()
                starts = np.concatenate([[0], np.cumsum((g.counts + 127) // 128 * 128)])
                per_e = max(1, rows // 4)        # 32 experts: a quarter of the rows each
                r = np.sort(np.concatenate([starts[e] + rng.choice(int(g.counts[e]), size=min(per_e, int(g.counts[e])),
                                                                   replace=False)
                                            for e in range(E) if g.counts[e] > 0]))
                chunks = [c for c in np.array_split(r, threads) if len(c)]
                list(pool.map(lambda c: oracle.grouped_gemm_blockscaled(qa, sa, qb, sb, g.m_indices, rows=c), chunks))
                real_rows = int(g.counts.sum())
            elif isinstance(g, Masked):
                E, cap, K = g.A.shape
                qa, sa = act_1x128(pool, g.A.reshape(E * cap, K))
                N = g.B.shape[1]
                live = [e for e in range(E) if g.counts[e] > 0]
                qs = dict(zip(live, pool.map(oracle.quant_w_128x128, [g.B[e] for e in live])))
                t1 = time.perf_counter()
                jobs = [(e, np.sort(rng.choice(int(g.counts[e]), size=min(rows, int(g.counts[e])), replace=False)))
                        for e in live]
                list(pool.map(lambda j: oracle.gemm_blockscaled(
                    qa[j[0] * cap:j[0] * cap + int(g.counts[j[0]])],
                    np.ascontiguousarray(sa[:, j[0] * cap:(j[0] + 1) * cap]), qs[j[0]][0], qs[j[0]][1], 0,
                    rows=j[1]), jobs))
                r = np.concatenate([j[1] for j in jobs])
                real_rows = int(g.counts.sum())
            else:
                continue
            t2 = time.perf_counter()
            flops += 2.0 * len(r) * N * K
            secs += t2 - t0
            full += (t1 - t0) + (t2 - t1) * (real_rows / len(r))
    return flops, secs, full


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(work, args):
    """The oracle on the host cores: the reference arm's per-step sample
    (every operand of the step quantized in full, args.cpu_rows seeded rows of
    each GEMM against all N) run args.cpu_reps times with different rows."""
    threads = _cores()
    flops = dt = full = 0.0
    for rep in range(args.cpu_reps):
        f, d, fu = oracle_sample(work, args.cpu_rows, threads, seed=rep)
        flops, dt, full = flops + f, dt + d, full + fu
    return {"value": round(flops / dt / 1e12, 9), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "seconds": round(dt, 2), "full_step_seconds_extrapolated": round(full / args.cpu_reps, 1),
            "sample": f"{args.cpu_reps} x (every operand of the step quantized in full -- A 1x128, B 128x128 -- and "
                      f"{args.cpu_rows} seeded rows of each GEMM's output against all N in binary64); plain C "
                      f"oracle on {threads} host threads; the full step's time is extrapolated from it "
                      f"(GEMM part x M/rows)"}


def workload_oracle(work, args):
    """The oracle on the host cores for one workload of the workloads key:
    one sample (every operand quantized in full, args.cpu_rows seeded output
    rows of each GEMM -- of each expert for the grouped layouts -- against all
    N), its measured seconds and the workload's time extrapolated from it."""
    threads = _cores()
    f, d, fu = oracle_sample(work, args.cpu_rows, threads, seed=7)
    return {"GFLOP/s": round(f / d / 1e9, 4), "seconds": round(d, 2), "cores": threads, "kind": "oracle",
            "workload_seconds_extrapolated": round(fu, 1),
            "sample": f"every operand quantized in full and {args.cpu_rows} seeded output rows of each GEMM "
                      f"(per live expert for the masked layout, {max(1, args.cpu_rows // 4)} per expert for the "
                      f"grouped one) against all N, binary64, {threads} host threads"}


def run_reference(args, rank, world):
    """The reference arm is the oracle, run on the host cores on a bounded
    sample of the same workload each step, the sample cpu_baseline repeats
    (every operand of the step quantized in full, args.cpu_rows seeded rows of
    each GEMM against all N); rank 0 alone runs it."""
    if rank != 0:
        return None
    work = make_workload(args.workload)
    threads = _cores()
    for i in range(args.warmup):
        oracle_sample(work, args.cpu_rows, threads, seed=1000 + i)
    flops = secs = 0.0
    for i in range(args.steps):
        f, dt, _ = oracle_sample(work, args.cpu_rows, threads, seed=i)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    sample = (f"per step: every operand of the step quantized in full (A 1x128, B 128x128) and {args.cpu_rows} "
              f"seeded rows of each GEMM's output against all N in binary64 (plain C oracle, {threads} host threads)")
    return {"metric": METRIC, "value": round(value, 9), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy normals, bf16)",
            "config": {"workload": work.name, "parallelism": f"host oracle, {threads} threads"}, "impl": "reference",
            "cpu_baseline": {"value": round(value, 9), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 9), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_gemm(args):
    """One warm-up and one timed launch of a single GEMM (for ncu captures)."""
    import torch
    import fine_grained_fp8_weight_b300 as fg
    from fine_grained_fp8_weight_b300 import workloads as wl
    dev = torch.device("cuda", 0)
    g = make_workload(args.workload).gemms[args.gemm_index]
    A = wl.bf16_bits_to_torch(g.A).to(dev)
    B = wl.bf16_bits_to_torch(g.B).to(dev)
    qa, sa, _, _ = fg.fp8_quant_act_1x128(A)
    qb, sb = fg.fp8_quant_w_128x128(B)
    C = torch.empty((A.shape[0], B.shape[0]), dtype=torch.bfloat16, device=dev)
    for _ in range(2):
        fg.fp8_gemm_blockscaled(qa, sa, qb, sb, out=C)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    fg.fp8_gemm_blockscaled(qa, sa, qb, sb, out=C)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    print(json.dumps({"gemm": g.name, "ms": ms, "TFLOP/s": gemm_flops(g) / (ms * 1e-3) / 1e12}))


def profile_op(args):
    """Run the workload's ops once, then the named op four more times (for ncu
    captures of a single kernel; `-k`/`-s`/`-c` select the launches)."""
    import torch
    dev = torch.device("cuda", 0)
    path = DevicePath(make_workload(args.workload), dev)
    ops = {name: fn for _, name, fn, _ in path.ops}
    if args.profile_op not in ops:
        raise SystemExit(f"unknown op {args.profile_op}; ops of this workload: {sorted(ops)}")
    path.step()
    for _ in range(4):
        ops[args.profile_op]()
    torch.cuda.synchronize()
    print(json.dumps({"profiled_op": args.profile_op, "workload": args.workload}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="prefill", choices=["prefill", "decode", "moe", "moe_decode", "wgrad", "dgrad",
                                                               "tiny"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=4, help="oracle sample: output rows per GEMM")
    ap.add_argument("--cpu-reps", type=int, default=3, help="oracle baseline: samples (different rows)")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other workloads' kernel times")
    ap.add_argument("--moe-decode", action="store_true", help="also time the masked-layout MoE decode GEMM")
    ap.add_argument("--op-reps", type=int, default=20)
    ap.add_argument("--profile-gemm", action="store_true")
    ap.add_argument("--gemm-index", type=int, default=0)
    ap.add_argument("--profile-op", default=None, help="run one op of the workload repeatedly (for ncu)")
    ap.add_argument("--workspace", default="full", choices=["full", "least"],
                    help="dense GEMM workspace: the recommended size (last-wave split allowed) or the least "
                         "accepted size (whole output tiles only)")
    ap.add_argument("--fused-a", action="store_true",
                    help="GEMMs with at most 256 tokens quantize their BF16 tokens inside the GEMM")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3 and not (args.profile_gemm or args.profile_op):
        print("note: fewer than 3 warm-up steps do not make a valid measurement", file=sys.stderr)
    if args.profile_gemm:
        profile_gemm(args)
        return
    if args.profile_op:
        profile_op(args)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_device(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
