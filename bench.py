#!/usr/bin/env python
"""Benchmark: adjoint-gradient tokens/sec per layer on one GB300, with the roofline of
the dominant kernel, an end-to-end number through the C ABI with host buffers, and
the fp64 CPU oracle timed beside it.

Headline workload: ssm4_p2048, the largest one that fits one GPU -- K = 4 residual
layers, P = 2048, N = 256, T = 131072, B = 1, bf16 GEMM operands and fp32 scans,
truncated adjoint with window Tbar = 8192.  One step = one pass of the whole path over
one batch: for every layer adj_rms_norm (k >= 2) and adj_fwd_scan, then adj_loss_mse,
then for every layer (top down) adj_bwd_trunc, adj_param_grad and adj_rms_norm_bwd
(k >= 2).  The timed steps replay a CUDA graph of one step; L2 is flushed (a 256 MB
write) before every timed step; ms_per_step is the median over the timed steps.

The other workloads (ssm1_1m at both windows, ssm8_p512, ssm1_p128 at both windows)
are measured the same way and reported under "workloads" as context lines.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs its own batch (independent sequences: weak scaling,
no collective on the data path); rank 0 prints one JSON line.
"""
import argparse
import glob
import hashlib
import json
import re
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = ("ssm4_p2048", 8192)
CONTEXT = (("ssm1_1m", 4096), ("ssm1_1m", None), ("ssm8_p512", 4096), ("ssm1_p128", None), ("ssm1_p128", 2048))
# the general selective layer (one layer), measured the same way
SEL_CONTEXT = (("sel1_p1024", 8192, 1), ("sel1_p1024", None, 1), ("sel1_p1024", None, 4))
METRIC = "adjoint-gradient tokens/sec per layer on 1 GB300; % of HBM/tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# CPU oracle samples (prefixes of one sequence of the headline workload): all cores on
# CPU_ALL_T tokens, one core on CPU_ONE_T tokens; the reference arm runs CPU_REF_T tokens
# a step so that its warm-up and timed steps end within a few minutes
CPU_ALL_T, CPU_ONE_T, CPU_REF_T = 16384, 1024, 4096


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the context lines of the other workloads")
    ap.add_argument("--workload", default=None,
                    help="KEY[:WINDOW]: run this workload (full window unless WINDOW) as the headline instead (testing)")
    return ap.parse_args()


def workload_arg(spec):
    """--workload KEY[:WINDOW] -> (key, window); no WINDOW, or "full", is the full window."""
    key, _, win = spec.partition(":")
    return key, (int(win) if win and win != "full" else None)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))

            def find(keys, node=None, depth=0):
                # a top-level number, else the first one found one or two levels down
                node = d if node is None else node
                for k in keys:
                    if isinstance(node, dict) and isinstance(node.get(k), (int, float)):
                        return float(node[k])
                if depth < 2 and isinstance(node, dict):
                    for v in node.values():
                        r = find(keys, v, depth + 1) if isinstance(v, dict) else None
                        if r is not None:
                            return r
                return None
            hbm = find(["hbm_gbs", "hbm_GBps", "hbm_gb_s"])
            bf = find(["bf16_tflops", "bf16_TFLOPs"])
            bfs = find(["bf16_tflops_sustained"])
            if hbm and bf:
                return {"hbm_gbs": hbm, "bf16_tflops": bf, "bf16_tflops_sustained": bfs or bf}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.lines = []
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)
        return summarize_clocks(self.lines)


def summarize_clocks(lines):
    """Median SM clock, maximum clock and the throttle reasons seen in nvidia-smi csv lines."""
    sm, mx, power, reasons = [], [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        f = [x.strip() for x in ln.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            mx.append(float(f[2]))
        except ValueError:
            continue
        try:
            power.append(float(f[3]))
        except ValueError:
            pass
        for nm, v in zip(names, f[5:9]):
            if v.lower() == "active":
                reasons.add(nm)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
            "samples": len(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ multi-rank reduction (weak scaling)
def max_over_ranks(v, world, device=None):
    """Max of a per-rank timing over all ranks (any torch.distributed backend)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank, world, ms_per_step_max):
    """Whole-job throughput: all ranks' tokens over the slowest rank's step time."""
    return tokens_per_rank * world / (ms_per_step_max * 1e-3)


# ------------------------------------------------------------------ per-kernel algorithmic work
def kernel_table(P, N, xb, db, trunc, K=1):
    """Algorithmic bytes (and flops) per token of one launch of each kernel kind, as the
    step runs it.  xb / db: bytes of a GEMM operand / of a VJP seed.  In a stack of K
    layers the first layer's residual is its bf16 input and the others' the fp32 stream,
    so proj_out's residual bytes are the mean over the K launches."""
    res = (P * xb + (K - 1) * 4 * P) / K
    # bf16 layers: the forward scan also reads c and writes c . h in bf16, which the
    # output projection reads instead of c and h in fp32
    chb = 2 * N if xb == 2 else 0
    # bf16 layers: the cotangent gy also has a bf16 copy (written with it), which the
    # backward GEMMs read instead of the fp32 values
    gyx = 2 * P if xb == 2 else 0
    gyr = 2 * P if xb == 2 else 4 * P
    return {
        "proj_in": dict(bytes=P * xb + 3 * N * 4, flops=2 * P * 3 * N),
        "fwd_scan": dict(bytes=3 * N * 4 + (N * 4 + chb if chb else 0)),
        "proj_out": dict(bytes=(chb if chb else 2 * N * 4) + res + P * 4, flops=2 * N * P),
        "loss": dict(bytes=3 * P * 4 + gyx),
        "cot_proj": dict(bytes=gyr + N * 4, flops=2 * P * N),
        "win_scan": dict(bytes=4 * N * 4),
        "bwd_scan": dict(bytes=4 * N * 4 + 4 * N * db + (N * 4 if trunc else 0)),
        "param_dW_in": dict(bytes=P * xb + 3 * N * db, flops=2 * P * 3 * N),
        "param_dW_o": dict(bytes=N * db + gyr, flops=2 * N * P),
        "colsum": dict(bytes=N * db),
        # in a stack the input gradient goes through the normalised input in its epilogue: it
        # reads gy, xhat, r and the row dots dz and writes gy_prev (and its bf16 copy); with
        # one layer it is gy + dxhat
        "input_grad": dict(bytes=3 * N * db + 2 * P * 4 + ((P * xb + 4 + 4 * ((N + 127) // 128) + gyx) if K > 1 else 0),
                           flops=2 * 3 * N * P),
        "rms_norm": dict(bytes=4 * P + P * xb + 4),
        "rms_norm_bwd": dict(bytes=16 * P + 4),
    }


def sel_kernel_table(P, N, xb, db, K=1):
    """The general selective layer: algorithmic bytes (and flops) per token of each call's
    kernels (each scan counts its three launches together).  The forward scan reads z and
    xhat and writes h and y; the reverse scan reads z, xhat, gy and h and writes dz (the
    truncated form also writes and reads the window sums R, 8 P N bytes a token beyond
    these counts).  In a stack of K layers, layers 2..K also read the residual input in the
    forward scan and, in the reverse scan, read r and write gadd and the row dots (the
    table gives the mean over the K launches); sel_dx (the input GEMM with the
    normalisation in its epilogue: dz, gadd, xhat, r and the row dots in, gy_prev out) and
    rms_norm run K - 1 times."""
    zw = P + 2 * N
    nsl = -(-P // (256 // (N // 8)))
    f = (K - 1) / K
    tab = {
        "sel_proj": dict(bytes=P * xb + zw * 4, flops=2 * P * zw),
        "sel_fwd": dict(bytes=zw * 4 + P * xb + 4 * P * N + 4 * P + f * 4 * P),
        "loss": dict(bytes=3 * P * 4),
        "sel_bwd": dict(bytes=zw * 4 + P * xb + 4 * P + 4 * P * N + zw * db + f * (4 + 4 * P + 4 * (nsl + 1))),
        "sel_dW": dict(bytes=P * xb + zw * db, flops=2 * P * zw),
        "colsum": dict(bytes=P * db),
    }
    if K > 1:
        tab["sel_dx"] = dict(bytes=zw * db + 4 * P + P * xb + 4 + 4 * (nsl + 1) + 4 * P, flops=2 * zw * P)
        tab["rms_norm"] = dict(bytes=4 * P + P * xb + 4)
    return tab


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a kernel of a
# workload, from the committed ncu summary (profiles/); each summary records a hash of the
# library sources it was captured from, and a summary whose hash differs from the current
# sources gives no traffic (the kernel has changed since).
PROFILE_OF = {
    ("ssm1_p128", "bwd_scan"): "k_bwd_scan_ssm1_p128.md",
    ("ssm1_p128", "fwd_scan"): "k_fwd_scan_ssm1_p128.md",
    ("ssm4_p2048", "input_grad"): "k_gemm_tc_input_grad_ssm4_p2048.md",
    ("ssm4_p2048", "proj_out"): "k_gemm_tc_proj_out_ssm4_p2048.md",
    ("ssm4_p2048", "param_dW_in"): "k_gemm_tc_param_dWin_ssm4_p2048.md",
    ("ssm4_p2048", "proj_in"): "k_gemm_tc_proj_in_ssm4_p2048.md",
    ("ssm4_p2048", "cot_proj"): "k_gemm_tc_cot_proj_ssm4_p2048.md",
    ("ssm4_p2048", "param_dW_o"): "k_gemm_tc_param_dWo_ssm4_p2048.md",
    ("ssm4_p2048", "bwd_scan"): "k_trunc_scan_ssm4_p2048.md",
    ("ssm4_p2048", "rms_norm"): "k_rms_norm_ssm4_p2048.md",
    ("ssm4_p2048", "fwd_scan"): "k_fwd_scan_ssm4_p2048.md",
    ("ssm4_p2048", "loss"): "k_loss_ssm4_p2048.md",
}


# The translation unit that holds each kernel kind; a summary's hash covers that file and
# the headers it includes, so a change elsewhere in the library leaves it fresh.
KERNEL_TU = {
    "input_grad": "adj_gemm_tc.cu", "proj_out": "adj_gemm_tc.cu", "param_dW_in": "adj_gemm_tc.cu",
    "proj_in": "adj_gemm_tc.cu", "cot_proj": "adj_gemm_tc.cu", "param_dW_o": "adj_gemm_tc.cu",
    "bwd_scan": "adj_scan.cu", "fwd_scan": "adj_scan.cu", "win_scan": "adj_scan.cu",
    "rms_norm": "adj_misc.cu", "loss": "adj_misc.cu", "colsum": "adj_misc.cu",
    "sel_fwd": "adj_sel.cu", "sel_bwd": "adj_sel.cu", "sel_proj": "adj_gemm_tc.cu", "sel_dW": "adj_gemm_tc.cu",
    "sel_dx": "adj_gemm_tc.cu",
}


def _includes(path, seen):
    """path and the local headers it includes, recursively (#include "...")."""
    if path in seen or not os.path.exists(path):
        return
    seen.add(path)
    for line in open(path, encoding="utf-8", errors="replace"):
        m = re.match(r'\s*#\s*include\s+"([^"]+)"', line)
        if m:
            _includes(os.path.normpath(os.path.join(os.path.dirname(path), m.group(1))), seen)


def source_hash(tu=None):
    """Hash of library sources, as recorded in profiles/: one translation unit of csrc (tu)
    with the library headers it includes, or every source and the public header (tu None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "adjoint_gradients_long_gb300", "csrc")
    if tu is None:
        files = sorted(glob.glob(os.path.join(csrc, "*.cu*"))) + [os.path.join(ROOT, "include", "adj.h")]
    else:
        # the public header only declares the C entry points (no device code reads it), so a
        # new or changed declaration there leaves every kernel's summary fresh
        seen = set()
        _includes(os.path.join(csrc, tu), seen)
        files = sorted((f for f in seen if os.path.basename(f) != "adj.h"), key=os.path.basename)
    for f in files:
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(name, workload="ssm1_p128"):
    """(bytes per launch, source hash of the capture, whether it matches the sources now);
    (None, None, False) when no summary covers the kernel."""
    fn = PROFILE_OF.get((workload, name))
    path = os.path.join(ROOT, "profiles", fn) if fn else None
    if not path or not os.path.exists(path):
        return None, None, False
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    tot, state, per_launch_scale = 0.0, None, 1.0
    for line in open(path):
        for key in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            if line.startswith("| " + key + " |"):
                val, unit = line.split("|")[2].split()
                tot += float(val) * scale[unit]
        if line.startswith("Source hash:"):
            state = line.split(":", 1)[1].strip().split()[0]
        if line.startswith("Traffic scale:"):
            per_launch_scale = float(line.split(":", 1)[1].strip().split()[0])
    if tot <= 0:
        return None, state, False
    return tot * per_launch_scale, state, state == source_hash(KERNEL_TU.get(name))


def roofline_of(name, ent, peaks, split3):
    """Roofline entry of one kernel: HBM-bound kernels against the copy bandwidth; GEMMs
    against both the bandwidth and the tensor peak of their arithmetic (the fp32-accurate
    three-term bf16 split issues 3 bf16 MMAs per product, so its tensor peak is 1/3 of
    bf16's), reporting the bound they sit closer to.  The tensor fraction is taken against
    the burst bf16 peak; the fraction of the sustained (power-capped) figure is given
    beside it."""
    gbs = ent.get("achieved_gbs")
    hbm = {"kernel": name, "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
           "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"] if gbs is not None else None, "traffic": None}
    if "achieved_tflops" not in ent:
        return hbm
    div = 3.0 if split3 else 1.0
    tpk = peaks["bf16_tflops"] / div
    tps = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) / div
    ten = {"kernel": name, "bound": "tensor", "achieved": ent["achieved_tflops"], "peak": tpk, "unit": "TFLOP/s",
           "frac": ent["achieved_tflops"] / tpk, "peak_sustained": tps,
           "frac_sustained": ent["achieved_tflops"] / tps, "traffic": None,
           "note": "fp32-accurate 3-term bf16 split: peak = bf16 peak / 3" if split3 else "bf16"}
    return ten if hbm["frac"] is None or ten["frac"] >= hbm["frac"] else hbm


def kernels_summary(prof, tab, tokens, peaks, split3):
    """Per kernel kind: launches, mean device time, share of the step and, where the kind
    has an algorithmic count, achieved GB/s (TFLOP/s) and its roofline fraction."""
    tot = sum(ms for _, ms in prof.values())
    out = {}
    for name, (n, ms) in sorted(prof.items(), key=lambda kv: -kv[1][1]):
        per = ms / n
        ent = {"launches": n, "ms_per_launch": per, "share": ms / tot if tot else None}
        if name in tab:
            ent["algo_bytes_per_launch"] = tab[name]["bytes"] * tokens
            ent["achieved_gbs"] = tab[name]["bytes"] * tokens / (per * 1e-3) / 1e9
            ent["hbm_frac"] = ent["achieved_gbs"] / peaks["hbm_gbs"]
            if "flops" in tab[name]:
                ent["algo_flops_per_launch"] = tab[name]["flops"] * tokens
                ent["achieved_tflops"] = tab[name]["flops"] * tokens / (per * 1e-3) / 1e12
            r = roofline_of(name, ent, peaks, split3)
            ent["roofline_bound"], ent["roofline_frac"] = r["bound"], r["frac"]
        out[name] = ent
    return out


# ------------------------------------------------------------------ oracle (CPU baseline / reference arm)
def cpu_model():
    """The host CPU's model name (/proc/cpuinfo on x86, lscpu on Arm), else the machine type."""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith(("model name", "vendor id")):
                name = line.split(":", 1)[1].strip()
                if line.strip().lower().startswith("model name"):
                    return f"{name} ({platform.machine()})"
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def oracle_sample(T, threads, key=None, window=None):
    """Seconds the fp64 oracle takes for one gradient step (forward, loss, adjoint with the
    workload's window, parameter gradients) on the first T tokens of one sequence of the
    workload, with `threads` threads (0: all cores).  Returns (tokens, seconds, threads)."""
    import numpy as np
    import oracle
    from adjoint_gradients_long_gb300 import synth
    key = key or HEADLINE[0]
    window = HEADLINE[1] if key == HEADLINE[0] and window is None else window
    inp = synth.make_inputs(key, T=T, B=1)
    layers = [{k: np.asarray(v, np.float64) for k, v in W.items()} for W in inp["layers"]]
    used = oracle.threads(threads if threads > 0 else (os.cpu_count() or 1))
    t0 = time.perf_counter()
    oracle.stack_grad(layers, inp["xhat"], inp["target"], window, oracle.AGGREGATED)
    dt = time.perf_counter() - t0
    return T, dt, used


def cpu_baseline(K):
    """The oracle on the host cores: all cores on a CPU_ALL_T-token prefix (the value) and
    one core on a CPU_ONE_T-token prefix (beside it), in tokens/s per layer."""
    toks, dt, used = oracle_sample(CPU_ALL_T, 0)
    toks1, dt1, _ = oracle_sample(CPU_ONE_T, 1)
    key, window = HEADLINE
    return {"value": toks * K / dt, "unit": "tokens/s per layer", "cores": used, "kind": "oracle",
            "sample": f"first {toks} tokens of one sequence of {key} ({K} layers, window {window}: every "
                      f"pair is inside it), aggregated-literal fp64 mode, {used} threads ({dt:.1f} s)",
            "single_thread": {"value": toks1 * K / dt1, "unit": "tokens/s per layer",
                              "sample": f"first {toks1} tokens, 1 thread ({dt1:.1f} s)"},
            "nproc": os.cpu_count(), "cpu_model": cpu_model()}


SEL_CPU_T = 1024   # tokens of the selective workload's oracle sample


def sel_cpu_baseline(key, window):
    """The selective layer's fp64 oracle on the host cores (forward, loss, adjoint with the
    window, parameter gradients) on the first SEL_CPU_T tokens of the workload, all cores."""
    import numpy as np
    import oracle
    from oracle import selective
    from adjoint_gradients_long_gb300 import synth
    inp = synth.make_sel_inputs(key, T=SEL_CPU_T, B=1)
    W = {k: np.asarray(inp[k], np.float64) for k in ("W_in", "b_dt", "A")}
    used = oracle.threads(os.cpu_count() or 1)
    t0 = time.perf_counter()
    st = selective.forward(W, inp["xhat"])
    _, gy = selective.loss_and_cotangent(st["y"], inp["target"])
    selective.grad(W, st, gy, window)
    dt = time.perf_counter() - t0
    return {"value": SEL_CPU_T / dt, "unit": "tokens/s per layer", "cores": used, "kind": "oracle",
            "sample": f"first {SEL_CPU_T} tokens of {key} (window {window if window else 'full'}: every pair "
                      f"of the sample is inside it), aggregated fp64 mode, {used} threads ({dt:.1f} s)"}


def run_reference(args, rank):
    """The reference arm: the fp64 oracle (this path has no other reference code), one
    step = one gradient step on a CPU_REF_T-token prefix of the headline workload."""
    if rank != 0:
        return
    import oracle
    from adjoint_gradients_long_gb300 import synth
    oracle.build()
    key, window = HEADLINE
    K = synth.workload(key).K
    for _ in range(args.warmup):
        oracle_sample(CPU_REF_T, 0)
    times, used = [], 1
    for _ in range(args.steps):
        _, dt, used = oracle_sample(CPU_REF_T, 0)
        times.append(dt)
    med = statistics.median(times)
    value = CPU_REF_T * K / med
    sample = (f"first {CPU_REF_T} tokens of one sequence of {key} ({K} layers, window {window}), "
              f"aggregated-literal fp64 mode, {used} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s per layer", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": med * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": key, "window": window, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "tokens/s per layer", "cores": used, "kind": "oracle",
                         "sample": sample, "nproc": os.cpu_count(), "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s per layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ one workload on the GPU
class Workload:
    """Device buffers of one workload, its captured steps and the timing helpers."""

    def __init__(self, key, window, dev, rank=0):
        import torch
        from adjoint_gradients_long_gb300 import synth
        from adjoint_gradients_long_gb300.stack import AdjStack
        self.torch = torch
        self.w = synth.workload(key)
        self.key, self.window, self.dev = key, window, dev
        w = self.w
        self.bf16 = w.x_dtype == "bf16"
        self.inputs = synth.make_inputs(w, seed=w.seed + 7919 * rank)
        self.st = AdjStack(w.B, w.T, w.P, w.N, w.K, x_bf16=self.bf16, d_bf16=self.bf16, Tbar=window, device=dev)
        self.st.load(self.inputs)
        self.stream = torch.cuda.current_stream(dev)
        self.flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        self.tokens = w.B * w.T * w.K

    def capture(self):
        from adjoint_gradients_long_gb300 import lib
        n0 = lib.launch_count()
        g = self.st.capture(self.window)
        self.torch.cuda.synchronize(self.dev)
        return g, (lib.launch_count() - n0) // 2      # capture() runs one eager step first

    def timed(self, steps, graph=None, profile=False, barrier=None):
        """Per-step CUDA-event times of `steps` steps, each after an L2 flush: replays of a
        captured step, or eager library calls."""
        from adjoint_gradients_long_gb300 import lib
        torch = self.torch
        if profile:
            lib.profile_reset()
            lib.profile_enable(True)
        if barrier:
            barrier()
        ev = []
        for _ in range(steps):
            self.flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            if graph is not None:
                graph.replay()
            else:
                self.st.step(self.window)
            e1.record(self.stream)
            ev.append((e0, e1))
        if barrier:
            barrier()
        torch.cuda.synchronize(self.dev)
        if profile:
            lib.profile_enable(False)
        return [a.elapsed_time(b) for a, b in ev]

    def kernels(self, steps, peaks):
        from adjoint_gradients_long_gb300 import lib
        self.timed(steps, profile=True)
        prof = lib.profile_read()
        lib.profile_reset()
        w = self.w
        trunc = self.window is not None and self.window < w.T
        xb = 2 if self.bf16 else 4
        tab = kernel_table(w.P, w.N, xb, xb, trunc, w.K)
        return kernels_summary(prof, tab, w.B * w.T, peaks, split3=not self.bf16)

    def e2e(self, steps, barrier):
        """The same steps through the C ABI with host buffers: each step's inputs are copied
        from pinned host memory (double-buffered on a second stream, so step i+1's copy
        overlaps step i) and the loss and every parameter gradient are copied back."""
        import numpy as np
        from adjoint_gradients_long_gb300.synth import bf16_bits
        torch, st, dev, stream = self.torch, self.st, self.dev, self.stream
        if self.bf16:
            bits = bf16_bits(np.ascontiguousarray(self.inputs["xhat"], np.float32)).view(np.int16)
            hx = torch.from_numpy(bits).view(torch.bfloat16).pin_memory()
        else:
            hx = torch.from_numpy(np.ascontiguousarray(self.inputs["xhat"], np.float32)).pin_memory()
        ht = torch.from_numpy(np.ascontiguousarray(self.inputs["target"], np.float32)).pin_memory()
        hl = torch.empty(1, dtype=torch.float64).pin_memory()
        grads = [t for k in range(st.K) for t in (st.dW_in[k], st.db_a[k], st.dW_o[k])]
        hg = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in grads]
        h2d = hx.numel() * hx.element_size() + ht.numel() * 4
        d2h = 8 + sum(t.numel() * 4 for t in hg)
        copy_stream = torch.cuda.Stream(dev)
        bufs = [(st.x[0], st.target), (st.x[0].clone(), st.target.clone())]
        landed = [torch.cuda.Event(), torch.cuda.Event()]
        used = [torch.cuda.Event(), torch.cuda.Event()]
        graphs = []
        for b in range(2):
            st.x[0], st.target = bufs[b]
            graphs.append(st.capture(self.window))
        st.x[0], st.target = bufs[0]
        torch.cuda.synchronize(dev)

        def stage_inputs(b, after):
            copy_stream.wait_event(after)
            with torch.cuda.stream(copy_stream):
                bufs[b][0].copy_(hx, non_blocking=True)
                bufs[b][1].copy_(ht, non_blocking=True)
                landed[b].record(copy_stream)

        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        stage_inputs(0, e0)
        for i in range(steps):
            b = i % 2
            stream.wait_event(landed[b])
            if i + 1 < steps:
                stage_inputs(1 - b, used[1 - b] if i > 0 else e0)
            graphs[b].replay()
            used[b].record(stream)
            hl.copy_(st.loss, non_blocking=True)
            for hgt, dg in zip(hg, grads):
                hgt.copy_(dg, non_blocking=True)
        e1.record(stream)
        barrier()
        st.x[0], st.target = bufs[0]
        del graphs, bufs
        return e0.elapsed_time(e1) / steps, h2d, d2h

    def release(self):
        del self.st, self.flush, self.inputs
        self.torch.cuda.empty_cache()


def context_line(key, window, dev, peaks, steps, warmup):
    """One of the other workloads, measured like the headline (graph replay, L2 flushed
    before every step, median), without the end-to-end and CPU legs."""
    wl = Workload(key, window, dev)
    for _ in range(warmup):
        wl.st.step(window)
    g, per = wl.capture()
    for _ in range(warmup):
        g.replay()
    ms = wl.timed(steps, graph=g)
    status = wl.st.status()
    kern = wl.kernels(min(steps, 5), peaks)
    w = wl.w
    from adjoint_gradients_long_gb300 import lib
    med = statistics.median(ms)
    out = {"workload": key, "window": window if window is not None else "full", "B": w.B, "T": w.T, "P": w.P,
           "N": w.N, "K": w.K, "dtype": "bf16 GEMM operands, fp32 scans" if wl.bf16 else "f32",
           "value": wl.tokens / (med * 1e-3), "unit": "tokens/s per layer", "ms_per_step": med,
           "ms_mean": sum(ms) / len(ms), "steps": steps, "gpu_launches_per_step": per,
           "device_status": lib.STATUS.get(status, status), "kernels": kern}
    del g
    wl.release()
    return out


def sel_context_line(key, window, dev, peaks, steps, warmup, cpu=False, K=1):
    """The general selective layer on one of its workloads, alone (K = 1) or as a residual
    stack of K layers: graph replay of one step (forward, loss, reverse, parameter
    gradients and, in a stack, the cotangents passed down), L2 flushed before every step,
    median."""
    import torch
    from adjoint_gradients_long_gb300 import lib, synth
    from adjoint_gradients_long_gb300.sel_layer import SelLayer, SelStack
    w = synth.SEL_WORKLOADS[key]
    bf16 = w.x_dtype == "bf16"
    if K == 1:
        L = SelLayer(w.B, w.T, w.P, w.N, x_bf16=bf16, Tbar=window, device=dev)
        L.load(synth.make_sel_inputs(w))
    else:
        L = SelStack(w.B, w.T, w.P, w.N, K, x_bf16=bf16, Tbar=window, device=dev)
        L.load(synth.make_sel_stack_inputs(w, K))
    for _ in range(warmup):
        L.step(window)
    n0 = lib.launch_count()
    g = L.capture(window)
    torch.cuda.synchronize(dev)
    per = (lib.launch_count() - n0) // 2
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(n, replay=True):
        ev = []
        for _ in range(n):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if replay:
                g.replay()
            else:
                L.step(window)
            e1.record(stream)
            ev.append((e0, e1))
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in ev]

    for _ in range(warmup):
        g.replay()
    ms = timed(steps)
    status = L.status()
    lib.profile_reset()
    lib.profile_enable(True)
    timed(min(steps, 5), replay=False)
    lib.profile_enable(False)
    prof = lib.profile_read()
    lib.profile_reset()
    xb = 2 if bf16 else 4
    kern = kernels_summary(prof, sel_kernel_table(w.P, w.N, xb, xb, K), w.B * w.T, peaks, split3=not bf16)
    med = statistics.median(ms)
    out = {"workload": key, "layer": "general selective (softplus step, exp(dt A) decay, input-dependent B_t, C_t)"
           + (f", residual stack of {K} with normalised inputs" if K > 1 else ""),
           "window": window if window is not None else "full", "B": w.B, "T": w.T, "P": w.P, "N": w.N, "K": K,
           "dtype": "bf16 GEMM operands, fp32 scans" if bf16 else "f32",
           "value": w.B * w.T * K / (med * 1e-3), "unit": "tokens/s per layer", "ms_per_step": med,
           "ms_mean": sum(ms) / len(ms), "steps": steps, "gpu_launches_per_step": per,
           "device_status": lib.STATUS.get(status, status), "kernels": kern}
    if cpu and K == 1:
        out["cpu_baseline"] = sel_cpu_baseline(key, window)
    del g, L, flush
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from adjoint_gradients_long_gb300 import build as adj_build, lib

    adj_build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    key, window = HEADLINE
    if args.workload:
        key, window = workload_arg(args.workload)
    peaks, peak_src = load_peaks()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    wl = Workload(key, window, dev, rank)
    w = wl.w
    for _ in range(max(3, args.warmup)):
        wl.st.step(window)
    barrier()
    assert wl.st.status() == 0

    # The timed steps replay a CUDA graph of one step (the library enqueues only kernels and
    # memsets on the caller's stream, so a step captures whole); the replay does the same
    # work as the eager calls without their launch gaps.  Eager steps are timed too.
    g, per_step = wl.capture()
    for _ in range(max(3, args.warmup)):
        g.replay()
    barrier()
    assert wl.st.status() == 0

    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    ms = wl.timed(args.steps, graph=g, barrier=barrier)
    t_end = time.time() + 1.0      # keep the same load for a few clock samples if the region was short
    while time.time() < t_end:
        g.replay()
        torch.cuda.synchronize(dev)
    clk = clocks.stop()
    status = wl.st.status()
    ms_eager = wl.timed(args.steps, barrier=barrier)
    kern = wl.kernels(args.steps, peaks)
    e2e_ms, h2d, d2h = wl.e2e(args.steps, barrier)
    del g

    med = max_over_ranks(statistics.median(ms), world, dev)
    mean = max_over_ranks(sum(ms) / len(ms), world, dev)
    med_eager = max_over_ranks(statistics.median(ms_eager), world, dev)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    tokens = wl.tokens * world

    # the dominant kernel among those with an algorithmic count
    dom = next((n for n, e in kern.items() if "achieved_gbs" in e), next(iter(kern)))
    roof = roofline_of(dom, kern[dom], peaks, split3=not wl.bf16)
    traffic, state, fresh = profiled_traffic(dom, key)
    roof["traffic"] = traffic if fresh else None
    if traffic is not None:
        roof["traffic_unit"] = "bytes per launch"
        roof["traffic_source"] = (f"ncu dram__bytes_read.sum + dram__bytes_write.sum, "
                                  f"profiles/{PROFILE_OF[(key, dom)]} (sources {state})")
        if not fresh:
            roof["traffic_stale"] = f"captured from sources {state}, current sources {source_hash(KERNEL_TU.get(dom))}"
    roof["algo_per_launch"] = kern[dom].get("algo_flops_per_launch" if roof["bound"] == "tensor"
                                            else "algo_bytes_per_launch")
    roof["ms_per_launch"] = kern[dom]["ms_per_launch"]
    roof["peak_source"] = f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.workload:
        cpu = cpu_baseline(w.K)

    others = []
    if rank == 0 and world == 1 and not args.no_other_workloads and not args.workload:
        wl.release()
        del wl
        for k2, w2 in CONTEXT:
            others.append(context_line(k2, w2, dev, peaks, min(args.steps, 10), max(3, min(args.warmup, 3))))
        for k2, w2, K2 in SEL_CONTEXT:
            others.append(sel_context_line(k2, w2, dev, peaks, min(args.steps, 10), max(3, min(args.warmup, 3)),
                                           cpu=not args.no_cpu_baseline, K=K2))

    if rank == 0:
        line = {
            "metric": METRIC, "value": weak_scaling_value(w.B * w.T * w.K, world, med),
            "unit": "tokens/s per layer", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": med, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.x_dtype == "bf16" else "f32",
            "data": "synthetic",
            "config": {"workload": key, "B": w.B, "T": w.T, "P": w.P, "N": w.N, "K": w.K,
                       "window": window if window is not None else "full",
                       "precision": ("bf16 GEMM operands (xhat, W, seeds), fp32 accumulate, fp32 scans and "
                                     "residual stream") if w.x_dtype == "bf16" else "f32",
                       "l2": "flushed before every timed step (256 MB write)", "tokens_per_step": tokens,
                       "launch": "each step replays a CUDA graph of its library calls",
                       "ms_per_step": "median of the timed steps"},
            "ms_mean": mean,
            "eager": {"ms_per_step": med_eager, "value": tokens / (med_eager * 1e-3),
                      "note": "the same step as direct library calls (no graph)"},
            "gpu_launches": per_step * args.steps,
            "gpu_launches_per_step": per_step,
            "roofline": roof,
            "kernels": kern,
            "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s per layer", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "note": "inputs copied H2D from pinned memory every step (double-buffered), loss and all "
                            "parameter gradients copied D2H every step, inside the timed region"},
            "cpu_baseline": cpu,
            "clocks": clk,
            "peaks": {"source": peak_src, **peaks},
            "device_status": lib.STATUS.get(status, status),
            "workloads": others,
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
