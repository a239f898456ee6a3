#!/usr/bin/env python
"""Benchmark: adjoint-gradient tokens/sec per layer on one GB300, with the roofline of
the dominant kernel, an end-to-end number through the C ABI with host buffers, and
the fp64 CPU oracle timed beside it.

One step = one pass of the whole path over one batch of the workload
ssm1_p128 (P=128, N=256, T=16384, B=4, one layer, fp32): adj_fwd_scan,
adj_loss_mse, adj_bwd_full (or adj_bwd_trunc with Tbar=2048), adj_param_grad.
The headline value is the full (exact) adjoint; the Tbar=2048 variant is reported
beside it.  L2 is flushed (a 256 MB write) before every timed step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs its own batch (independent sequences: weak scaling,
no collective on the data path); rank 0 prints one JSON line.
"""
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

WORKLOAD = "ssm1_p128"
TBAR = 2048
METRIC = "adjoint-gradient tokens/sec per layer on 1 GB300; % of HBM/tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CPU_SAMPLE_T = 4096          # oracle sample: first CPU_SAMPLE_T tokens of one sequence


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the short runs of the bf16 workloads reported under 'workloads'")
    return ap.parse_args()


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
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


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
def kernel_table(P, N, xb, db, trunc):
    """Algorithmic bytes (and flops) per token of each kernel kind, as built."""
    return {
        "proj_in": dict(bytes=P * xb + 3 * N * 4, flops=2 * P * 3 * N),
        "fwd_scan": dict(bytes=3 * N * 4),
        "proj_out": dict(bytes=2 * N * 4 + P * xb + P * 4, flops=2 * N * P),
        "loss": dict(bytes=3 * P * 4),
        "cot_proj": dict(bytes=P * 4 + N * 4, flops=2 * P * N),
        "win_scan": dict(bytes=4 * N * 4),
        "bwd_scan": dict(bytes=4 * N * 4 + 4 * N * db + (N * 4 if trunc else 0)),
        "param_dW_in": dict(bytes=P * xb + 3 * N * db, flops=2 * P * 3 * N),
        "param_dW_o": dict(bytes=N * db + P * 4, flops=2 * N * P),
        "colsum": dict(bytes=N * db),
        "input_grad": dict(bytes=3 * N * db + 2 * P * 4, flops=2 * 3 * N * P),
    }


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a kernel, from
# the committed ncu summary of the bench workload (profiles/), with the code state it
# was captured at; None when no summary covers the kernel.
PROFILE_OF = {"bwd_scan": "k_bwd_scan_ssm1_p128.md", "fwd_scan": "k_fwd_scan_ssm1_p128.md",
              "proj_in": "k_gemm_tc_proj_in_ssm1_p128.md", "proj_out": "k_gemm_tc_proj_out_ssm1_p128.md",
              "cot_proj": "k_gemm_tc_cot_proj_ssm1_p128.md", "param_dW_in": "k_gemm_tc_param_dWin_ssm1_p128.md"}


def profiled_traffic(name):
    fn = PROFILE_OF.get(name)
    path = os.path.join(ROOT, "profiles", fn) if fn else None
    if not path or not os.path.exists(path):
        return None, None
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    tot, state = 0.0, None
    for line in open(path):
        for key in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            if line.startswith("| " + key + " |"):
                val, unit = line.split("|")[2].split()
                tot += float(val) * scale[unit]
        if line.startswith("Code state:"):
            state = line.split(":", 1)[1].split("(")[0].strip().rstrip(".")
    return (tot if tot > 0 else None), state


def roofline_of(name, ent, peaks, split3):
    """Roofline entry of one kernel: HBM-bound kernels against the copy bandwidth; GEMMs
    against both the bandwidth and the tensor peak of their arithmetic (the fp32-accurate
    three-term bf16 split issues 3 bf16 MMAs per product, so its tensor peak is 1/3 of
    bf16's), reporting the bound they sit closer to."""
    gbs = ent.get("achieved_gbs")
    hbm = {"kernel": name, "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
           "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"] if gbs is not None else None, "traffic": None}
    if "achieved_tflops" not in ent:
        return hbm
    # the GEMMs are timed inside a long step: the sustained (power-capped) bf16 figure
    tpk = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) / (3.0 if split3 else 1.0)
    ten = {"kernel": name, "bound": "tensor", "achieved": ent["achieved_tflops"], "peak": tpk, "unit": "TFLOP/s",
           "frac": ent["achieved_tflops"] / tpk, "traffic": None,
           "note": "fp32-accurate 3-term bf16 split: peak = bf16 peak / 3" if split3 else "bf16"}
    return ten if hbm["frac"] is None or ten["frac"] >= hbm["frac"] else hbm


# ------------------------------------------------------------------ oracle (CPU baseline / reference arm)
def oracle_sample(seconds_hint=False):
    import numpy as np
    import oracle
    from adjoint_gradients_long_gb300 import synth
    inp = synth.make_inputs(WORKLOAD, T=CPU_SAMPLE_T, B=1)
    layers = [{k: np.asarray(v, np.float64) for k, v in W.items()} for W in inp["layers"]]
    t0 = time.perf_counter()
    oracle.stack_grad(layers, inp["xhat"], inp["target"], None, oracle.AGGREGATED)
    dt = time.perf_counter() - t0
    return CPU_SAMPLE_T, dt


def run_reference(args, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        oracle_sample()
    times = []
    toks = 0
    for _ in range(args.steps):
        toks, dt = oracle_sample()
        times.append(dt)
    mean = sum(times) / len(times)
    value = toks / mean
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"first {toks} tokens of one sequence", "window": "full"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {toks} tokens of one sequence of {WORKLOAD}, full window, "
                                   "aggregated-literal mode, single thread"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ the other workloads (context lines)
OTHER = (("ssm8_p512", 4096), ("ssm1_1m", 4096), ("ssm1_1m", None), ("ssm4_p2048", 8192))


def measure_workload(key, window, dev, peaks, steps=3, warmup=2):
    """Short device-timed run of one of the bf16 workloads at full size (weak evidence:
    few steps, L2 not flushed, inputs larger than L2).  Returns tokens/s per layer and
    the per-kernel roofline entries."""
    import torch
    from adjoint_gradients_long_gb300 import lib, synth
    from adjoint_gradients_long_gb300.stack import AdjStack
    w = synth.workload(key)
    inputs = synth.make_inputs(w)
    st = AdjStack(w.B, w.T, w.P, w.N, w.K, x_bf16=True, d_bf16=True, Tbar=window, device=dev)
    st.load(inputs)
    del inputs
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        st.step(window)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        st.step(window)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    lib.profile_reset()
    lib.profile_enable(True)
    st.step(window)
    torch.cuda.synchronize(dev)
    lib.profile_enable(False)
    prof = lib.profile_read()
    lib.profile_reset()
    status = st.status()
    tab = kernel_table(w.P, w.N, 2, 2, window is not None and window < w.T)
    tok = w.B * w.T
    kern = {}
    tot = sum(v[1] for v in prof.values())
    for name, (n, t) in sorted(prof.items(), key=lambda kv: -kv[1][1]):
        per = t / n
        ent = {"launches": n, "ms_per_launch": per, "share": t / tot}
        if name in tab:
            ent["achieved_gbs"] = tab[name]["bytes"] * tok / (per * 1e-3) / 1e9
            if "flops" in tab[name]:
                ent["achieved_tflops"] = tab[name]["flops"] * tok / (per * 1e-3) / 1e12
            r = roofline_of(name, ent, peaks, split3=False)
            ent["roofline_bound"], ent["roofline_frac"] = r["bound"], r["frac"]
        kern[name] = ent
    del st
    torch.cuda.empty_cache()
    return {"workload": key, "window": window if window is not None else "full", "B": w.B, "T": w.T, "P": w.P,
            "N": w.N, "K": w.K, "dtype": "bf16 GEMM operands, fp32 scans",
            "value": tok * w.K / (ms * 1e-3), "unit": "tokens/s per layer", "ms_per_step": ms, "steps": steps,
            "device_status": lib.STATUS.get(status, status), "kernels": dict(list(kern.items())[:6])}


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist
    from adjoint_gradients_long_gb300 import build as adj_build, lib, synth
    from adjoint_gradients_long_gb300.stack import AdjStack

    adj_build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = synth.workload(WORKLOAD)
    B, T, P, N, K = w.B, w.T, w.P, w.N, w.K
    inputs = synth.make_inputs(w, seed=w.seed + 7919 * rank)
    st = AdjStack(B, T, P, N, K, Tbar=TBAR, device=dev)
    st.load(inputs)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(window, steps, profile=False, graph=None, per_step=0):
        """Per-step CUDA-event times of `steps` steps, each after an L2 flush: eager library
        calls, or replays of a captured step (graph; its launches counted at capture)."""
        times = []
        n0 = lib.launch_count()
        if profile:
            lib.profile_reset()
            lib.profile_enable(True)
        barrier()
        for _ in range(steps):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if graph is not None:
                graph.replay()
            else:
                st.step(window)
            e1.record(stream)
            times.append((e0, e1))
        barrier()
        if profile:
            lib.profile_enable(False)
        launches = per_step * steps if graph is not None else lib.launch_count() - n0
        ms = [a.elapsed_time(b) for a, b in times]
        return ms, launches

    for _ in range(max(3, args.warmup)):
        st.step(None)
        st.step(TBAR)
    barrier()
    assert st.status() == 0

    # The timed steps replay a CUDA graph of one step (the library enqueues only kernels and
    # memsets on the caller's stream, so a step captures whole); the replay does the same
    # work as the eager calls without their launch gaps.  Eager steps are timed too.
    def capture(window):
        n0 = lib.launch_count()
        g = st.capture(window)
        torch.cuda.synchronize(dev)
        return g, (lib.launch_count() - n0) // 2     # capture() runs one eager step first
    g_full, per_full = capture(None)
    g_trunc, per_trunc = capture(TBAR)
    for _ in range(max(3, args.warmup)):
        g_full.replay()
        g_trunc.replay()
    barrier()
    assert st.status() == 0

    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    ms_full, launches_full = timed(None, args.steps, graph=g_full, per_step=per_full)
    ms_trunc, launches_trunc = timed(TBAR, args.steps, graph=g_trunc, per_step=per_trunc)
    t_end = time.time() + 1.0      # keep the same load for a few clock samples if the region was short
    while time.time() < t_end:
        g_full.replay()
        torch.cuda.synchronize(dev)
    clk = clocks.stop()
    status = st.status()
    ms_eager, _ = timed(None, args.steps)

    # per-kernel device time, recorded with CUDA events on the launching stream
    _, _ = timed(None, args.steps, profile=True)
    prof_full = lib.profile_read()
    _, _ = timed(TBAR, args.steps, profile=True)
    prof_trunc = lib.profile_read()
    lib.profile_reset()

    # end to end through the C ABI with host buffers: H2D of the step's inputs from pinned
    # memory, the step, D2H of the loss and the gradients
    hx = torch.from_numpy(np.ascontiguousarray(inputs["xhat"], np.float32)).pin_memory()
    ht = torch.from_numpy(np.ascontiguousarray(inputs["target"], np.float32)).pin_memory()
    hl = torch.empty(1, dtype=torch.float64).pin_memory()
    hg = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (st.dW_in[0], st.db_a[0], st.dW_o[0])]
    h2d = hx.numel() * 4 + ht.numel() * 4
    d2h = 8 + sum(t.numel() * 4 for t in hg)
    # Inputs are double-buffered: step i+1's inputs are copied on a second stream while step
    # i computes; every step's copies stay inside the timed region.
    copy_stream = torch.cuda.Stream(dev)
    bufs = [(st.x[0], st.target), (st.x[0].clone(), st.target.clone())]
    landed = [torch.cuda.Event(), torch.cuda.Event()]      # inputs of buffer b copied
    used = [torch.cuda.Event(), torch.cuda.Event()]        # step that read buffer b done
    # one captured step per input buffer (a graph keeps the pointers it was captured with)
    graphs = []
    for b in range(2):
        st.x[0], st.target = bufs[b]
        graphs.append(st.capture(None))
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
    for i in range(args.steps):
        b = i % 2
        stream.wait_event(landed[b])
        if i + 1 < args.steps:
            # the other buffer was last read by step i-1
            stage_inputs(1 - b, used[1 - b] if i > 0 else e0)
        graphs[b].replay()
        used[b].record(stream)
        hl.copy_(st.loss, non_blocking=True)
        for hgt, dg in zip(hg, (st.dW_in[0], st.db_a[0], st.dW_o[0])):
            hgt.copy_(dg, non_blocking=True)
    e1.record(stream)
    barrier()
    st.x[0], st.target = bufs[0]
    e2e_ms = e0.elapsed_time(e1) / args.steps

    # max over ranks
    mean_full = max_over_ranks(sum(ms_full) / len(ms_full), world, dev)
    mean_trunc = max_over_ranks(sum(ms_trunc) / len(ms_trunc), world, dev)
    mean_eager = max_over_ranks(sum(ms_eager) / len(ms_eager), world, dev)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    tokens = B * T * K * world

    peaks, peak_src = load_peaks()
    table = kernel_table(P, N, 4, 4, False)
    tableT = kernel_table(P, N, 4, 4, True)

    def kernels_summary(prof, tab):
        tot = sum(ms for _, ms in prof.values())
        out = {}
        for name, (n, ms) in sorted(prof.items(), key=lambda kv: -kv[1][1]):
            per = ms / n
            ent = {"launches": n, "ms_per_launch": per, "share": ms / tot if tot else None}
            if name in tab:
                tok = B * T
                ent["algo_bytes_per_launch"] = tab[name]["bytes"] * tok
                ent["achieved_gbs"] = tab[name]["bytes"] * tok / (per * 1e-3) / 1e9
                ent["hbm_frac"] = ent["achieved_gbs"] / peaks["hbm_gbs"]
                if "flops" in tab[name]:
                    ent["algo_flops_per_launch"] = tab[name]["flops"] * tok
                    ent["achieved_tflops"] = tab[name]["flops"] * tok / (per * 1e-3) / 1e12
            out[name] = ent
        return out

    kf = kernels_summary(prof_full, table)
    kt = kernels_summary(prof_trunc, tableT)
    # the dominant kernel among those with an algorithmic byte count
    dom = next((n for n, e in kf.items() if "achieved_gbs" in e), next(iter(kf)))
    roof = roofline_of(dom, kf[dom], peaks, split3=True)
    roof["traffic"], state = profiled_traffic(dom)
    if roof["traffic"] is not None:
        roof["traffic_unit"] = "bytes per launch"
        roof["traffic_source"] = f"ncu dram__bytes_read.sum + dram__bytes_write.sum, profiles/{PROFILE_OF[dom]} ({state})"
    roof["peak_source"] = f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})"
    for name, ent in kf.items():
        if "achieved_gbs" in ent:
            r = roofline_of(name, ent, peaks, split3=True)
            ent["roofline_bound"], ent["roofline_frac"] = r["bound"], r["frac"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        toks, dt = oracle_sample()
        cpu = {"value": toks / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"first {toks} tokens of one sequence of {WORKLOAD}, full window, aggregated-literal "
                         f"mode, single thread ({dt:.1f} s)"}

    others = []
    if rank == 0 and world == 1 and not args.no_other_workloads:
        del st
        torch.cuda.empty_cache()
        for key, window in OTHER:
            others.append(measure_workload(key, window, dev, peaks))

    if rank == 0:
        line = {
            "metric": METRIC, "value": weak_scaling_value(B * T * K, world, mean_full), "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_full, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": B, "T": T, "P": P, "N": N, "K": K, "window": "full",
                       "l2": "flushed before every timed step (256 MB write)", "tokens_per_step": tokens,
                       "launch": "each step replays a CUDA graph of its library calls"},
            "eager": {"ms_per_step": mean_eager, "value": tokens / (mean_eager * 1e-3),
                      "note": "the same step as direct library calls (no graph)"},
            "truncated": {"window": TBAR, "value": tokens / (mean_trunc * 1e-3), "ms_per_step": mean_trunc,
                          "gpu_launches": launches_trunc},
            "gpu_launches": launches_full,
            "roofline": roof,
            "kernels": kf,
            "kernels_truncated": kt,
            "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
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
