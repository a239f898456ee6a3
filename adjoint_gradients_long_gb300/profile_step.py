"""Run a few gradient steps of one workload, resized, through the library: the command
the ncu captures under profiles/ are taken with.

  python -m adjoint_gradients_long_gb300.profile_step WORKLOAD [--T T] [--K K] [--B B]
         [--window W|full] [--steps N]

WORKLOAD is a diagonal-stack workload or a general selective-layer one (sel1_*).

The default window is the workload's first.  Inputs are the workload's seeded synthetic
inputs (synth.make_inputs), resized; every step is adj_fwd_scan per layer, adj_loss_mse,
then adj_bwd_* and adj_param_grad per layer, as in the benchmark.  Launch order of one
step of a one-layer bf16 workload: weight prep, proj_in, fwd_scan, proj_out, loss,
cot_proj, [win_scan], bwd_scan, dW_in, colsum, dW_o, param_reduce.
"""
from __future__ import annotations

import argparse

import torch

from . import build, lib, synth
from .stack import AdjStack


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("workload")
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--K", type=int, default=None)
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--window", default=None)
    ap.add_argument("--steps", type=int, default=1)
    a = ap.parse_args(argv)
    build.build()
    if a.workload in synth.SEL_WORKLOADS:
        return sel_main(a)
    w = synth.workload(a.workload)
    inputs = synth.make_inputs(w, T=a.T, K=a.K, B=a.B)
    window = w.windows[0] if a.window is None else (None if a.window == "full" else int(a.window))
    B, T, P, N, K = (inputs[k] for k in ("B", "T", "P", "N", "K"))
    bf16 = w.x_dtype == "bf16"
    st = AdjStack(B, T, P, N, K, x_bf16=bf16, d_bf16=bf16, Tbar=window)
    st.load(inputs)
    torch.cuda.synchronize()
    n0 = lib.launch_count()
    for _ in range(a.steps):
        st.step(window)
    torch.cuda.synchronize()
    status = st.status()
    print(f"{a.workload} B={B} T={T} P={P} N={N} K={K} window={window}: {a.steps} steps, "
          f"{lib.launch_count() - n0} launches, status {lib.STATUS.get(status, status)}")
    return 0 if status == 0 else 1


def sel_main(a):
    """The general selective layer: launch order of one step: [weight split], sel_proj, the
    forward scan's three launches (aggregates, carries, outputs), loss, [the window scan's
    three], the reverse scan's three, dB/dC sums, dA sum, sel_dW, colsum, param_reduce."""
    from .sel_layer import SelLayer
    w = synth.SEL_WORKLOADS[a.workload]
    inputs = synth.make_sel_inputs(w, T=a.T, B=a.B)
    window = w.windows[0] if a.window is None else (None if a.window == "full" else int(a.window))
    B, T, P, N = (inputs[k] for k in ("B", "T", "P", "N"))
    L = SelLayer(B, T, P, N, x_bf16=w.x_dtype == "bf16", Tbar=window)
    L.load(inputs)
    torch.cuda.synchronize()
    n0 = lib.launch_count()
    for _ in range(a.steps):
        L.step(window)
    torch.cuda.synchronize()
    status = L.status()
    print(f"{a.workload} B={B} T={T} P={P} N={N} window={window}: {a.steps} steps, "
          f"{lib.launch_count() - n0} launches, status {lib.STATUS.get(status, status)}")
    return 0 if status == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
