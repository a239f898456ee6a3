"""Gradient error of truncated adjoint sharding against the full adjoint, over the window
T̄ and the decay rate of the state.

Source: the review page "Adjoint sharding for very long context training of state space
models" ([AS]).  Truncated adjoint sharding keeps, for each token's loss, only the VJPs of
the T̄ most recent states ([AS] Core claim, truncated adjoint sharding).  The page leaves
its accuracy unmeasured ([AS] Referee Report, major comment 4 on Section 4.3) and expects
the right window to depend on how fast the products of A_t decay ([AS] Reading between
the lines).  For the diagonal layer here the decay per token is a_t = sigmoid(x̂ W_a + b_a),
so the gate bias b_a sets it: a ≈ 0.73, 0.88, 0.95, 0.98 for b_a = 1, 2, 3, 4.

``truncation_errors`` runs one layer on the GPU path (``AdjStack``, every step in the
library's kernels) once with the full adjoint and once per window, and reports the relative
Frobenius error of each truncated parameter gradient against the full one.  W_c and W_o do
not depend on the window (their VJPs involve no product of A_t); they are reported as a
check of the run's own reproducibility.

    python -m adjoint_gradients_long_gb300.study --T 16384 --B 4 --P 128 --N 256

``memory_report`` measures the device memory a full-size step of each workload takes through
the library, beside the stored-state counts of ``accounting`` (this library, reverse-mode
differentiation, and reverse mode with activation checkpointing): the page's central claim
is a memory saving over backpropagation ([AS] Referee Report, major comment 3).

    python -m adjoint_gradients_long_gb300.study --memory
"""
from __future__ import annotations

import argparse
import dataclasses
import json

import numpy as np

PARAMS = ("W_a", "W_B", "b_a", "W_c", "W_o")


def rel_err(x: np.ndarray, ref: np.ndarray) -> float:
    den = float(np.linalg.norm(ref))
    return float(np.linalg.norm(x - ref)) / den if den > 0 else float(np.linalg.norm(x))


def truncation_errors(B: int, T: int, P: int, N: int, b_a_values, windows, seed: int = 2024,
                      wa_var: float = 0.01, device="cuda") -> list:
    """One row per (b_a, window): relative gradient errors of the truncated adjoint."""
    import torch
    from . import synth
    from .stack import AdjStack

    base = synth.workload("ssm1_p128")
    rows = []
    for b_a in b_a_values:
        w = dataclasses.replace(base, B=B, T=T, P=P, N=N, b_a=float(b_a), wa_var=wa_var)
        inputs = synth.make_inputs(w, seed=seed)
        short = [W for W in windows if W < T]
        st = AdjStack(B, T, P, N, 1, device=device, Tbar=min(short) if short else None)
        st.load(inputs)
        st.step(None)
        torch.cuda.synchronize()
        full = st.grads_numpy(0)
        a_mean = float(st.a[0].double().mean().item())
        for W in windows:
            st.step(W)
            torch.cuda.synchronize()
            g = st.grads_numpy(0)
            rows.append({"b_a": float(b_a), "a_mean": a_mean, "window": int(W),
                         **{f"err_{p}": rel_err(g[p], full[p]) for p in PARAMS},
                         "a_mean_pow_window": a_mean ** int(W)})
        if st.status() != 0:
            raise RuntimeError("device status after the study run: %d" % st.status())
        del st
        torch.cuda.empty_cache()
    return rows


def memory_report(key: str, window=None, device="cuda", T=None, K=None) -> dict:
    """Device memory of one step of workload `key` (optionally resized) through the library:
    every buffer the stack driver allocates (stored states, residual streams, seeds,
    cotangents, gradients, workspace), measured with the torch allocator after the inputs
    are loaded, and the growth during the step itself (the library allocates nothing, so 0),
    beside the counts of ``accounting``."""
    import torch
    from . import accounting, synth
    from .stack import AdjStack

    w = synth.workload(key)
    T = w.T if T is None else T
    K = w.K if K is None else K
    xb = 2 if w.x_dtype == "bf16" else 4
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated(device)
    st = AdjStack(w.B, T, w.P, w.N, K, x_bf16=xb == 2, d_bf16=xb == 2, device=device,
                  Tbar=window if window is not None and window < T else None)
    st.load(synth.make_inputs(w, T=T, K=K))
    torch.cuda.synchronize()
    held = torch.cuda.memory_allocated(device) - base
    # the stack's own device tensors, byte for byte (the allocator's figure above rounds
    # every allocation up, to 512 bytes or to a whole cached block)
    tensors = []
    for v in vars(st).values():
        for t in (v if isinstance(v, list) else [v]):
            if isinstance(t, torch.Tensor) and t.is_cuda:
                tensors.append(t)
    tensor_bytes = sum(t.untyped_storage().nbytes() for t in tensors if t is not st.ws)
    torch.cuda.reset_peak_memory_stats(device)
    before = torch.cuda.memory_allocated(device)
    st.step(window)
    torch.cuda.synchronize()
    growth = torch.cuda.max_memory_allocated(device) - before
    ok = st.status() == 0
    bufs = accounting.stack_buffer_bytes(w.B, T, K, w.N, w.P, xb, xb)
    out = {"workload": key, "window": window if window is not None else "full", "B": w.B, "T": T, "K": K,
           "P": w.P, "N": w.N, "device_peak_bytes": int(held + growth), "held_bytes": int(held),
           "tensor_bytes": int(tensor_bytes), "tensor_count": len(tensors) - 1,
           "step_growth_bytes": int(growth), "workspace_bytes": int(st.ws_bytes),
           "buffer_bytes": {k: v for k, v in bufs.items() if k != "buffers"}, "buffer_count": bufs["buffers"],
           "stored_bytes": accounting.stored_bytes(w.B, T, K, w.N, w.P, xb),
           "bptt_saved_bytes": accounting.bptt_saved_bytes(w.B, T, K, w.N, w.P, xb),
           "checkpoint_saved_bytes": accounting.checkpoint_saved_bytes(w.B, T, K, w.N, w.P, xb),
           "device_status_ok": ok}
    del st
    torch.cuda.empty_cache()
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--B", type=int, default=4)
    ap.add_argument("--T", type=int, default=16384)
    ap.add_argument("--P", type=int, default=128)
    ap.add_argument("--N", type=int, default=256)
    ap.add_argument("--b-a", type=float, nargs="+", default=[1.0, 2.0, 3.0, 4.0])
    ap.add_argument("--windows", type=int, nargs="+", default=[16, 64, 256, 1024, 2048, 4096])
    ap.add_argument("--seed", type=int, default=2024)
    ap.add_argument("--memory", action="store_true", help="device memory of each workload's step instead")
    args = ap.parse_args(argv)
    from . import build
    build.build()
    if args.memory:
        from . import synth
        for key, w in synth.WORKLOADS.items():
            print(json.dumps(memory_report(key, w.windows[0])), flush=True)
        return
    for row in truncation_errors(args.B, args.T, args.P, args.N, args.b_a, args.windows, seed=args.seed):
        print(json.dumps(row), flush=True)


if __name__ == "__main__":
    main()
