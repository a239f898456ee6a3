"""The general selective layer's fp64 oracle pinned to things other than itself: an
independent step-by-step BPTT, per-term truncated BPTT, the complex step and central
differences, closed forms of special cases, the adjoint recursion, and the pair count.

Source: the review page "Adjoint sharding for very long context training of state space
models" ([AS]): the general form h_t = A_t h_{t-1} + B_t xhat_t, y_t = C_t h_t
(Circularity Check, assumptions), the gradient as a sum of independent VJPs over pairs
(Core claim, Proposition 2), its truncation to a window (Core claim, last sentence) and
the claim that it equals backpropagation (The reading; If this is right).
"""
import numpy as np
import pytest

from adjoint_gradients_long_gb300 import synth
from oracle import sel_bptt, selective as sel


def tiny(T=24, B=1, P=4, N=3, seed=7):
    d = synth.make_sel_inputs("sel1_p16", T=T, B=B, P=P, N=N, seed=seed)
    W = {k: d[k].astype(np.float64) for k in ("W_in", "b_dt", "A")}
    # larger steps than the workload's so every product term matters at this length
    W["b_dt"] = W["b_dt"] + 4.0
    return W, d["xhat"].astype(np.float64), d["target"].astype(np.float64)


def rel(a, b):
    return float(np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-300))


def oracle_grad(W, x, tgt, Tbar=None, mode=sel.AGGREGATED, want_mu=False):
    st = sel.forward(W, x)
    _, gy = sel.loss_and_cotangent(st["y"], tgt)
    return sel.grad(W, st, gy, Tbar, mode, want_mu), st, gy


def test_forward_matches_bptt_forward():
    W, x, tgt = tiny()
    st = sel.forward(W, x)
    c = sel_bptt.forward(W, x)
    assert rel(st["h"], c["h"]) < 1e-13 and rel(st["y"], c["y"]) < 1e-13 and rel(st["z"], c["z"]) < 1e-13


def test_literal_full_equals_bptt():
    W, x, tgt = tiny()
    g, _, _ = oracle_grad(W, x, tgt, mode=sel.LITERAL)
    ref = sel_bptt.bptt_grad(W, x, tgt)
    for k in ("dW_in", "db_dt", "dA", "dz"):
        assert rel(g[k], ref[k]) < 1e-11, k


@pytest.mark.parametrize("Tbar", [None, 1, 5, 23, 24, 100])
def test_aggregated_equals_literal(Tbar):
    W, x, tgt = tiny(T=20, B=2)
    a, _, _ = oracle_grad(W, x, tgt, Tbar, sel.AGGREGATED, want_mu=True)
    l, _, _ = oracle_grad(W, x, tgt, Tbar, sel.LITERAL, want_mu=True)
    for k in ("dW_in", "db_dt", "dA", "dz", "mu"):
        assert rel(a[k], l[k]) < 1e-12, (k, Tbar)
    assert a["vjp_count"] == l["vjp_count"]


@pytest.mark.parametrize("Tbar", [1, 4, 9])
def test_truncated_equals_per_term_tbptt(Tbar):
    W, x, tgt = tiny(T=22, B=2)
    g, _, _ = oracle_grad(W, x, tgt, Tbar)
    ref = sel_bptt.bptt_grad(W, x, tgt, Tbar)
    for k in ("dW_in", "db_dt", "dA", "dz"):
        assert rel(g[k], ref[k]) < 1e-11, (k, Tbar)


def test_complex_step():
    W, x, tgt = tiny(T=12, P=3, N=2)
    g, _, _ = oracle_grad(W, x, tgt)
    cs = sel_bptt.complex_step_grad(W, x, tgt)
    for k in ("W_in", "b_dt", "A"):
        assert rel(g["d" + k], cs[k]) < 1e-10, k


def test_central_differences():
    W, x, tgt = tiny(T=10, P=2, N=2)
    g, _, _ = oracle_grad(W, x, tgt)
    cd = sel_bptt.central_diff_grad(W, x, tgt)
    for k in ("W_in", "b_dt", "A"):
        assert rel(g["d" + k], cd[k]) < 1e-7, k


def test_forward_closed_form_without_decay():
    """A = 0: no decay, every h is the running sum of dt B x."""
    W, x, _ = tiny(T=16)
    W["A"] = np.zeros_like(W["A"])
    st = sel.forward(W, x)
    P, N = W["A"].shape
    z = x @ W["W_in"]
    z[..., :P] += W["b_dt"]
    dt = np.log1p(np.exp(z[..., :P]))
    u = dt[..., :, None] * z[..., None, P:P + N] * x[..., :, None]
    assert rel(st["h"], np.cumsum(u, axis=1)) < 1e-13


def test_full_window_mu_is_the_adjoint_recursion():
    """Full window: mu_i = gy_i C_i + Abar_{i+1} mu_{i+1} ([AS] What carries the argument,
    Proposition 1), mu_T = 0."""
    W, x, tgt = tiny(T=18, B=2)
    g, st, gy = oracle_grad(W, x, tgt, want_mu=True)
    P, N = W["A"].shape
    z = st["z"]
    Ab = np.exp(np.log1p(np.exp(z[..., :P]))[..., :, None] * W["A"])
    mu = np.zeros_like(g["mu"])
    nxt = np.zeros_like(mu[:, 0])
    for i in range(x.shape[1] - 1, -1, -1):
        nxt = gy[:, i, :, None] * z[:, i, None, P + N:] + (Ab[:, i + 1] * nxt if i + 1 < x.shape[1] else 0.0)
        mu[:, i] = nxt
    assert rel(g["mu"], mu) < 1e-13


def test_window_one_keeps_only_the_diagonal_pairs():
    """Tbar = 1: mu_i = gy_i C_i, no product at all."""
    W, x, tgt = tiny(T=14)
    g, st, gy = oracle_grad(W, x, tgt, Tbar=1, want_mu=True)
    P, N = W["A"].shape
    assert rel(g["mu"], gy[..., :, None] * st["z"][..., None, P + N:]) < 1e-15


@pytest.mark.parametrize("T,Tbar", [(30, None), (30, 7), (30, 30), (5, 64)])
def test_vjp_count(T, Tbar):
    W, x, tgt = tiny(T=T)
    g, _, _ = oracle_grad(W, x, tgt, Tbar)
    Wn = T if Tbar is None else min(Tbar, T)
    assert g["vjp_count"] == sum(min(t + 1, Wn) for t in range(T))


def test_dC_does_not_depend_on_the_window():
    W, x, tgt = tiny(T=20)
    P, N = W["A"].shape
    full, _, _ = oracle_grad(W, x, tgt)
    part, _, _ = oracle_grad(W, x, tgt, Tbar=3)
    assert rel(part["dz"][..., P + N:], full["dz"][..., P + N:]) < 1e-15
    assert rel(part["dz"][..., :P + N], full["dz"][..., :P + N]) > 1e-6


def test_sequences_are_independent():
    """Two sequences in one batch give the sums of their separate gradients."""
    W, x, tgt = tiny(T=12, B=2)
    both, _, _ = oracle_grad(W, x, tgt, Tbar=5)
    a, _, _ = oracle_grad(W, x[:1], tgt[:1], Tbar=5)
    b, _, _ = oracle_grad(W, x[1:], tgt[1:], Tbar=5)
    for k in ("dW_in", "db_dt", "dA"):
        assert rel(both[k], a[k] + b[k]) < 1e-13, k


@pytest.mark.parametrize("Tbar", [None, 6])
def test_sampled_rows_equal_the_whole_gradient(Tbar):
    """The sampled-row evaluation (for sequences too long for the whole sum) gives the
    same dz rows as the aggregated gradient."""
    W, x, tgt = tiny(T=30, B=2)
    g, _, _ = oracle_grad(W, x, tgt, Tbar)
    rows = [(0, 0), (0, 17), (1, 29), (1, 3)]
    got = sel.dz_rows(W, x, tgt, rows, Tbar)
    for s, (b, t) in enumerate(rows):
        assert rel(got[s], g["dz"][b, t]) < 1e-12, (b, t)


# ---------------------------------------------------------------- residual stacks of selective layers
def tiny_stack(K=3, T=16, B=2, P=4, N=3):
    out = []
    for k in range(K):
        W, x, tgt = tiny(T=T, B=B, P=P, N=N, seed=11 + k)
        out.append(W)
    _, x, tgt = tiny(T=T, B=B, P=P, N=N, seed=7)
    return out, x, tgt


def test_input_gradient_is_bptt():
    """A lone layer's input-path cotangent (the projection and the input term) against BPTT."""
    W, x, tgt = tiny(T=18, B=2)
    g, _, _ = oracle_grad(W, x, tgt)
    ref = sel_bptt.bptt_grad(W, x, tgt)
    assert rel(g["dxhat"], ref["dxhat"]) < 1e-11


@pytest.mark.parametrize("Tbar", [None, 5])
def test_stack_equals_bptt(Tbar):
    layers, x, tgt = tiny_stack()
    res = sel.stack_grad(layers, x, tgt, Tbar)
    ref = sel_bptt.stack_bptt_grad(layers, x, tgt, Tbar)
    for k in range(len(layers)):
        for nm in ("W_in", "b_dt", "A"):
            assert rel(res["grads"][k]["d" + nm], ref[k]["d" + nm]) < 1e-10, (k, nm, Tbar)


def test_stack_complex_step():
    """Every layer's parameters of a 2-layer stack against the complex step on the loss."""
    layers, x, tgt = tiny_stack(K=2, T=10, B=1, P=3, N=2)
    res = sel.stack_grad(layers, x, tgt)
    for k in range(2):
        for nm in ("W_in", "b_dt", "A"):
            cs = sel_bptt.stack_complex_step_grad(layers, x, tgt, k, nm)
            assert rel(res["grads"][k]["d" + nm], cs) < 1e-9, (k, nm)


def test_stack_of_one_is_the_layer():
    W, x, tgt = tiny(T=12, B=2)
    res = sel.stack_grad([W], x, tgt, 4)
    g, _, _ = oracle_grad(W, x, tgt, 4)
    for k in ("dW_in", "db_dt", "dA", "dz"):
        assert rel(res["grads"][0][k], g[k]) < 1e-15, k
