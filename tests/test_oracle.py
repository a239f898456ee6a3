"""Pins for the fp64 oracle against things other than itself (CPU only).

Source: the review page "Adjoint sharding for very long context training of state
space models" ([AS]).  Each test names what pins the oracle:
  * independent step-by-step BPTT, complex-step and central finite differences
    -- the full adjoint equals backpropagation ([AS] The reading; If this is right);
  * brute-force per-term truncated BPTT -- truncation to the last Tbar states
    ([AS] Core claim, last sentence);
  * closed forms of the scan and of the adjoint sum at constant a;
  * the VJP counts O(T^2) / O(T Tbar) ([AS] Core claim);
  * per-token independence of the VJP sums ([AS] Core claim, first sentence);
  * the blockwise truncation identity the CUDA path is built on;
  * the Section 4.5 storage figures printed on the page (tests/golden).
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import bptt
from adjoint_gradients_long_gb300 import synth, accounting
from conftest import rel_fro

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(key="ssm1_p16", **kw):
    d = synth.make_inputs(key, **kw)
    layers = [{k: np.asarray(v, np.float64) for k, v in W.items()} for W in d["layers"]]
    return layers, d["xhat"].astype(np.float64), d["target"].astype(np.float64)


def _check(og, ref, tol, names=("W_a", "W_B", "W_c", "b_a", "W_o")):
    for nm in names:
        e = rel_fro(og["d" + nm], ref[nm])
        assert e <= tol, (nm, e)


# ---------------------------------------------------------------- full adjoint == BPTT

def test_literal_full_equals_bptt_ssm1_p16():
    """Full workload ssm1_p16 (P=16, N=8, T=256), every lambda_{t,i} by explicit product."""
    layers, x, tgt = _inputs()
    res = oracle.stack_grad(layers, x, tgt, None, oracle.LITERAL)
    ref = bptt.bptt_grad(layers, x, tgt)
    assert abs(res["loss"] - ref["loss"]) <= 1e-12 * abs(ref["loss"])
    _check(res["grads"][0], ref["grads"][0], 1e-9)
    assert rel_fro(res["gx"], ref["gx"]) <= 1e-9
    assert res["vjp_count"] == 256 * 257 // 2


@pytest.mark.parametrize("Tbar", [None, 1, 5, 37, 64])
def test_aggregated_equals_literal(Tbar):
    layers, x, tgt = _inputs(T=64, B=2)
    lit = oracle.stack_grad(layers, x, tgt, Tbar, oracle.LITERAL)
    agg = oracle.stack_grad(layers, x, tgt, Tbar, oracle.AGGREGATED)
    _check(agg["grads"][0], {k: lit["grads"][0]["d" + k] for k in bptt.PARAMS}, 1e-12)
    assert rel_fro(agg["grads"][0]["mu"], lit["grads"][0]["mu"]) <= 1e-12
    assert agg["vjp_count"] == lit["vjp_count"]


def test_stack_full_equals_bptt():
    """K=2 residual layers: the total-cotangent reading of Proposition 3 equals BPTT."""
    layers, x, tgt = _inputs("ssm8_p512", T=24, B=2, P=8, N=8, K=2)
    res = oracle.stack_grad(layers, x, tgt, None, oracle.AGGREGATED)
    ref = bptt.bptt_grad(layers, x, tgt)
    for k in range(2):
        _check(res["grads"][k], ref["grads"][k], 1e-9)
    assert rel_fro(res["gx"], ref["gx"]) <= 1e-9


# ---------------------------------------------------------------- derivative checks

def test_complex_step_single_layer():
    layers, x, tgt = _inputs(T=32)
    res = oracle.stack_grad(layers, x, tgt, None, oracle.LITERAL)
    cs = bptt.complex_step_grad(layers, x, tgt)
    _check(res["grads"][0], cs[0], 1e-9)


def test_complex_step_stack():
    layers, x, tgt = _inputs("ssm4_p2048", T=16, B=1, P=8, N=8, K=2)
    res = oracle.stack_grad(layers, x, tgt, None, oracle.AGGREGATED)
    cs = bptt.complex_step_grad(layers, x, tgt)
    for k in range(2):
        _check(res["grads"][k], cs[k], 1e-9)


def test_central_differences_stack():
    layers, x, tgt = _inputs("ssm8_p512", T=16, B=1, P=8, N=8, K=2)
    res = oracle.stack_grad(layers, x, tgt, None, oracle.AGGREGATED)
    fd = bptt.central_diff_grad(layers, x, tgt)
    for k in range(2):
        _check(res["grads"][k], fd[k], 1e-9)


# ---------------------------------------------------------------- truncated adjoint

@pytest.mark.parametrize("Tbar", [1, 3, 7, 16, 40])
def test_truncated_equals_per_term_tbptt(Tbar):
    layers, x, tgt = _inputs("ssm8_p512", T=40, B=2, P=8, N=8, K=2)
    res = oracle.stack_grad(layers, x, tgt, Tbar, oracle.AGGREGATED)
    cache = bptt.forward(layers, x)
    r = cache[-1]["y"] - tgt
    grads, gx = bptt.backward(layers, cache, r, Tbar)
    for k in range(2):
        _check(res["grads"][k], grads[k], 1e-12)
        assert rel_fro(res["grads"][k]["mu"], grads[k]["mu"]) <= 1e-12
    assert rel_fro(res["gx"], gx) <= 1e-12


def test_truncated_edge_windows():
    layers, x, tgt = _inputs(T=50, B=2)
    full = oracle.stack_grad(layers, x, tgt, None)
    big = oracle.stack_grad(layers, x, tgt, 50)
    bigger = oracle.stack_grad(layers, x, tgt, 10 ** 6)
    for nm in ("dW_a", "dW_B", "dW_c", "db_a", "dW_o", "mu"):
        assert np.array_equal(big["grads"][0][nm], full["grads"][0][nm])
        assert np.array_equal(bigger["grads"][0][nm], full["grads"][0][nm])
    one = oracle.stack_grad(layers, x, tgt, 1)
    st = one["states"][0]
    g = one["gy"][0] @ layers[0]["W_o"].T
    assert rel_fro(one["grads"][0]["mu"], g * st["c"]) <= 1e-14


@pytest.mark.parametrize("T,Tbar", [(64, None), (64, 1), (64, 10), (64, 64), (37, 8)])
def test_vjp_count(T, Tbar):
    layers, x, tgt = _inputs(T=T, B=3)
    res = oracle.stack_grad(layers, x, tgt, Tbar, oracle.AGGREGATED)
    w = T if Tbar is None else Tbar
    assert res["vjp_count"] == 3 * sum(min(t, w) for t in range(1, T + 1))


# ---------------------------------------------------------------- closed forms

def _const_layer(P=8, N=8, b=2.0):
    rng = np.random.default_rng(7)
    return dict(W_a=np.zeros((P, N)), W_B=rng.standard_normal((P, N)), W_c=rng.standard_normal((P, N)),
                b_a=np.full(N, b) + 0.1 * np.arange(N), W_o=rng.standard_normal((N, P)))


def test_forward_closed_form_constant_gate():
    """W_a = 0 and a constant input: a = sigmoid(b_a), u constant, h_t = u (1 - a^t) / (1 - a)."""
    W = _const_layer()
    T = 30
    x = np.tile(np.random.default_rng(3).standard_normal(8), (1, T, 1))
    st = oracle.layer_forward(W, x)
    a = 1.0 / (1.0 + np.exp(-W["b_a"]))
    u = x[0, 0] @ W["W_B"]
    t = np.arange(1, T + 1)[:, None]
    assert rel_fro(st["h"][0], u * (1 - a ** t) / (1 - a)) <= 1e-13
    assert rel_fro(st["a"][0], np.broadcast_to(a, (T, 8))) <= 1e-15


def test_adjoint_closed_form_constant_gate():
    """Constant a and constant e = g c: mu_i = e (1 - a^{T-i+1}) / (1 - a) (1-based i);
    truncated to Tbar: mu_i = e (1 - a^{min(Tbar, T-i+1)}) / (1 - a)."""
    W = _const_layer()
    T = 30
    x = np.tile(np.random.default_rng(3).standard_normal(8), (1, T, 1))
    st = oracle.layer_forward(W, x)
    gy = np.tile(np.random.default_rng(4).standard_normal(8), (1, T, 1))
    a = 1.0 / (1.0 + np.exp(-W["b_a"]))
    e = (gy[0, 0] @ W["W_o"].T) * (x[0, 0] @ W["W_c"])
    i = np.arange(1, T + 1)[:, None]
    full = oracle.layer_grad(W, st, gy, None)
    assert rel_fro(full["mu"][0], e * (1 - a ** (T - i + 1)) / (1 - a)) <= 1e-13
    tr = oracle.layer_grad(W, st, gy, 7)
    assert rel_fro(tr["mu"][0], e * (1 - a ** np.minimum(7, T - i + 1)) / (1 - a)) <= 1e-13


# ---------------------------------------------------------------- independence of the VJP sums

def test_per_token_independence():
    """The gradient is the sum over t of the gradients of the single-token losses l_t."""
    layers, x, tgt = _inputs(T=20, B=1)
    W = layers[0]
    st = oracle.layer_forward(W, x)
    gy = st["y"] - tgt
    tot = oracle.layer_grad(W, st, gy, None)
    acc = {k: 0.0 for k in ("dW_a", "dW_B", "dW_c", "db_a", "dW_o")}
    for t in range(20):
        gt = np.zeros_like(gy)
        gt[:, t] = gy[:, t]
        part = oracle.layer_grad(W, st, gt, None)
        for k in acc:
            acc[k] = acc[k] + part[k]
    for k in acc:
        assert rel_fro(acc[k], tot[k]) <= 1e-13


def test_top_cotangent_reading_differs_for_stacks():
    layers, x, tgt = _inputs("ssm8_p512", T=16, B=1, P=8, N=8, K=2)
    tot = oracle.stack_grad(layers, x, tgt, None, cotangent="total")
    top = oracle.stack_grad(layers, x, tgt, None, cotangent="top")
    assert np.array_equal(tot["grads"][1]["dW_a"], top["grads"][1]["dW_a"])
    assert rel_fro(top["grads"][0]["dW_B"], tot["grads"][0]["dW_B"]) > 1e-3
    l1, x1, t1 = _inputs(T=16)
    a1 = oracle.stack_grad(l1, x1, t1, None, cotangent="total")
    b1 = oracle.stack_grad(l1, x1, t1, None, cotangent="top")
    assert np.array_equal(a1["grads"][0]["dW_B"], b1["grads"][0]["dW_B"])


# ---------------------------------------------------------------- blockwise truncation identity

def _blockwise_mu(a, e, Tbar):
    """mu^Tbar_i = S_i + Q_i R(min(i+Tbar-1, T-1)) with blocks of Tbar tokens (0-based rows):
    S: reverse scan inside the block, Q_i = prod_{j=i+1}^{s} a_j up to the next block start s,
    R(m) = sum_{t=s}^{m} e_t prod_{j=s+1}^{t} a_j over the next block."""
    B, T, N = a.shape
    mu = np.zeros_like(e)
    for s0 in range(0, T, Tbar):
        s = s0 + Tbar
        R = np.zeros((B, T + 1, N))
        if s < T:
            P = np.ones((B, N))
            run = np.zeros((B, N))
            for m in range(s, min(s + Tbar, T)):
                if m > s:
                    P = P * a[:, m]
                run = run + e[:, m] * P
                R[:, m] = run
        S = np.zeros((B, N))
        Q = a[:, s] if s < T else np.zeros((B, N))
        for i in range(min(s, T) - 1, s0 - 1, -1):
            if i < min(s, T) - 1:
                S = S * a[:, i + 1]
                Q = Q * a[:, i + 1]
            S = S + e[:, i]
            m = min(i + Tbar - 1, T - 1)
            mu[:, i] = S + (Q * R[:, m] if m >= s else 0.0)
    return mu


@pytest.mark.parametrize("T,Tbar", [(64, 8), (61, 8), (64, 64), (64, 1), (50, 13), (64, 100)])
def test_blockwise_truncation_identity(T, Tbar):
    layers, x, tgt = _inputs(T=T, B=2)
    W = layers[0]
    st = oracle.layer_forward(W, x)
    gy = st["y"] - tgt
    ref = oracle.layer_grad(W, st, gy, Tbar)["mu"]
    e = (gy @ W["W_o"].T) * st["c"]
    assert rel_fro(_blockwise_mu(st["a"], e, Tbar), ref) <= 1e-13
    # the subtraction form, exact in fp64: mu^Tbar_i = mu_i - prod_{j=i+1}^{i+Tbar} a_j mu_{i+Tbar}
    full = oracle.layer_grad(W, st, gy, None)["mu"]
    sub = full.copy()
    for i in range(T - Tbar if Tbar < T else 0):
        sub[:, i] -= np.prod(st["a"][:, i + 1:i + Tbar + 1], axis=1) * full[:, i + Tbar]
    assert rel_fro(sub, ref) <= 1e-10


# ---------------------------------------------------------------- the pages' printed figures

def test_section45_storage_figures():
    g = json.load(open(os.path.join(GOLDEN, "section45_storage.json")))
    i, p = g["inputs"], g["printed"]
    vals = accounting.paper_state_values(i["T"], i["K"], i["N"], i["P"])
    assert float(f"{vals:.{p['values_sig_figs'] - 1}e}") == p["values"]
    gb = vals * i["bytes_per_value"] / 1e9
    assert round(gb) == p["total_GB"]
    assert round(gb / i["gpus"]) == p["per_gpu_GB"]


# ---------------------------------------------------------------- normalised stack inputs

def test_normalized_inputs_have_unit_rms():
    layers, x, tgt = _inputs("ssm8_p512", T=20, B=2, P=16, N=8, K=3)
    states = oracle.stack_forward(layers, x)
    for st in states[1:]:
        rms = np.sqrt(np.mean(st["xhat"] ** 2, axis=-1))
        assert np.allclose(rms, 1.0, atol=1e-6)


def test_normalize_vjp_mutation_is_caught(monkeypatch):
    """Drop the projection term of the normalisation VJP: BPTT must disagree."""
    layers, x, tgt = _inputs("ssm8_p512", T=12, B=1, P=8, N=8, K=2)
    ref = bptt.bptt_grad(layers, x, tgt)
    monkeypatch.setattr(oracle.oracle, "normalize_vjp", lambda xh, r, dx: dx / r)
    bad = oracle.stack_grad(layers, x, tgt, None)
    assert rel_fro(bad["grads"][0]["dW_B"], ref["grads"][0]["W_B"]) > 1e-6
