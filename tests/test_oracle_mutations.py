"""Plant plausible mistakes in copies of the C oracle (on the CPU) and check that the
pins catch each of them: a dropped term, a wrong index or sign, a transposed operand."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from oracle import bptt
from adjoint_gradients_long_gb300 import synth
from conftest import rel_fro

SRC = os.path.join(os.path.dirname(oracle.__file__), "adj_oracle.c")

MUTATIONS = {
    "h_i_for_h_im1": ("i > 0 ? hb + (i - 1) * N : NULL", "hb + i * N"),
    "no_sigmoid_slope": ("a_i[n] * (1.0 - a_i[n])", "a_i[n]"),
    "dropped_db_a": ("db_a[n] += s_scratch[n];", ";"),
    "W_o_transposed": ("acc += gyb[t * P + p] * W_o[n * P + p];", "acc += gyb[t * P + p] * W_o[p * N + n];"),
    "gate_index_shift": ("v[n] *= ab[i * 8 + n];", "v[n] *= ab[(i > 0 ? i - 1 : 0) * 8 + n];"),
    "literal_product_short": ("for (int64_t j = i + 1; j <= t; ++j)", "for (int64_t j = i + 1; j < t; ++j)"),
    "dx_sign": ("acc += s_scratch[n] * W_a[p * N + n] + v[n] * W_B[p * N + n];",
                "acc -= s_scratch[n] * W_a[p * N + n] + v[n] * W_B[p * N + n];"),
    "no_gate_in_scan": ("ht[n] = at[n] * (hprev ? hprev[n] : 0.0) + ut[n];",
                        "ht[n] = (hprev ? hprev[n] : 0.0) + ut[n];"),
    "window_off_by_one": ("int64_t lo = t - Tbar + 1;", "int64_t lo = t - Tbar;"),
}


@pytest.fixture(scope="module")
def case():
    d = synth.make_inputs("ssm8_p512", T=20, B=2, P=8, N=8, K=2)
    layers = [{k: np.asarray(v, np.float64) for k, v in W.items()} for W in d["layers"]]
    x, tgt = d["xhat"].astype(np.float64), d["target"].astype(np.float64)
    return layers, x, tgt, bptt.bptt_grad(layers, x, tgt)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, case, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, name
    path_c = tmp_path / "mut.c"
    path_c.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", str(so), str(path_c), "-lm"])
    layers, x, tgt, ref = case
    oracle.use_library(str(so))
    try:
        worst = 0.0
        for mode in (oracle.LITERAL, oracle.AGGREGATED):
            res = oracle.stack_grad(layers, x, tgt, None, mode)
            for k in range(2):
                for nm in bptt.PARAMS:
                    worst = max(worst, rel_fro(res["grads"][k]["d" + nm], ref["grads"][k][nm]))
            # a window of 5 against per-term truncated BPTT
            cache = bptt.forward(layers, x)
            tr, _ = bptt.backward(layers, cache, cache[-1]["y"] - tgt, 5)
            res5 = oracle.stack_grad(layers, x, tgt, 5, mode)
            for k in range(2):
                for nm in bptt.PARAMS:
                    worst = max(worst, rel_fro(res5["grads"][k]["d" + nm], tr[k][nm]))
    finally:
        oracle.use_library(None)
    assert worst > 1e-6, (name, worst)


# ---------------------------------------------------------------- the general selective layer
SEL_SRC = os.path.join(os.path.dirname(oracle.__file__), "sel_oracle.c")

SEL_MUTATIONS = {
    "dropped_input_term": ("ddt[p] += vv * (A[p * N + n] * ab * hp + zr[P + n] * xr[p]);",
                           "ddt[p] += vv * (A[p * N + n] * ab * hp);"),
    "decay_of_the_wrong_token": ("const double *ab = Ab + ri * PN + p * N;",
                                 "const double *ab = Ab + (ri > 0 ? ri - 1 : 0) * PN + p * N;"),
    "literal_product_short": ("for (int64_t j = i + 1; j <= t; ++j) {", "for (int64_t j = i + 1; j < t; ++j) {"),
    "no_softplus_slope": ("dz[r * Z + p] = ddt[r * P + p] * sigmoid(z[r * Z + p]);", "dz[r * Z + p] = ddt[r * P + p];"),
    "B_and_C_swapped": ("v[p * N + n] = gy[rt * P + p] * z[rt * Z + P + N + n] * prod;",
                        "v[p * N + n] = gy[rt * P + p] * z[rt * Z + P + n] * prod;"),
    "B_and_C_swapped_agg": ("vv[n] = gy[rt * P + p] * z[rt * Z + P + N + n];", "vv[n] = gy[rt * P + p] * z[rt * Z + P + n];"),
    "dA_without_step": ("dA[p * N + n] += vv * dt * ab * hp;", "dA[p * N + n] += vv * ab * hp;"),
    "window_off_by_one": ("int64_t lo = t - W + 1;", "int64_t lo = t - W;"),
    "h_i_for_h_im1": ("i > 0 ? h + (ri - 1) * PN : NULL", "h + ri * PN"),
    "bias_on_the_wrong_columns": ("zr[j] = acc + (j < P ? b_dt[j] : 0.0);", "zr[j] = acc + (j < N ? b_dt[j] : 0.0);"),
    "dropped_direct_input_term": ("if (dx) dx[p] += vv * dt * zr[P + n];", ";"),
    "residual_from_xhat": ("*rr = (xres ? xres : x) + r * P;", "*rr = x + r * P;"),
    "projection_transposed": ("acc += dz[r * Z + j] * W_in[p * Z + j];", "acc += dz[r * Z + j] * W_in[(j % P) * Z + p];"),
}


@pytest.fixture(scope="module")
def sel_case():
    from oracle import sel_bptt
    d = synth.make_sel_inputs("sel1_p16", T=18, B=2, P=4, N=3)
    W = {k: d[k].astype(np.float64) for k in ("W_in", "b_dt", "A")}
    W["b_dt"] = W["b_dt"] + 4.0
    W2 = {k: synth.make_sel_inputs("sel1_p16", T=18, B=2, P=4, N=3, seed=99)[k].astype(np.float64)
          for k in ("W_in", "b_dt", "A")}
    W2["b_dt"] = W2["b_dt"] + 4.0
    x, tgt = d["xhat"].astype(np.float64), d["target"].astype(np.float64)
    return (W, x, tgt, sel_bptt.bptt_grad(W, x, tgt), sel_bptt.bptt_grad(W, x, tgt, 5), [W, W2],
            sel_bptt.stack_bptt_grad([W, W2], x, tgt, 5))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(SEL_MUTATIONS))
def test_selective_mutation_is_caught(name, sel_case, tmp_path):
    from oracle import selective as sel
    old, new = SEL_MUTATIONS[name]
    src = open(SEL_SRC).read()
    assert src.count(old) >= 1, name
    path_c = tmp_path / "mut.c"
    path_c.write_text(src.replace(old, new))
    so = sel.build(force=True, src=str(path_c), out=str(tmp_path / "libmut.so"))
    W, x, tgt, ref_full, ref5, layers, ref_stack = sel_case
    sel.use_library(so)
    try:
        worst = 0.0
        for mode in (sel.LITERAL, sel.AGGREGATED):
            for Tbar, ref in ((None, ref_full), (5, ref5)):
                st = sel.forward(W, x)
                g = sel.grad(W, st, st["y"] - tgt, Tbar, mode)
                for k in ("W_in", "b_dt", "A"):
                    worst = max(worst, rel_fro(g["d" + k], ref["d" + k]))
            # a 2-layer stack (the input gradient and the residual input) against its BPTT
            res = sel.stack_grad(layers, x, tgt, 5, mode)
            for kk in range(2):
                for k in ("W_in", "b_dt", "A"):
                    worst = max(worst, rel_fro(res["grads"][kk]["d" + k], ref_stack[kk]["d" + k]))
    finally:
        sel.use_library(None)
    assert worst > 1e-6, (name, worst)
