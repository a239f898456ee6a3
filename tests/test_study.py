"""The truncation-error study: gradient error of truncated adjoint sharding against the
full adjoint over the window and the decay rate.

CPU: with W_a = 0 the decay a = sigmoid(b_a) is the same for every token, so the adjoint's
truncation error is a geometric tail, |mu_i - mu_i^W| <= a^W max|g c| / (1 - a), and it is
zero once the window covers the sequence; the oracle's truncated adjoint must obey both.
GPU: the study's errors, from the CUDA path, match the same errors computed by the oracle.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from adjoint_gradients_long_gb300 import synth
from adjoint_gradients_long_gb300.study import PARAMS, rel_err


def _inputs(b_a, wa_var, T=96, B=2, P=8, N=16, seed=77):
    w = dataclasses.replace(synth.workload("ssm1_p128"), B=B, T=T, P=P, N=N, b_a=b_a, wa_var=wa_var)
    return synth.make_inputs(w, seed=seed)


@pytest.mark.parametrize("b_a", [0.5, 2.0])
def test_oracle_truncation_error_is_a_geometric_tail(b_a):
    inp = _inputs(b_a, 0.0)
    W = {k: np.asarray(v, np.float64) for k, v in inp["layers"][0].items()}
    st = oracle.layer_forward(W, inp["xhat"])
    _, gy = oracle.loss_and_cotangent(st["y"], inp["target"])
    a = 1.0 / (1.0 + np.exp(-b_a))
    assert np.allclose(st["a"], a, rtol=0, atol=1e-15)        # W_a = 0: one decay rate
    full = oracle.layer_grad(W, st, gy, None)
    e_max = np.abs((gy @ W["W_o"].T) * st["c"]).max()
    T = inp["T"]
    for win in (1, 4, 16, 40):
        tr = oracle.layer_grad(W, st, gy, win)
        err = np.abs(tr["mu"] - full["mu"]).max()
        bound = a ** win * e_max / (1.0 - a)
        assert err <= bound * (1 + 1e-12), (win, err, bound)
        assert err > 0.0
    same = oracle.layer_grad(W, st, gy, T)
    for p in PARAMS:
        assert rel_err(same["d" + p], full["d" + p]) <= 1e-14, p


@pytest.mark.gpu
def test_study_matches_oracle_errors():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adjoint_gradients_long_gb300 import build
    from adjoint_gradients_long_gb300.study import truncation_errors
    build.build()
    B, T, P, N, seed = 2, 512, 16, 32, 5
    windows = (8, 32, 128)
    rows = truncation_errors(B, T, P, N, (1.0, 3.0), windows, seed=seed)
    assert len(rows) == 6
    for row in rows:
        w = dataclasses.replace(synth.workload("ssm1_p128"), B=B, T=T, P=P, N=N, b_a=row["b_a"], wa_var=0.01)
        inp = synth.make_inputs(w, seed=seed)
        W = {k: np.asarray(v, np.float64) for k, v in inp["layers"][0].items()}
        full = oracle.stack_grad([W], inp["xhat"], inp["target"], None)["grads"][0]
        tr = oracle.stack_grad([W], inp["xhat"], inp["target"], row["window"])["grads"][0]
        for p in ("W_a", "W_B", "b_a"):
            ref = rel_err(tr["d" + p], full["d" + p])
            # fp32 gradients: agree with the fp64 error to 2% of it, above a 1e-5 floor
            assert abs(row["err_" + p] - ref) <= 0.02 * ref + 1e-5, (row, p, ref)
        for p in ("W_c", "W_o"):
            assert row["err_" + p] <= 1e-5, (row, p)


def test_storage_counts_relations():
    """Stored-state counts: a stack of one layer gains nothing from checkpointing (it keeps
    its input and the whole layer); a deep stack keeps less with it than reverse mode does;
    reverse mode saves the product c . h beyond this library's a, c, h, xhat."""
    from adjoint_gradients_long_gb300 import accounting as A
    B, T, N, P = 2, 1000, 256, 128
    for xb in (2, 4):
        assert A.checkpoint_saved_bytes(B, T, 1, N, P, xb) == B * T * P * 4 + A.bptt_saved_bytes(B, T, 1, N, P, xb)
        assert A.checkpoint_saved_bytes(B, T, 100, N, P, xb) < A.bptt_saved_bytes(B, T, 100, N, P, xb)
        assert A.checkpoint_saved_bytes(B, T, 100, N, P, xb, segment=100) == (
            B * T * P * 4 + A.bptt_saved_bytes(B, T, 100, N, P, xb))
        for K in (1, 8, 100):
            assert A.bptt_saved_bytes(B, T, K, N, P, xb) - A.stored_bytes(B, T, K, N, P, xb) == B * T * K * N * 4


@pytest.mark.gpu
@pytest.mark.parametrize("key,T,K,window", [("ssm8_p512", 1024, 3, 256), ("ssm1_p128", 2048, 1, None)])
def test_step_memory_is_the_counted_buffers(key, T, K, window):
    """The device memory one step holds is the buffers the stack driver allocates, exactly as
    counted from the shapes (accounting.stack_buffer_bytes), plus the caller-sized
    workspace; the step itself allocates nothing; what is kept between the passes is at
    least the stored-state count."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adjoint_gradients_long_gb300 import build, study
    build.build()
    r = study.memory_report(key, window, T=T, K=K)
    assert r["device_status_ok"]
    # every buffer the stack holds, byte for byte, is one the count names
    assert r["tensor_bytes"] == sum(r["buffer_bytes"].values()), r
    assert r["tensor_count"] == r["buffer_count"], r
    # the allocator holds those plus the workspace (rounded up); the step allocates nothing
    assert r["held_bytes"] >= r["tensor_bytes"] + r["workspace_bytes"], r
    assert r["step_growth_bytes"] == 0, r
    assert r["held_bytes"] >= r["stored_bytes"]
