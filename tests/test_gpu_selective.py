"""GPU parity of the general selective layer: the CUDA path (through the C ABI) against the
fp64 CPU oracle (oracle/sel_oracle.c) on the same seeded inputs.

Tolerances, relative Frobenius error per tensor: 1e-4 where every stored operand is fp32;
with bf16 storage (xhat, W_in, and dz, the parameter GEMM's operand) 2e-2 on what passes
through a bf16 operand (dz, dW_in, db_dt) and 1e-4 on the rest (z, h, y, dA: fp32
products of bf16-exact inputs).

Source: the review page "Adjoint sharding for very long context training of state space
models" ([AS]): the general form h_t = A_t h_{t-1} + B_t xhat_t, y_t = C_t h_t
(Circularity Check, assumptions) and its gradient as a sum of VJPs over token pairs,
full or truncated (Core claim).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from adjoint_gradients_long_gb300 import synth  # noqa: E402
from conftest import rel_fro  # noqa: E402
from oracle import selective as sel  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adjoint_gradients_long_gb300 import build
    build.build()


def run(inputs, Tbar, bf16):
    from adjoint_gradients_long_gb300.sel_layer import SelLayer
    B, T, P, N = (inputs[k] for k in ("B", "T", "P", "N"))
    L = SelLayer(B, T, P, N, x_bf16=bf16, Tbar=Tbar)
    L.load(inputs)
    L.step(Tbar)
    torch.cuda.synchronize()
    assert L.status() == 0
    return L


def reference(inputs, Tbar):
    W = {k: np.asarray(inputs[k], np.float64) for k in ("W_in", "b_dt", "A")}
    st = sel.forward(W, inputs["xhat"])
    loss, gy = sel.loss_and_cotangent(st["y"], inputs["target"])
    g = sel.grad(W, st, gy, Tbar)
    return st, loss, g


def compare(inputs, Tbar, bf16):
    L = run(inputs, Tbar, bf16)
    st, loss, g = reference(inputs, Tbar)
    P = inputs["P"]
    z = L.z.double().cpu().numpy()
    z[..., :P] += np.asarray(inputs["b_dt"], np.float64)
    lo, hi = 1e-4, (2e-2 if bf16 else 1e-4)
    errs = {
        "z": (rel_fro(z, st["z"]), lo),
        "h": (rel_fro(L.h.double().cpu().numpy(), st["h"]), lo),
        "y": (rel_fro(L.y.double().cpu().numpy(), st["y"]), lo),
        "loss": (abs(float(L.loss.item()) - loss) / abs(loss), lo),
        "dz": (rel_fro(L.dz.double().cpu().numpy(), g["dz"]), hi),
        "dA": (rel_fro(L.dA.double().cpu().numpy(), g["dA"]), lo),
        "dW_in": (rel_fro(L.dW_in.double().cpu().numpy(), g["dW_in"]), hi),
        "db_dt": (rel_fro(L.db_dt.double().cpu().numpy(), g["db_dt"]), hi),
    }
    # the three column blocks of dz separately (dt, B, C)
    N = inputs["N"]
    for nm, sl in (("dz_dt", slice(0, P)), ("dz_B", slice(P, P + N)), ("dz_C", slice(P + N, P + 2 * N))):
        errs[nm] = (rel_fro(L.dz.double().cpu().numpy()[..., sl], g["dz"][..., sl]), hi)
    print(f"selective parity B={inputs['B']} T={inputs['T']} P={P} N={N} window={Tbar} bf16={bf16}: "
          + " ".join(f"{k}={v:.2e}" for k, (v, _) in errs.items()))
    bad = {k: v for k, (v, tol) in errs.items() if not v <= tol}
    assert not bad, (Tbar, bf16, {k: f"{v:.3e}" for k, (v, _) in errs.items()})
    return errs


@pytest.mark.parametrize("Tbar", [None, 64])
def test_tiny_workload(Tbar):
    compare(synth.make_sel_inputs("sel1_p16"), Tbar, False)


@pytest.mark.parametrize("Tbar", [None, 256])
def test_mid_workload(Tbar):
    """P = 64, N = 16, T = 2048, B = 2: several chunks of 256 tokens, two sequences."""
    compare(synth.make_sel_inputs("sel1_p64"), Tbar, False)


@pytest.mark.parametrize("T,B,P,N,Tbar", [
    (300, 2, 200, 16, None),    # ragged last chunk, a partial channel slice
    (300, 2, 200, 16, 48),      # 16-token chunks, window ends past the sequence end
    (700, 1, 64, 16, 96),       # 32-token chunks
    (1000, 1, 40, 8, 256),      # N = 8 (one thread a channel), 4 blocks
    (100, 3, 16, 8, None),      # shorter than one chunk
    (1, 1, 24, 16, None),       # one token
    (520, 1, 32, 16, 512),      # window one block short of T
    (512, 1, 32, 16, 512),      # window = T (the full adjoint)
])
def test_small_and_ragged(T, B, P, N, Tbar):
    compare(synth.make_sel_inputs("sel1_p64", T=T, B=B, P=P, N=N), Tbar, False)


@pytest.mark.parametrize("Tbar", [None, 256])
def test_bf16_operands(Tbar):
    inputs = synth.make_sel_inputs("sel1_p1024", T=1024, P=128)
    compare(inputs, Tbar, True)


def test_window_must_be_whole_small_chunks():
    from adjoint_gradients_long_gb300 import lib
    d = lib.dims(1, 1000, 32, 16)
    assert lib.workspace_bytes(d, lib.OP_SEL_BWD, 100) == 0      # not a multiple of 16
    assert lib.workspace_bytes(d, lib.OP_SEL_BWD, 96) > 0


def test_empty_batch_is_a_noop():
    """B = 0: the calls launch nothing but zero the outputs that are sums over tokens.  The
    token arrays are empty, so a stand-in buffer (never read or written) takes their place."""
    from adjoint_gradients_long_gb300 import lib
    P, N = 32, 16
    d = lib.dims(0, 64, P, N)
    dev = "cuda"
    stand_in = torch.zeros(64, device=dev)
    ws_bytes = max(lib.workspace_bytes(d, op) for op in (lib.OP_SEL_FWD, lib.OP_SEL_BWD, lib.OP_SEL_PARAM,
                                                          lib.OP_LOSS))
    ws = torch.zeros(ws_bytes // 4 + 64, dtype=torch.int32, device=dev)
    W_in, b_dt, A = torch.zeros(P, P + 2 * N, device=dev), torch.zeros(P, device=dev), torch.zeros(P, N, device=dev)
    w = lib.sel_weights(W_in, b_dt, A)
    dA, dW, db = torch.full((P, N), 7.0, device=dev), torch.full((P, P + 2 * N), 7.0, device=dev), \
        torch.full((P,), 7.0, device=dev)
    loss = torch.full((1,), 7.0, dtype=torch.float64, device=dev)
    s = stand_in
    lib.sel_fwd(d, w, s, s, s, s, ws, ws_bytes)
    lib.loss_mse(d, s, s, s, loss, ws, ws_bytes)
    lib.sel_bwd(d, w, s, s, s, s, None, s, dA, ws, ws_bytes)
    lib.sel_param_grad(d, s, s, dW, db, 0, ws, ws_bytes)
    torch.cuda.synchronize()
    assert float(dA.abs().max()) == 0.0 and float(dW.abs().max()) == 0.0 and float(db.abs().max()) == 0.0
    assert float(loss.item()) == 0.0
    assert float(stand_in.abs().max()) == 0.0


def test_graph_replay_matches_eager():
    from adjoint_gradients_long_gb300.sel_layer import SelLayer
    inputs = synth.make_sel_inputs("sel1_p64", T=1024, B=1)
    L = SelLayer(1, 1024, 64, 16, Tbar=256)
    L.load(inputs)
    L.step(256)
    torch.cuda.synchronize()
    eager = {k: getattr(L, k).clone() for k in ("dW_in", "db_dt", "dA")}
    g = L.capture(256)
    g.replay()
    torch.cuda.synchronize()
    for k, v in eager.items():
        assert torch.equal(getattr(L, k), v), k


def _full_samples(T, Tbar):
    w = Tbar if Tbar is not None else 8192
    out = []
    for i in (0, 5, w - 1, w, T // 2 + 77, T - w - 1, T - 1):
        if 0 <= i < T and i not in out:
            out.append(i)
    return out


@pytest.mark.parametrize("Tbar", [8192, None])
def test_full_size(Tbar):
    """The benchmark's selective workload (P = 1024, N = 16, T = 65536, bf16 operands) in its
    own launch configuration.  The oracle cannot sum every pair at this size, so:
      * sampled tokens: dz at sampled rows by the oracle's sampled-row evaluation (the
        window sums and VJPs of those tokens exactly, the forward recurrence run over every
        token before them);
      * properties at any size: dW_in = xhat^T dz and db_dt = sum_t dz[:, :P] in fp64 from
        the device's own operands (dz as the GEMM reads it), L = 1/2 ||y - target||^2 from
        the device's y."""
    from adjoint_gradients_long_gb300.sel_layer import SelLayer
    w = synth.SEL_WORKLOADS["sel1_p1024"]
    inputs = synth.make_sel_inputs(w)
    B, T, P, N = w.B, w.T, w.P, w.N
    L = SelLayer(B, T, P, N, x_bf16=True, Tbar=Tbar)
    L.load(inputs)
    L.step(Tbar)
    torch.cuda.synchronize()
    assert L.status() == 0
    Wd = {k: np.asarray(inputs[k], np.float64) for k in ("W_in", "b_dt", "A")}
    rows = [(0, i) for i in _full_samples(T, Tbar)]
    ref = sel.dz_rows(Wd, inputs["xhat"], inputs["target"], rows, Tbar)
    dz = L.dz.float().cpu().numpy().reshape(B * T, P + 2 * N)
    errs = {}
    for s, (b, i) in enumerate(rows):
        errs[f"dz[{i}]"] = rel_fro(dz[b * T + i], ref[s])
    x = L.x.float().cpu().numpy().reshape(B * T, P).astype(np.float64)
    errs["dW_in=x^T dz"] = rel_fro(L.dW_in.double().cpu().numpy(), x.T @ dz.astype(np.float64))
    errs["db_dt=sum dz"] = rel_fro(L.db_dt.double().cpu().numpy(), dz[:, :P].astype(np.float64).sum(axis=0))
    y = L.y.double().cpu().numpy()
    lref = 0.5 * float(np.sum((y - inputs["target"]) ** 2))
    errs["loss"] = abs(float(L.loss.item()) - lref) / lref
    print(f"selective full size window={Tbar}: " + " ".join(f"{k}={v:.2e}" for k, v in errs.items()))
    assert all(v <= 2e-2 for k, v in errs.items() if k.startswith("dz")), errs
    assert errs["dW_in=x^T dz"] <= 1e-4 and errs["db_dt=sum dz"] <= 1e-4 and errs["loss"] <= 1e-5, errs
