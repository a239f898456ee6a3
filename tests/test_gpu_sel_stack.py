"""GPU parity of residual stacks of general selective layers: the CUDA path (through the
C ABI: adj_rms_norm, adj_sel_fwd with the residual input, adj_sel_bwd and
adj_sel_param_grad with the input path) against the fp64 oracle's stack
(oracle/selective.py stack_grad) on the same seeded inputs.

Tolerances, relative Frobenius error per tensor: 1e-4 where every stored operand is fp32.
With bf16 storage the layer inputs xhat^k (k >= 2) are the normalised residual stream
rounded to bf16 (relative error up to 2^-8 a value, the bf16 unit roundoff) while the
oracle keeps them exact; everything downstream of a bf16 operand is held to 3e-2, and
the residual stream y and the loss, which stay fp32 but take each layer's output from a
rounded input, to 4e-3 (about 2^-8).

Source: the review page "Adjoint sharding for very long context training of state space
models" ([AS]): the residual stack y^K = y^0 + sum_k ytilde^k (What carries the argument),
normalised layer inputs (Load-bearing premise), and each layer's gradient from its total
cotangent, full or truncated (Core claim, Proposition 3).
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
    from adjoint_gradients_long_gb300.sel_layer import SelStack
    B, T, P, N, K = (inputs[k] for k in ("B", "T", "P", "N", "K"))
    S = SelStack(B, T, P, N, K, x_bf16=bf16, Tbar=Tbar)
    S.load(inputs)
    S.step(Tbar)
    torch.cuda.synchronize()
    assert S.status() == 0
    return S


def reference(inputs, Tbar):
    layers = [{k: np.asarray(W[k], np.float64) for k in ("W_in", "b_dt", "A")} for W in inputs["layers"]]
    return sel.stack_grad(layers, inputs["xhat"], inputs["target"], Tbar)


def compare(inputs, Tbar, bf16):
    S = run(inputs, Tbar, bf16)
    ref = reference(inputs, Tbar)
    lo, hi, res = 1e-4, (3e-2 if bf16 else 1e-4), (4e-3 if bf16 else 1e-4)
    errs = {"loss": (abs(float(S.loss.item()) - ref["loss"]) / abs(ref["loss"]), res)}
    for k in range(S.K):
        errs[f"y{k}"] = (rel_fro(S.y[k].double().cpu().numpy(), ref["states"][k]["y"]), res)
        g = S.grads_numpy(k)
        for nm in ("W_in", "b_dt", "A"):
            errs[f"d{nm}{k}"] = (rel_fro(g[nm], ref["grads"][k]["d" + nm]), hi if (bf16 or nm != "A") else lo)
    # layer 1's total cotangent: every layer's input path above it
    errs["seed0"] = (rel_fro(S.seed0().double().cpu().numpy(), ref["gy"][0]), hi)
    print(f"selective stack parity K={S.K} B={S.B} T={S.T} P={S.P} N={S.N} window={Tbar} bf16={bf16}: "
          + " ".join(f"{k}={v:.2e}" for k, (v, _) in errs.items()))
    bad = {k: v for k, (v, tol) in errs.items() if not v <= tol}
    assert not bad, (Tbar, bf16, {k: f"{v:.3e}" for k, (v, _) in errs.items()})
    return errs


@pytest.mark.parametrize("Tbar", [None, 64])
def test_tiny_stack(Tbar):
    compare(synth.make_sel_stack_inputs("sel1_p16", 3, T=256, B=2), Tbar, False)


@pytest.mark.parametrize("Tbar", [None, 256])
def test_mid_stack(Tbar):
    """P = 64, N = 16, T = 2048, B = 2, K = 2: several chunks, two sequences."""
    compare(synth.make_sel_stack_inputs("sel1_p64", 2), Tbar, False)


@pytest.mark.parametrize("K,T,B,P,N,Tbar", [
    (2, 300, 2, 200, 16, 48),    # ragged last chunk, a partial channel slice
    (3, 1000, 1, 40, 8, None),   # N = 8 (one thread a channel)
    (2, 100, 3, 16, 8, 32),      # shorter than one chunk of the full adjoint
    (4, 1, 1, 24, 16, None),     # one token
])
def test_small_and_ragged_stacks(K, T, B, P, N, Tbar):
    compare(synth.make_sel_stack_inputs("sel1_p64", K, T=T, B=B, P=P, N=N), Tbar, False)


@pytest.mark.parametrize("Tbar", [None, 256])
def test_bf16_stack(Tbar):
    compare(synth.make_sel_stack_inputs("sel1_p1024", 3, T=1024, P=128), Tbar, True)


def test_bf16_stack_four_cta_clusters():
    """P=1024: the input GEMM (K = P + 2N = 1056) and dW_in run as four-CTA clusters; T=600
    gives three 256-row pair tiles, the last cluster half past the last token."""
    compare(synth.make_sel_stack_inputs("sel1_p1024", 2, T=600), None, True)


def test_stack_of_one_is_the_layer():
    """K = 1 makes no normalisation and no input-path call: the lone layer's results."""
    from adjoint_gradients_long_gb300.sel_layer import SelLayer
    inputs = synth.make_sel_stack_inputs("sel1_p64", 1, T=512, B=1)
    S = run(inputs, 128, False)
    L = SelLayer(1, 512, 64, 16, Tbar=128)
    L.load(inputs)
    L.step(128)
    torch.cuda.synchronize()
    for nm in ("dW_in", "db_dt", "dA"):
        assert torch.equal(getattr(S, nm)[0], getattr(L, nm)), nm


def test_input_path_leaves_the_parameter_gradients_alone():
    """The input-path outputs are extra: a stacked layer's dz and dA are bitwise those of
    the same call without them (gy[0] still holds layer 2's seed after the step)."""
    from adjoint_gradients_long_gb300 import lib
    inputs = synth.make_sel_stack_inputs("sel1_p64", 2, T=512, B=1)
    S = run(inputs, None, False)
    args = (S.dims, S.w[1], S.x[1], S.z[1], S.h[1], S.gy[0], None, S.dz, S.dA[1], S.ws, S.ws_bytes)
    lib.sel_bwd(*args, r=S.r[0], gadd=S.gadd, rowdot=S.rowdot)
    torch.cuda.synchronize()
    dz_inp, dA_inp = S.dz.clone(), S.dA[1].clone()
    lib.sel_bwd(*args)
    torch.cuda.synchronize()
    assert torch.equal(S.dz, dz_inp) and torch.equal(S.dA[1], dA_inp)


def test_stack_graph_replay_matches_eager():
    from adjoint_gradients_long_gb300.sel_layer import SelStack
    inputs = synth.make_sel_stack_inputs("sel1_p64", 3, T=1024, B=1)
    S = SelStack(1, 1024, 64, 16, 3, Tbar=256)
    S.load(inputs)
    S.step(256)
    torch.cuda.synchronize()
    eager = {(nm, k): getattr(S, nm)[k].clone() for nm in ("dW_in", "db_dt", "dA") for k in range(3)}
    g = S.capture(256)
    g.replay()
    torch.cuda.synchronize()
    for (nm, k), v in eager.items():
        assert torch.equal(getattr(S, nm)[k], v), (nm, k)
