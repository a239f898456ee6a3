"""Full-size parity on the workload the benchmark times (P=128, N=256, T=16384, B=4,
fp32; full adjoint and window 2048), in the benchmark's launch configuration.

The oracle cannot sum all 4 * 16384^2 / 2 VJP pairs in test time, so:
  * sampled tokens: the oracle evaluates the layer on a slice of 2W tokens around
    each sampled token (state h = 0 at the slice start, sums cut at the slice end).
    The error of the cut is bounded by max(a)^W times the state / adjoint size and
    the test asserts that bound is negligible before comparing h_t and mu_t;
  * properties that hold at any size: dW_in = xhat^T [D_a|D_u|D_c], db_a = sum_t D_a,
    dW_o = E^T gy and L = 1/2 ||y - target||^2, recomputed in fp64 from the device's
    own operands (checks the full-size reductions).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from adjoint_gradients_long_gb300 import synth  # noqa: E402
from conftest import rel_fro  # noqa: E402

pytestmark = pytest.mark.gpu
W = 1024
SAMPLES = [(0, 0), (0, 5), (1, 4097), (2, 9000), (3, 16383), (3, 12345)]


@pytest.fixture(scope="module")
def full_inputs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adjoint_gradients_long_gb300 import build
    build.build()
    return synth.make_inputs("ssm1_p128")


@pytest.mark.parametrize("Tbar", [None, 2048])
def test_full_size_sampled_and_properties(full_inputs, Tbar):
    from adjoint_gradients_long_gb300.stack import AdjStack
    inp = full_inputs
    B, T, P, N = inp["B"], inp["T"], inp["P"], inp["N"]
    st = AdjStack(B, T, P, N, 1, Tbar=Tbar)
    st.load(inp)
    cap = {}

    def grab(k, s):
        cap["D"] = [t.double() for t in s.D]

    st.forward()
    st.loss_grad()
    st.backward(Tbar, on_layer=grab)
    torch.cuda.synchronize()
    assert st.status() == 0

    # ---- properties at full size, fp64 on the device's own operands
    x = st.x[0].double().reshape(B * T, P)
    Da, Du, Dc, E = (d.reshape(B * T, N) for d in cap["D"])
    gy = st.gy[0].double().reshape(B * T, P)
    dW_in = x.T @ torch.cat([Da, Du, Dc], dim=1)
    assert rel_fro(st.dW_in[0].cpu().numpy(), dW_in.cpu().numpy()) <= 1e-4
    assert rel_fro(st.db_a[0].cpu().numpy(), Da.sum(0).cpu().numpy()) <= 1e-4
    assert rel_fro(st.dW_o[0].cpu().numpy(), (E.T @ gy).cpu().numpy()) <= 1e-4
    r = st.y[0].double() - st.target.double()
    assert abs(st.loss.item() - 0.5 * float((r * r).sum())) <= 1e-6 * abs(st.loss.item())

    # ---- sampled tokens against the oracle on a 2W-token slice
    Wl = {k: np.asarray(v, np.float64) for k, v in inp["layers"][0].items()}
    h_dev = st.h[0].cpu().numpy()
    mu_dev = cap["D"][1].cpu().numpy().reshape(B, T, N)
    for b, i in SAMPLES:
        s0, s1 = max(0, i - W), min(T, i + W)
        xs = inp["xhat"][b:b + 1, s0:s1].astype(np.float64)
        ts = inp["target"][b:b + 1, s0:s1].astype(np.float64)
        stt = oracle.layer_forward(Wl, xs)
        gys = stt["y"] - ts
        mu = oracle.layer_grad(Wl, stt, gys, Tbar)["mu"]
        amax = float(stt["a"].max())
        cut_fwd = 0.0 if s0 == 0 else amax ** (i - s0) * float(np.abs(stt["h"]).max())
        reach = T if Tbar is None else min(T, i + Tbar)
        cut_bwd = 0.0 if s1 >= reach else amax ** (s1 - i) * float(np.abs(mu).max()) * 10.0
        assert cut_fwd <= 1e-9 and cut_bwd <= 1e-9, (cut_fwd, cut_bwd)
        j = i - s0
        assert rel_fro(h_dev[b, i], stt["h"][0, j]) <= 1e-4, (b, i)
        assert rel_fro(mu_dev[b, i], mu[0, j]) <= 1e-4, (b, i)
