"""Full-length parity on every workload except the tiny one, in the benchmark's launch
configuration (the same library calls on buffers of the full size).

The oracle cannot sum all the VJP pairs of 131072 to 1048576 tokens in test time, so
each layer k is checked two ways:
  * sampled tokens: the oracle evaluates layer k on a slice of tokens around each
    sampled token i, fed the device's own layer input (xhat^k and the residual y^{k-1})
    and the device's cotangent gy^k on that slice.  Everything a layer computes at token
    i is then exact except for what crosses the slice ends: the state entering the slice
    (its effect on h_i is prod_{j=s0..i} a_j h_{s0-1}) and, with the full window, the
    adjoint entering from past the slice end (prod_{j=i+1..s1} a_j mu_{s1}).  The test
    computes both bounds from the actual gate values and requires them negligible before
    comparing h_i, mu_i (= D_u), D_a, D_c and E at token i.  With a window the slice
    reaches i + Tbar, so the window lies wholly inside it;
  * properties that hold at any size: dW_in = xhat^T [D_a|D_u|D_c], db_a = sum_t D_a,
    dW_o = E^T gy and L = 1/2 ||y - target||^2, recomputed in fp64 from the device's own
    operands as the GEMMs read them (gy rounded to bf16 in bf16 workloads), which checks
    the full-size reductions.
Tolerances: 1e-4 (fp32 workloads), 2e-2 (bf16 GEMM operands and seeds).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from adjoint_gradients_long_gb300 import synth  # noqa: E402
from conftest import rel_fro  # noqa: E402

pytestmark = pytest.mark.gpu
W_BACK = 4096      # tokens of the slice before the sampled token


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adjoint_gradients_long_gb300 import build
    build.build()


def _samples(T, B, Tbar):
    """Sampled (b, token) pairs: both ends, block edges of the window, and interior tokens."""
    w = Tbar if Tbar is not None else 4096
    cand = [(0, 0), (0, 5), (B - 1, T - 1), (B - 1, min(T - 1, w)), (0, min(T - 1, w - 1)), (B - 1, T // 2 + 77)]
    if B > 1:
        cand.append((1, min(T - 1, 4097)))
    out = []
    for b, i in cand:
        if (b, i) not in out:
            out.append((b, i))
    return out


_CACHE = {}


def _inputs(key):
    """Full-size inputs of a workload, kept for the next test of the same workload."""
    if key not in _CACHE:
        _CACHE.clear()
        _CACHE[key] = synth.make_inputs(key)
    return _CACHE[key]


def run_full(key, Tbar, samples_per_layer=None):
    from adjoint_gradients_long_gb300.stack import AdjStack
    w = synth.workload(key)
    bf16 = w.x_dtype == "bf16"
    tol = 2e-2 if bf16 else 1e-4
    inp = _inputs(key)
    B, T, P, N, K = w.B, w.T, w.P, w.N, w.K
    st = AdjStack(B, T, P, N, K, x_bf16=bf16, d_bf16=bf16, Tbar=Tbar)
    st.load(inp)
    cap = {}

    def grab(k, s):
        cap[k] = dict(D=[t.clone() for t in s.D], gy=s.gy[(s.K - 1 - k) % 2].clone())

    st.forward()
    st.loss_grad()
    st.backward(Tbar, on_layer=grab)
    torch.cuda.synchronize()
    assert st.status() == 0

    r = st.y[-1].double() - st.target.double()
    assert abs(st.loss.item() - 0.5 * float((r * r).sum())) <= 1e-6 * abs(st.loss.item())
    del r
    samples = _samples(T, B, Tbar)
    if samples_per_layer:
        samples = samples[:samples_per_layer]
    target = inp["target"]
    for k in range(K):
        Da, Du, Dc, E = cap[k]["D"]
        gy = cap[k]["gy"]
        # ---- the full-size reductions, fp64 on the device's own operands
        x = st.x[k].double().reshape(B * T, P)
        D = torch.cat([d.double().reshape(B * T, N) for d in (Da, Du, Dc)], dim=1)
        assert rel_fro(st.dW_in[k].cpu().numpy(), (x.T @ D).cpu().numpy()) <= 1e-4, k
        assert rel_fro(st.db_a[k].cpu().numpy(), D[:, :N].sum(0).cpu().numpy()) <= 1e-4, k
        del x, D
        # the GEMM's operands as it reads them: bf16 workloads round gy to bf16
        Ed = E.double().reshape(B * T, N)
        gop = (gy.to(torch.bfloat16) if bf16 else gy).double().reshape(B * T, P)
        assert rel_fro(st.dW_o[k].cpu().numpy(), (Ed.T @ gop).cpu().numpy()) <= 1e-4, k
        del Ed, gop
        # ---- sampled tokens against the oracle on a slice, from the device's layer input
        Wl = {nm: np.asarray(v, np.float64) for nm, v in inp["layers"][k].items()}
        for b, i in samples:
            s0 = max(0, i - W_BACK)
            s1 = min(T, i + (Tbar if Tbar is not None else 4096))
            xs = st.x[k][b:b + 1, s0:s1].double().cpu().numpy()
            xr = None if k == 0 else st.y[k - 1][b:b + 1, s0:s1].double().cpu().numpy()
            sto = oracle.layer_forward(Wl, xs, xr)
            gys = gy[b:b + 1, s0:s1].double().cpu().numpy()
            mu = oracle.layer_grad(Wl, sto, gys, Tbar)["mu"][0]
            a_s = sto["a"][0]
            j = i - s0
            # what crosses the slice ends, from the actual gates
            cut_fwd = 0.0
            if s0 > 0:
                h_in = st.h[k][b, s0 - 1].double().cpu().numpy()
                cut_fwd = float(np.max(np.prod(a_s[:j + 1], axis=0) * np.abs(h_in)))
            cut_bwd = 0.0
            if Tbar is None and s1 < T:
                mu_in = Du[b, s1].double().cpu().numpy()
                a_next = st.a[k][b, s1].double().cpu().numpy()
                cut_bwd = float(np.max(np.prod(a_s[j + 1:], axis=0) * a_next * np.abs(mu_in)))
            h_ref = sto["h"][0, j]
            assert cut_fwd <= 1e-7 * np.linalg.norm(h_ref) and cut_bwd <= 1e-7 * np.linalg.norm(mu[j]), \
                (k, b, i, cut_fwd, cut_bwd)
            dev = {nm: t[b, i].double().cpu().numpy() for nm, t in
                   (("h", st.h[k]), ("D_u", Du), ("D_a", Da), ("D_c", Dc), ("E", E))}
            g = gys[0, j] @ Wl["W_o"].T
            h_prev = sto["h"][0, j - 1] if j > 0 else np.zeros(N)
            ref = {"h": h_ref, "D_u": mu[j],
                   "D_a": mu[j] * h_prev * a_s[j] * (1.0 - a_s[j]),
                   "D_c": g * h_ref, "E": sto["c"][0, j] * h_ref}
            if s0 == 0 and j == 0:
                ref["D_a"] = np.zeros(N)
            for nm in ref:
                if np.linalg.norm(ref[nm]) > 0:
                    assert rel_fro(dev[nm], ref[nm]) <= tol, (key, Tbar, k, b, i, nm, rel_fro(dev[nm], ref[nm]))
                else:
                    assert np.linalg.norm(dev[nm]) == 0.0, (k, b, i, nm)
        if k == K - 1:
            # the top layer's cotangent is y^K - target
            yb = st.y[k][0, :64].double().cpu().numpy()
            assert rel_fro(gy[0, :64].double().cpu().numpy(), yb - target[0, :64]) <= 1e-6
        del cap[k]
    del st
    torch.cuda.empty_cache()


@pytest.mark.parametrize("Tbar", [None, 2048])
def test_ssm1_p128_full_size(Tbar):
    """P=128, N=256, T=16384, B=4, fp32 (the fp32 workload)."""
    run_full("ssm1_p128", Tbar)


@pytest.mark.parametrize("Tbar", [4096, None])
def test_ssm1_1m_full_length(Tbar):
    """One layer, P=256, N=256, T=2^20 tokens, bf16 GEMM operands, b_a=4: both windows."""
    run_full("ssm1_1m", Tbar)


def test_ssm8_p512_full_length():
    """K=8 residual layers, P=512, N=256, T=65536, bf16 GEMM operands, window 4096."""
    run_full("ssm8_p512", 4096, samples_per_layer=3)


def test_ssm4_p2048_full_length():
    """K=4 residual layers, P=2048, N=256, T=131072, bf16 GEMM operands, window 8192."""
    run_full("ssm4_p2048", 8192, samples_per_layer=3)
