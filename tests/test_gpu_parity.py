"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on the
same seeded inputs.  Tolerances (relative Frobenius error per tensor) are the ones
fixed for this path: 1e-4 where every operand is fp32, 2e-2 where the GEMM
operands (xhat, W, D, E) are bf16.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from adjoint_gradients_long_gb300 import synth  # noqa: E402
from conftest import rel_fro  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = {False: 1e-4, True: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adjoint_gradients_long_gb300 import build
    build.build()


def _layers64(inputs):
    return [{k: np.asarray(v, np.float64) for k, v in W.items()} for W in inputs["layers"]]


def run_gpu(inputs, Tbar, bf16):
    from adjoint_gradients_long_gb300.stack import AdjStack
    B, T, P, N, K = (inputs[k] for k in ("B", "T", "P", "N", "K"))
    st = AdjStack(B, T, P, N, K, x_bf16=bf16, d_bf16=bf16, Tbar=Tbar)
    st.load(inputs)
    seeds = {}

    def grab(k, s):
        seeds[k] = [t.float().cpu().numpy() for t in s.D] + [s.gy[(s.K - 1 - k) % 2].cpu().numpy()]

    st.forward()
    st.loss_grad()
    st.backward(Tbar, on_layer=grab)
    torch.cuda.synchronize()
    assert st.status() == 0
    return st, seeds


def compare(inputs, Tbar, bf16, check_states=True):
    tol = TOL[bf16]
    st, seeds = run_gpu(inputs, Tbar, bf16)
    ref = oracle.stack_grad(_layers64(inputs), inputs["xhat"], inputs["target"], Tbar)
    errs = {}
    errs["loss"] = abs(float(st.loss.item()) - ref["loss"]) / abs(ref["loss"])
    for k in range(inputs["K"]):
        g = st.grads_numpy(k)
        r = ref["grads"][k]
        for nm in ("W_a", "W_B", "W_c", "b_a", "W_o"):
            errs[f"d{nm}[{k}]"] = rel_fro(g[nm], r["d" + nm])
        errs[f"mu[{k}]"] = rel_fro(seeds[k][1], r["mu"])
        errs[f"gy[{k}]"] = rel_fro(seeds[k][4], ref["gy"][k])
        if check_states:
            so = ref["states"][k]
            for nm in ("a", "c", "h"):
                errs[f"{nm}[{k}]"] = rel_fro(getattr(st, nm)[k].cpu().numpy(), so[nm])
            errs[f"y[{k}]"] = rel_fro(st.y[k].cpu().numpy(), so["y"])
    errs["gx"] = None
    bad = {k: v for k, v in errs.items() if v is not None and not v <= tol}
    assert not bad, (bad, tol)
    return errs


# --------------------------------------------------------------- the five workloads, resized

@pytest.mark.parametrize("Tbar", [None, 1, 5, 37, 256, 1000])
def test_ssm1_p16_full_size(Tbar):
    """P=16, N=8, T=256, B=1 at its full size (fp32); windows incl. the degenerate ones."""
    compare(synth.make_inputs("ssm1_p16"), Tbar, False)


@pytest.mark.parametrize("Tbar", [None, 128, 100])
def test_ssm1_p128_shape(Tbar):
    """P=128, N=256, B=2, T=1000 (ragged against every chunk size), fp32."""
    compare(synth.make_inputs("ssm1_p128", T=1000, B=2), Tbar, False)


def test_ssm8_p512_shape():
    """K=8 residual layers, P=512, N=256, T=300, bf16 GEMM operands, window 64."""
    compare(synth.make_inputs("ssm8_p512", T=300), 64, True)


@pytest.mark.parametrize("Tbar", [256, None])
def test_ssm1_1m_shape(Tbar):
    """P=256, N=256, b_a=4, T=2000, bf16 GEMM operands, window 256 and full."""
    compare(synth.make_inputs("ssm1_1m", T=2000), Tbar, True)


def test_ssm4_p2048_shape():
    """K=4 residual layers, P=2048, N=256, T=200, bf16 GEMM operands, window 48."""
    compare(synth.make_inputs("ssm4_p2048", T=200), 48, True)


def test_bf16_stack_with_ragged_channels():
    """bf16 layers with P = 200 (not a multiple of the 32-column epilogue chunk): the input
    gradient's bf16 output copy and x-hat chunks move by TMA with boxes that cross the last
    column (clipped stores, zero-filled loads); three layers, window 64."""
    compare(synth.make_inputs("ssm8_p512", T=300, P=200, N=64, K=3), 64, True)


def test_four_cta_clusters_with_a_partial_last_cluster():
    """P=2048 (K = 2048 > 1024 in the input projection: four-CTA clusters sharing B), T=700:
    three 256-row pair tiles, so the second cluster's second pair lies wholly past the last
    token and its first pair partly; two layers, full window."""
    compare(synth.make_inputs("ssm4_p2048", T=700, K=2), None, True)


def test_streamed_output_projection_elementwise():
    """The output projection over an output far larger than L2 (34000 x 2048 fp32, 278 MB)
    keeps its B half resident and gives each epilogue warp separate residual and output
    buffers; 34000 tokens leave the last 256-row pair tile partly filled.  Each layer's output
    y^k is checked element by element against y^{k-1} (xhat for the first layer) + bf16(c h) W_o
    recomputed in fp64 from the same run's c, h and W_o ([AS] What carries the argument: the
    residual stack), so a chunk written from the wrong buffer or rows cannot hide in a norm.
    The bound is the fp32 accumulation of 256 products: 1e-4 of sum |a w| (about 2^-13)."""
    from adjoint_gradients_long_gb300.stack import AdjStack
    T, P, N, K = 34000, 2048, 256, 2
    st = AdjStack(1, T, P, N, K, x_bf16=True, d_bf16=True)
    st.load(synth.make_inputs("ssm4_p2048", T=T, K=K))
    st.forward()
    torch.cuda.synchronize()
    assert st.status() == 0
    for k in range(K):
        ch = synth.round_bf16(st.c[k][0].cpu().numpy() * st.h[k][0].cpu().numpy()).astype(np.float64)
        W = st.W_o[k].float().cpu().numpy().astype(np.float64)
        res = (st.x[0][0].float() if k == 0 else st.y[k - 1][0]).cpu().numpy()
        y = st.y[k][0].cpu().numpy()
        for r0 in range(0, T, 4096):
            sl = slice(r0, r0 + 4096)
            ref = res[sl].astype(np.float64) + ch[sl] @ W
            bound = 1e-4 * (np.abs(ch[sl]) @ np.abs(W)) + 1e-6 * np.abs(ref) + 1e-30
            err = np.abs(y[sl].astype(np.float64) - ref)
            bad = err > bound
            assert not bad.any(), (k, r0, int(bad.sum()), np.argwhere(bad)[:4].tolist(), float((err / bound).max()))


# --------------------------------------------------------------- the bf16 workloads at their own windows

PREFIX = 16384


@pytest.mark.parametrize("key,Tbar", [("ssm1_1m", 4096), ("ssm1_1m", None), ("ssm8_p512", 4096),
                                      ("ssm4_p2048", 8192)])
def test_prefix_at_stated_window(key, Tbar):
    """Each bf16 workload on its first 16384 tokens, at the window it is stated with (full
    width, full depth): windows of 64-128 scan chunks, whose look-back runs several rounds
    before it meets a closed composite, and the bf16 split-K parameter reductions over 16K
    tokens.  Every tensor of every layer is compared with the oracle."""
    compare(synth.make_inputs(key, T=PREFIX), Tbar, True)


# --------------------------------------------------------------- edge cases

@pytest.mark.parametrize("T,B,Tbar", [(1, 1, None), (1, 2, 1), (33, 3, None), (33, 3, 32), (64, 1, 64), (65, 2, 2),
                                      (129, 1, 64), (300, 3, 64), (300, 2, 128), (640, 1, 64), (700, 2, 192)])
def test_small_and_ragged(T, B, Tbar):
    """Degenerate and ragged sizes; windows of whole 64-token chunks take the one-launch
    truncated adjoint (one-chunk blocks, a ragged last block, several blocks)."""
    compare(synth.make_inputs("ssm1_p16", T=T, B=B), Tbar, False)


def test_two_layer_fp32_stack():
    compare(synth.make_inputs("ssm8_p512", T=150, B=2, P=32, N=16, K=2), 40, False)


def test_repeat_calls_agree_to_rounding():
    """The look-back scans combine chunk carries along whichever chain is ready first, so
    repeated calls agree to fp32 rounding, not bit for bit."""
    inputs = synth.make_inputs("ssm1_p128", T=777, B=1)
    st1, _ = run_gpu(inputs, 128, False)
    st2, _ = run_gpu(inputs, 128, False)
    for k in range(1):
        a, b = st1.grads_numpy(k), st2.grads_numpy(k)
        for nm in a:
            assert rel_fro(a[nm], b[nm]) <= 1e-6, nm


def test_graph_replay_matches_eager_and_oracle():
    """A captured step (a CUDA graph of the library calls, as the bench times it) replays the
    same computation: its gradients match the eager step's to fp32 rounding and the oracle's
    within the fp32 tolerance."""
    from adjoint_gradients_long_gb300.stack import AdjStack
    inputs = synth.make_inputs("ssm1_p128", T=512, B=2)
    B, T, P, N, K = (inputs[k] for k in ("B", "T", "P", "N", "K"))
    st = AdjStack(B, T, P, N, K, Tbar=128)
    st.load(inputs)
    st.step(None)
    torch.cuda.synchronize()
    eager = st.grads_numpy(0)
    g = st.capture(None)
    for t in (st.dW_in[0], st.db_a[0], st.dW_o[0]):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert st.status() == 0
    rep = st.grads_numpy(0)
    ref = oracle.stack_grad(_layers64(inputs), inputs["xhat"], inputs["target"], None)["grads"][0]
    for nm in eager:
        assert rel_fro(rep[nm], eager[nm]) <= 1e-6, nm
        assert rel_fro(rep[nm], ref["d" + nm]) <= TOL[False], nm


@pytest.mark.parametrize("bf16", [False, True])
def test_param_grad_accumulate_adds(bf16):
    """accumulate = 1 adds a call's parameter gradients to the arrays: a second backward
    pass over the same step doubles dW_in, db_a and dW_o (fp32 seeds: db_a comes from the
    dW_in GEMM's producers; bf16 seeds: from the column-sum kernel)."""
    from adjoint_gradients_long_gb300.stack import AdjStack
    if bf16:
        inputs = synth.make_inputs("ssm8_p512", T=200, B=1, P=64, N=32, K=1)
    else:
        inputs = synth.make_inputs("ssm1_p128", T=300, B=2)
    B, T, P, N, K = (inputs[k] for k in ("B", "T", "P", "N", "K"))
    st = AdjStack(B, T, P, N, K, x_bf16=bf16, d_bf16=bf16)
    st.load(inputs)
    st.forward()
    st.loss_grad()
    st.backward(None)
    torch.cuda.synchronize()
    once = st.grads_numpy(0)
    st.backward(None, accumulate=True)
    torch.cuda.synchronize()
    assert st.status() == 0
    twice = st.grads_numpy(0)
    for nm in once:
        assert rel_fro(twice[nm], 2.0 * once[nm]) <= 1e-5, nm
