"""Failure detection without a GPU fault: the bounded device waits give up on objects
nobody releases, record ADJ_ETIMEOUT in the workspace status word, and the context
stays usable for the next call.

which = 1 runs the scans' decoupled look-back (the forward state scan kernel over a
problem whose first chunk is never launched: every other chunk waits for it until the
round limit, then finishes with a zero carry); which = 2 an mbarrier that is never
arrived on."""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adjoint_gradients_long_gb300 import build, lib as L
    build.build()
    return L


@pytest.mark.parametrize("which", [1, 2])
def test_bounded_wait_reports_timeout(lib, which):
    n = lib.selftest_ws_bytes()
    ws = torch.zeros((n + 255) // 4, dtype=torch.int32, device="cuda")
    assert lib.stream_status(ws) == 0
    t0 = time.time()
    lib.selftest_waits(ws, n, which)
    assert lib.STATUS[lib.stream_status(ws)] == "ADJ_ETIMEOUT"
    assert time.time() - t0 < 60.0                # the waits gave up on their own
    assert lib.stream_status(ws) == 0            # the status word is cleared by the read
    if which == 1:
        # the chunks that gave up finished with a zero carry: the state array (after the
        # 256-byte header and the a and u arrays of 768 x 128 fp32) is finite
        n_arr = 768 * 128
        h = ws[64 + 2 * n_arr:64 + 3 * n_arr].view(torch.float32)
        assert bool(torch.isfinite(h).all())
    # the context still works: a real call afterwards succeeds and matches the oracle
    import oracle
    from adjoint_gradients_long_gb300 import synth
    from adjoint_gradients_long_gb300.stack import AdjStack
    from conftest import rel_fro
    inputs = synth.make_inputs("ssm1_p16", T=300)
    st = AdjStack(1, 300, 16, 8, 1)
    st.load(inputs)
    st.step(None)
    torch.cuda.synchronize()
    assert st.status() == 0
    layers = [{k: np.asarray(v, np.float64) for k, v in W.items()} for W in inputs["layers"]]
    ref = oracle.stack_grad(layers, inputs["xhat"], inputs["target"], None)
    assert rel_fro(st.grads_numpy(0)["W_B"], ref["grads"][0]["dW_B"]) <= 1e-4
