"""Failure detection without a GPU fault: the bounded device waits give up on objects
nobody releases, record ADJ_ETIMEOUT in the workspace status word, and the context
stays usable for the next call."""
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
    ws = torch.zeros(1024 // 4, dtype=torch.int32, device="cuda")
    assert lib.stream_status(ws) == 0
    lib.selftest_waits(ws, 1024, which)
    assert lib.STATUS[lib.stream_status(ws)] == "ADJ_ETIMEOUT"
    assert lib.stream_status(ws) == 0            # the status word is cleared by the read
    # the context still works: a real call afterwards succeeds
    from adjoint_gradients_long_gb300 import synth
    from adjoint_gradients_long_gb300.stack import AdjStack
    st = AdjStack(1, 64, 16, 8, 1)
    st.load(synth.make_inputs("ssm1_p16", T=64))
    st.step(None)
    torch.cuda.synchronize()
    assert st.status() == 0
