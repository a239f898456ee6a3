"""adj_fwd_scan_noalloc, the forward pass for callers that cannot allocate device
memory (for example code inside a host application that owns the whole device pool,
or a plugin that must not touch the process allocator).  Its scratch is a fixed
32 MiB array inside the library; it must give the same results as adj_fwd_scan with a
caller workspace, on two calls in a row, and reject problems too large for the array.

Collected last (file name) so that a run stopping at the first failure has run every
other test first.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from conftest import rel_fro  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adjoint_gradients_long_gb300 import build, lib
    build.build()
    L = lib.load()
    # dims, w, then xhat, xres, a, c, h, y, y_x, status, stream
    L.adj_fwd_scan_noalloc.argtypes = [ctypes.POINTER(lib.Dims), ctypes.POINTER(lib.Weights)] + [ctypes.c_void_p] * 9
    L.adj_fwd_scan_noalloc.restype = ctypes.c_int
    return L


def test_noalloc_matches_workspace_path(L):
    from adjoint_gradients_long_gb300 import lib, synth
    from adjoint_gradients_long_gb300.stack import AdjStack
    B, T, P, N = 2, 2000, 128, 256
    inputs = synth.make_inputs("ssm1_p128", T=T, B=B)
    st = AdjStack(B, T, P, N, 1)
    st.load(inputs)
    st.forward()
    torch.cuda.synchronize()
    assert st.status() == 0
    ref = {k: getattr(st, k)[0].clone() for k in ("a", "c", "h", "y")}
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.ones(4, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = {k: torch.full_like(v, float("nan")) for k, v in ref.items()}
        s = L.adj_fwd_scan_noalloc(ctypes.byref(st.dims), ctypes.byref(st.w[0]), st.x[0].data_ptr(), None,
                                   out["a"].data_ptr(), out["c"].data_ptr(), out["h"].data_ptr(),
                                   out["y"].data_ptr(), None, status.data_ptr(), stream)
        assert s == 0, lib.STATUS.get(s, s)
        torch.cuda.synchronize()
        assert int(status[0].item()) == 0, call
        for k in ref:
            assert rel_fro(out[k].cpu().numpy(), ref[k].cpu().numpy()) <= 1e-4, (call, k)


@pytest.mark.parametrize("B,T", [(1024, 16384), (64, 16383)])   # fused and unfused forward
def test_noalloc_rejects_problems_beyond_its_scratch(L, B, T):
    from adjoint_gradients_long_gb300 import lib
    d = lib.dims(B, T, 128, 256)
    assert L.adj_workspace_bytes(ctypes.byref(d), lib.OP_FWD, 0) > (32 << 20)
    # Every array pointer is NULL: if the size check ever let this problem through,
    # adj_fwd_scan's own pointer checks would refuse it (ADJ_EINVAL) before any launch,
    # so nothing can run on memory that does not exist.
    w = lib.Weights(None, None, None)
    n0 = L.adj_launch_count()
    s = L.adj_fwd_scan_noalloc(ctypes.byref(d), ctypes.byref(w), None, None, None, None, None, None, None, None,
                               torch.cuda.current_stream().cuda_stream)
    assert lib.STATUS[s] == "ADJ_EWORKSPACE"
    assert L.adj_launch_count() == n0
