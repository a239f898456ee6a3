"""The C-ABI library builds, loads, exports every symbol include/adj.h declares, and
rejects bad arguments on the host before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

from adjoint_gradients_long_gb300 import build as adj_build, lib, synth, accounting

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    adj_build.build()
    return lib.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "adj.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(adj_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert set(lib.EXPORTS) <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for s in range(8):
        assert lib.status_str(s) != "unknown status"


FAKE = 1 << 40  # 16-byte aligned address never dereferenced by validation


def _w():
    return lib.Weights(FAKE, FAKE, FAKE)


def _call_fwd(d, w=None, xhat=FAKE, a=FAKE, ws=FAKE, ws_bytes=1 << 40, y=None, y_x=None, xres=None):
    w = w or _w()
    return lib.load().adj_fwd_scan(ctypes.byref(d), ctypes.byref(w), xhat, xres, a, FAKE, FAKE, y, y_x, ws,
                                   ws_bytes, None)


def test_rejects_bad_shapes(L):
    assert _call_fwd(lib.dims(1, 16, 12, 8)) == 2          # P not a multiple of 8
    assert _call_fwd(lib.dims(1, 16, 16, 6)) == 2          # N not a multiple of 8
    assert _call_fwd(lib.dims(-1, 16, 16, 8)) == 2
    assert _call_fwd(lib.dims(1, 16, 16, 8, 3, 0)) == 4    # bad dtype


def test_rejects_null_and_misaligned(L):
    d = lib.dims(1, 16, 16, 8)
    assert _call_fwd(d, xhat=None) == 1
    assert _call_fwd(d, a=FAKE + 4) == 3
    assert _call_fwd(d, ws=FAKE + 16) == 3                  # workspace must be 256-byte aligned
    assert _call_fwd(d, ws=None) == 1
    assert _call_fwd(d, y=FAKE, y_x=FAKE) == 1              # y_x needs bf16 operands


def test_rejects_small_workspace(L):
    d = lib.dims(2, 1000, 128, 256)
    need = lib.workspace_bytes(d, lib.OP_FWD)
    assert need > 0
    assert _call_fwd(d, ws_bytes=need - 1) == 5


def test_rejects_bad_window(L):
    d = lib.dims(1, 64, 16, 8)
    st = L.adj_bwd_trunc(ctypes.byref(d), ctypes.byref(_w()), *([FAKE] * 4), None, *([FAKE] * 4), None, 0, FAKE,
                         1 << 40, None)
    assert st == 1
    assert lib.workspace_bytes(d, lib.OP_BWD_TRUNC, 0) == 0


def test_rejects_misused_optional_outputs(L):
    """bf16 copies of the cotangent exist only for bf16 operands; the normalised-input
    cotangent needs both r and dz and an output; dz needs the gate bias.  Refused before
    anything launches (the pointers are never dereferenced)."""
    f32 = lib.dims(1, 64, 16, 8)
    bf = lib.dims(1, 64, 16, 8, lib.BF16, lib.BF16)
    w = _w()
    big = 1 << 40
    # adj_bwd_full with gy_x on fp32 operands
    assert L.adj_bwd_full(ctypes.byref(f32), ctypes.byref(w), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                          None, FAKE, big, None) == 1
    # dz without b_a
    wn = lib.Weights(FAKE, None, FAKE)
    assert L.adj_bwd_full(ctypes.byref(bf), ctypes.byref(wn), FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE,
                          FAKE, FAKE, big, None) == 1

    def pg(d, gy_x=None, gy_prev=None, gy_prev_x=None, dxhat=None, r=None, dz=None):
        return L.adj_param_grad(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, gy_x, FAKE, FAKE,
                                FAKE, gy_prev, gy_prev_x, dxhat, r, dz, 0, FAKE, big, None)
    assert pg(f32, gy_x=FAKE) == 1                         # bf16 copy with fp32 operands
    assert pg(bf, gy_prev_x=FAKE) == 1                     # a copy of an output not asked for
    assert pg(bf, gy_prev=FAKE, r=FAKE) == 1               # r without dz
    assert pg(bf, dxhat=FAKE, r=FAKE, dz=FAKE) == 1        # the normalised cotangent goes to gy_prev
    assert pg(bf, gy_prev=FAKE, dxhat=FAKE) == 1           # at most one input cotangent
    # adj_loss_mse: a bf16 copy needs gy
    assert L.adj_loss_mse(ctypes.byref(bf), FAKE, FAKE, None, FAKE, FAKE, FAKE, big, None) == 1


def test_workspace_sizes_grow_with_problem(L):
    small = lib.dims(1, 1024, 128, 256)
    big = lib.dims(4, 16384, 128, 256)
    for op in (lib.OP_FWD, lib.OP_BWD_FULL, lib.OP_PARAM, lib.OP_LOSS):
        assert 0 < lib.workspace_bytes(small, op) <= lib.workspace_bytes(big, op)
    assert lib.workspace_bytes(big, lib.OP_BWD_TRUNC, 2048) > lib.workspace_bytes(big, lib.OP_BWD_FULL)


def test_empty_problem_is_a_noop(L):
    d = lib.dims(0, 64, 16, 8)
    need = lib.workspace_bytes(d, lib.OP_FWD)
    assert _call_fwd(d, ws_bytes=need) == 0


def test_workload_table():
    w = synth.workload("ssm1_p128")
    assert (w.B, w.T, w.P, w.N, w.K) == (4, 16384, 128, 256, 1)
    assert synth.workload(5).P == 2048
    assert accounting.stored_bytes(4, 16384, 1, 256, 128, 4) == 4 * 16384 * (3 * 256 * 4 + 128 * 4)


def test_synth_prefix_is_a_slice():
    full = synth.make_inputs("ssm1_p16", T=5000)
    part = synth.make_inputs("ssm1_p16", T=1000, t0=4000)
    assert (full["xhat"][:, 4000:5000] == part["xhat"]).all()
    assert (full["target"][:, 4000:5000] == part["target"]).all()


def test_binding_arities_match_header(L):
    src = open(os.path.join(ROOT, "include", "adj.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    for name, params in re.findall(r"\b(adj_[a-z_]+)\s*\(([^)]*)\)\s*;", src):
        params = params.strip()
        n = 0 if params in ("", "void") else len(params.split(","))
        fn = getattr(L, name)
        if fn.argtypes is not None:
            assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)


def test_selective_layer_rejects_bad_arguments(L):
    """The general selective layer's calls: N must be 8 or 16, a truncation window a
    multiple of 16, every pointer present, the workspace large enough; refused before
    anything launches (the pointers are never dereferenced)."""
    big = 1 << 40
    w = lib.SelWeights(FAKE, FAKE, FAKE)

    def fwd(d, ws_bytes=big, h=FAKE):
        return L.adj_sel_fwd(ctypes.byref(d), ctypes.byref(w), FAKE, None, FAKE, h, FAKE, FAKE, ws_bytes, None)

    def bwd(d, Tbar=0, dz=FAKE, inp=(None, None, None)):
        return L.adj_sel_bwd(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE, FAKE, FAKE, Tbar, dz, FAKE, *inp, FAKE,
                             big, None)

    def param(d, dz=FAKE, wp=None, inp=(None, None, None, None), acc=0):
        return L.adj_sel_param_grad(ctypes.byref(d), wp, FAKE, dz, FAKE, FAKE, *inp, acc, FAKE, big, None)

    assert fwd(lib.dims(1, 64, 32, 24)) == 2                 # N = 24
    assert fwd(lib.dims(1, 64, 32, 32)) == 2                 # N = 32
    assert fwd(lib.dims(1, 64, 32, 16), h=None) == 1
    assert fwd(lib.dims(1, 64, 32, 16), h=FAKE + 4) == 3
    d = lib.dims(2, 1000, 64, 16)
    assert fwd(d, ws_bytes=lib.workspace_bytes(d, lib.OP_SEL_FWD) - 1) == 5
    assert L.adj_sel_fwd(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE + 4, FAKE, FAKE, FAKE, FAKE, big, None) == 3
    assert fwd(lib.dims(0, 64, 32, 16)) == 0                 # empty batch: nothing to do
    assert bwd(lib.dims(1, 1000, 32, 16), Tbar=100) == 1     # window not a multiple of 16
    assert bwd(lib.dims(1, 1000, 32, 16), dz=None) == 1
    assert param(lib.dims(1, 64, 32, 16), dz=None) == 1
    assert param(lib.dims(1, 64, 32, 16), acc=2) == 1
    # the input path of a stacked layer: all of its buffers or none, and W_in with it
    d1 = lib.dims(1, 64, 32, 16)
    assert bwd(d1, inp=(FAKE, FAKE, None)) == 1
    assert bwd(d1, inp=(None, FAKE, FAKE)) == 1
    assert bwd(d1, inp=(FAKE, FAKE, FAKE + 4)) == 3
    assert param(d1, inp=(FAKE, FAKE, FAKE, None)) == 1
    assert param(d1, inp=(FAKE, FAKE, FAKE, FAKE)) == 1                    # no weights
    assert param(d1, wp=ctypes.byref(lib.SelWeights(None, FAKE, FAKE)), inp=(FAKE,) * 4) == 1
    assert lib.sel_rowdot_cols(lib.dims(1, 64, 1024, 16)) == 1024 // 128 + 1
    assert lib.sel_rowdot_cols(lib.dims(1, 64, 1000, 8)) == 4 + 1
    assert lib.sel_rowdot_cols(lib.dims(1, 64, 32, 24)) == 0
    for op in (lib.OP_SEL_FWD, lib.OP_SEL_BWD, lib.OP_SEL_PARAM):
        assert lib.workspace_bytes(lib.dims(1, 64, 32, 24), op) == 0
    # the truncated window's scratch (aggregates and R) makes its workspace the larger
    assert lib.workspace_bytes(d, lib.OP_SEL_BWD, 256) > lib.workspace_bytes(d, lib.OP_SEL_BWD, 0)
