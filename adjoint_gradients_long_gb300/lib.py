"""ctypes binding of libadj.so (include/adj.h): argument marshalling only.

Every function takes device pointers as ints, torch tensors or None, forwards them
to the C ABI unchanged and raises ``AdjError`` on a non-zero status.  There is no
fallback: if the library has not been built the first call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libadj.so")

F32, BF16 = 0, 1
OP_FWD, OP_BWD_FULL, OP_BWD_TRUNC, OP_PARAM, OP_LOSS = 0, 1, 2, 3, 4
OP_SEL_FWD, OP_SEL_BWD, OP_SEL_PARAM = 5, 6, 7
STATUS = {0: "ADJ_OK", 1: "ADJ_EINVAL", 2: "ADJ_ESHAPE", 3: "ADJ_EALIGN", 4: "ADJ_EDTYPE",
          5: "ADJ_EWORKSPACE", 6: "ADJ_ECUDA", 7: "ADJ_ETIMEOUT"}
EXPORTS = ("adj_workspace_bytes", "adj_fwd_scan", "adj_loss_mse", "adj_bwd_full", "adj_bwd_trunc",
           "adj_param_grad", "adj_stream_status", "adj_status_str", "adj_launch_count", "adj_profile_enable",
           "adj_profile_reset", "adj_profile_kernels", "adj_profile_name", "adj_profile_read", "adj_rms_norm",
           "adj_rms_norm_bwd", "adj_selftest_waits", "adj_selftest_ws_bytes", "adj_sel_fwd", "adj_sel_bwd",
           "adj_sel_param_grad", "adj_sel_rowdot_cols")


class AdjError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("P", ctypes.c_int32), ("N", ctypes.c_int32),
                ("x_dtype", ctypes.c_int32), ("d_dtype", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [("W_in", ctypes.c_void_p), ("b_a", ctypes.c_void_p), ("W_o", ctypes.c_void_p)]


class SelWeights(ctypes.Structure):
    """adj_sel_weights: W_in [P, P+2N], b_dt [P], A [P,N]."""
    _fields_ = [("W_in", ctypes.c_void_p), ("b_dt", ctypes.c_void_p), ("A", ctypes.c_void_p)]


_lib = None
_VP, _SZ, _I64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64
_PD, _PW, _PS = ctypes.POINTER(Dims), ctypes.POINTER(Weights), ctypes.POINTER(SelWeights)


def load(path: str = LIB_PATH):
    """Open libadj.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libadj.so is not built ({path}); run adjoint_gradients_long_gb300.build.build()")
        lib = ctypes.CDLL(path)
        lib.adj_workspace_bytes.argtypes = [_PD, ctypes.c_int, _I64]
        lib.adj_workspace_bytes.restype = _SZ
        lib.adj_fwd_scan.argtypes = [_PD, _PW] + [_VP] * 8 + [_SZ, _VP]
        lib.adj_loss_mse.argtypes = [_PD] + [_VP] * 6 + [_SZ, _VP]
        lib.adj_bwd_full.argtypes = [_PD, _PW] + [_VP] * 11 + [_SZ, _VP]
        lib.adj_bwd_trunc.argtypes = [_PD, _PW] + [_VP] * 10 + [_I64, _VP, _SZ, _VP]
        lib.adj_param_grad.argtypes = [_PD, _PW] + [_VP] * 15 + [ctypes.c_int, _VP, _SZ, _VP]
        lib.adj_rms_norm.argtypes = [_PD] + [_VP] * 4
        lib.adj_sel_fwd.argtypes = [_PD, _PS] + [_VP] * 6 + [_SZ, _VP]
        lib.adj_sel_bwd.argtypes = [_PD, _PS] + [_VP] * 4 + [_I64] + [_VP] * 6 + [_SZ, _VP]
        lib.adj_sel_param_grad.argtypes = [_PD, _PS] + [_VP] * 8 + [ctypes.c_int, _VP, _SZ, _VP]
        lib.adj_sel_rowdot_cols.argtypes = [_PD]
        lib.adj_sel_rowdot_cols.restype = _SZ
        lib.adj_selftest_waits.argtypes = [_VP, _SZ, ctypes.c_int, _VP]
        lib.adj_selftest_waits.restype = ctypes.c_int
        lib.adj_selftest_ws_bytes.argtypes = []
        lib.adj_selftest_ws_bytes.restype = _SZ
        lib.adj_rms_norm_bwd.argtypes = [_PD] + [_VP] * 6
        lib.adj_stream_status.argtypes = [_VP, _VP]
        lib.adj_status_str.argtypes = [ctypes.c_int]
        lib.adj_status_str.restype = ctypes.c_char_p
        lib.adj_launch_count.restype = ctypes.c_ulonglong
        lib.adj_profile_enable.argtypes = [ctypes.c_int]
        lib.adj_profile_name.argtypes = [ctypes.c_int]
        lib.adj_profile_name.restype = ctypes.c_char_p
        lib.adj_profile_read.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)]
        lib.adj_profile_read.restype = ctypes.c_int
        for f in ("adj_fwd_scan", "adj_loss_mse", "adj_bwd_full", "adj_bwd_trunc", "adj_param_grad",
                  "adj_stream_status", "adj_rms_norm", "adj_rms_norm_bwd", "adj_sel_fwd", "adj_sel_bwd",
                  "adj_sel_param_grad"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def ptr(x):
    """Device address of a tensor / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(st: int, what: str):
    if st != 0:
        raise AdjError(what, st)


def dims(B, T, P, N, x_dtype=F32, d_dtype=F32) -> Dims:
    return Dims(B, T, P, N, x_dtype, d_dtype)


def weights(W_in, b_a, W_o) -> Weights:
    return Weights(ptr(W_in), ptr(b_a), ptr(W_o))


def workspace_bytes(d: Dims, op: int, Tbar: int = 0) -> int:
    return load().adj_workspace_bytes(ctypes.byref(d), op, Tbar)


def fwd_scan(d, w, xhat, xres, a, c, h, y, y_x, ws, ws_bytes, stream=None):
    _check(load().adj_fwd_scan(ctypes.byref(d), ctypes.byref(w), ptr(xhat), ptr(xres), ptr(a), ptr(c), ptr(h),
                               ptr(y), ptr(y_x), ptr(ws), ws_bytes, _stream(stream)), "adj_fwd_scan")


def loss_mse(d, y, target, gy, loss, ws, ws_bytes, stream=None, gy_x=None):
    _check(load().adj_loss_mse(ctypes.byref(d), ptr(y), ptr(target), ptr(gy), ptr(gy_x), ptr(loss), ptr(ws),
                               ws_bytes, _stream(stream)), "adj_loss_mse")


def bwd_full(d, w, a, c, h, gy, D_a, D_u, D_c, E, ws, ws_bytes, stream=None, dz=None, gy_x=None):
    _check(load().adj_bwd_full(ctypes.byref(d), ctypes.byref(w), ptr(a), ptr(c), ptr(h), ptr(gy), ptr(gy_x),
                               ptr(D_a), ptr(D_u), ptr(D_c), ptr(E), ptr(dz), ptr(ws), ws_bytes, _stream(stream)),
           "adj_bwd_full")


def bwd_trunc(d, w, a, c, h, gy, D_a, D_u, D_c, E, Tbar, ws, ws_bytes, stream=None, dz=None, gy_x=None):
    _check(load().adj_bwd_trunc(ctypes.byref(d), ctypes.byref(w), ptr(a), ptr(c), ptr(h), ptr(gy), ptr(gy_x),
                                ptr(D_a), ptr(D_u), ptr(D_c), ptr(E), ptr(dz), int(Tbar), ptr(ws), ws_bytes,
                                _stream(stream)), "adj_bwd_trunc")


def param_grad(d, w, xhat, D_a, D_u, D_c, E, gy, dW_in, db_a, dW_o, gy_prev, dxhat, accumulate, ws, ws_bytes,
               stream=None, r=None, dz=None, gy_x=None, gy_prev_x=None):
    _check(load().adj_param_grad(ctypes.byref(d), ctypes.byref(w), ptr(xhat), ptr(D_a), ptr(D_u), ptr(D_c), ptr(E),
                                 ptr(gy), ptr(gy_x), ptr(dW_in), ptr(db_a), ptr(dW_o), ptr(gy_prev), ptr(gy_prev_x),
                                 ptr(dxhat), ptr(r), ptr(dz), int(accumulate), ptr(ws), ws_bytes, _stream(stream)),
           "adj_param_grad")


def rms_norm(d, y, xhat, r, stream=None):
    _check(load().adj_rms_norm(ctypes.byref(d), ptr(y), ptr(xhat), ptr(r), _stream(stream)), "adj_rms_norm")


def rms_norm_bwd(d, y, r, dxhat, gy, gy_prev, stream=None):
    _check(load().adj_rms_norm_bwd(ctypes.byref(d), ptr(y), ptr(r), ptr(dxhat), ptr(gy), ptr(gy_prev),
                                   _stream(stream)), "adj_rms_norm_bwd")


def stream_status(ws, stream=None) -> int:
    return load().adj_stream_status(ptr(ws), _stream(stream))


def status_str(s: int) -> str:
    return load().adj_status_str(s).decode()


def launch_count() -> int:
    return int(load().adj_launch_count())


def profile_enable(on: bool = True):
    load().adj_profile_enable(int(on))


def profile_reset():
    load().adj_profile_reset()


def profile_read() -> dict:
    """{kernel kind: (launches, total device ms)} recorded since the last reset."""
    L = load()
    out = {}
    for i in range(L.adj_profile_kernels()):
        n, ms = ctypes.c_int64(0), ctypes.c_double(0.0)
        _check(L.adj_profile_read(i, ctypes.byref(n), ctypes.byref(ms)), "adj_profile_read")
        if n.value:
            out[L.adj_profile_name(i).decode()] = (int(n.value), float(ms.value))
    return out


def selftest_ws_bytes() -> int:
    return int(load().adj_selftest_ws_bytes())


def selftest_waits(ws, ws_bytes, which, stream=None):
    _check(load().adj_selftest_waits(ptr(ws), ws_bytes, int(which), _stream(stream)), "adj_selftest_waits")


# ---------------------------------------------------------------- the general selective layer
def sel_weights(W_in, b_dt, A) -> SelWeights:
    return SelWeights(ptr(W_in), ptr(b_dt), ptr(A))


def sel_fwd(d, w, xhat, z, h, y, ws, ws_bytes, stream=None, xres=None):
    _check(load().adj_sel_fwd(ctypes.byref(d), ctypes.byref(w), ptr(xhat), ptr(xres), ptr(z), ptr(h), ptr(y),
                              ptr(ws), ws_bytes, _stream(stream)), "adj_sel_fwd")


def sel_rowdot_cols(d) -> int:
    return int(load().adj_sel_rowdot_cols(ctypes.byref(d)))


def sel_bwd(d, w, xhat, z, h, gy, Tbar, dz, dA, ws, ws_bytes, stream=None, r=None, gadd=None, rowdot=None):
    _check(load().adj_sel_bwd(ctypes.byref(d), ctypes.byref(w), ptr(xhat), ptr(z), ptr(h), ptr(gy),
                              0 if Tbar is None else int(Tbar), ptr(dz), ptr(dA), ptr(r), ptr(gadd), ptr(rowdot),
                              ptr(ws), ws_bytes, _stream(stream)), "adj_sel_bwd")


def sel_param_grad(d, xhat, dz, dW_in, db_dt, accumulate, ws, ws_bytes, stream=None, w=None, r=None, gadd=None,
                   rowdot=None, gy_prev=None):
    _check(load().adj_sel_param_grad(ctypes.byref(d), None if w is None else ctypes.byref(w), ptr(xhat), ptr(dz),
                                     ptr(dW_in), ptr(db_dt), ptr(r), ptr(gadd), ptr(rowdot), ptr(gy_prev),
                                     int(accumulate), ptr(ws), ws_bytes, _stream(stream)), "adj_sel_param_grad")
