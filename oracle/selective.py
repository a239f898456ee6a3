"""Python side of the fp64 oracle of the general selective layer: builds and calls
``sel_oracle.c``.

TEST INFRASTRUCTURE ONLY: the product never imports this module.

Source: the review page "Adjoint sharding for very long context training of state
space models" (pith.science), cited as [AS].  The layer is the pages' general form
h_t = A_t h_{t-1} + B_t xhat_t, y_t = C_t h_t ([AS] Circularity Check, assumptions) in
its selective reading (``sel_oracle.c`` states it): per channel p and state n,
dt = softplus(xhat W_dt + b_dt), B_t = xhat W_B, C_t = xhat W_C, Abar = exp(dt A),
h_t = Abar h_{t-1} + dt B_t xhat_t, y_t = xhat_t + sum_n C_t,n h_t,pn.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

LITERAL = 0
AGGREGATED = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sel_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsel.so")
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile sel_oracle.c with gcc (OpenMP when the compiler has it; results do not
    depend on the thread count)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        base = ["gcc", "-O3", "-std=c99", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
        if subprocess.call(base[:1] + ["-fopenmp"] + base[1:], stderr=subprocess.DEVNULL) != 0:
            subprocess.check_call(base)
        os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.sel_forward.argtypes = [_I64] * 4 + [_D] * 8
    lib.sel_forward.restype = None
    lib.sel_grad.argtypes = [_I64] * 5 + [ctypes.c_int] + [_D] * 12
    lib.sel_grad.restype = _I64
    lib.sel_dz_rows.argtypes = [_I64] * 5 + [_D] * 4 + [_I64, ctypes.POINTER(_I64), ctypes.POINTER(_I64), _D]
    lib.sel_dz_rows.restype = None
    return lib


def use_library(path):
    """Point the oracle at another build of sel_oracle.c (None restores the default).

    Used only by the mutation tests, which compile deliberately broken copies."""
    global _lib
    _lib = None if path is None else _bind(path)


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def _p(x):
    return x.ctypes.data_as(_D)


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


PARAMS = ("W_in", "b_dt", "A")


def forward(W: dict, xhat: np.ndarray, xres=None) -> dict:
    """One selective layer forward in fp64.  W: W_in [P, P+2N], b_dt [P], A [P,N];
    xhat [B,T,P] (the layer input), xres [B,T,P] (the residual input, default xhat).
    Returns z [B,T,P+2N] (bias included), h [B,T,P,N], y [B,T,P]."""
    lib = _load()
    x = _f64(xhat)
    xr = None if xres is None else _f64(xres)
    B, T, P = x.shape
    N = W["A"].shape[1]
    Win, bdt, A = (_f64(W[k]) for k in PARAMS)
    assert Win.shape == (P, P + 2 * N) and bdt.shape == (P,) and A.shape == (P, N)
    z = np.empty((B, T, P + 2 * N))
    h = np.empty((B, T, P, N))
    y = np.empty((B, T, P))
    lib.sel_forward(B, T, P, N, _p(x), None if xr is None else _p(xr), _p(Win), _p(bdt), _p(A), _p(z), _p(h),
                    _p(y))
    return dict(xhat=x, z=z, h=h, y=y)


def grad(W: dict, st: dict, gy: np.ndarray, Tbar=None, mode: int = AGGREGATED, want_mu: bool = False) -> dict:
    """Adjoint-sharding gradient of one selective layer for gy = dL/dy (fp64).

    st: the forward states (xhat, z, h).  Tbar None = full adjoint.  Returns dz
    [B,T,P+2N] (the cotangent of z: dt part through the softplus, then dB, dC), dW_in,
    db_dt, dA, dxhat [B,T,P] (the input path's cotangent), the pair count and, with
    want_mu, mu [B,T,P,N] (the window sums of the adjoint vectors)."""
    lib = _load()
    x, z, h = (_f64(st[k]) for k in ("xhat", "z", "h"))
    gy = _f64(gy)
    B, T, P = x.shape
    N = h.shape[3]
    A, Win = _f64(W["A"]), _f64(W["W_in"])
    dz = np.empty_like(z)
    dWin = np.empty((P, P + 2 * N))
    dbdt = np.empty((P,))
    dA = np.empty((P, N))
    dx = np.empty((B, T, P))
    mu = np.empty((B, T, P, N)) if want_mu else None
    count = lib.sel_grad(B, T, P, N, 0 if Tbar is None else int(Tbar), mode, _p(x), _p(Win), _p(A), _p(z),
                         _p(h), _p(gy), _p(dz), _p(dWin), _p(dbdt), _p(dA), None if mu is None else _p(mu), _p(dx))
    out = dict(dz=dz, dW_in=dWin, db_dt=dbdt, dA=dA, dxhat=dx, vjp_count=int(count))
    if want_mu:
        out["mu"] = mu
    return out


def loss_and_cotangent(y: np.ndarray, target: np.ndarray):
    """L = sum 1/2 ||y - target||^2 and gy = y - target (fp64)."""
    d = _f64(y) - _f64(target)
    return 0.5 * float(np.sum(d * d)), d


def dz_rows(W: dict, xhat: np.ndarray, target: np.ndarray, rows, Tbar=None) -> np.ndarray:
    """dz at sampled rows [(b, t), ...] of a long sequence (fp64): the window sums and VJPs
    of those tokens only, with the forward recurrence run over every token before them.
    The projection z = xhat W_in + [b_dt, 0, 0] is taken with a library matmul."""
    lib = _load()
    x = _f64(xhat)
    B, T, P = x.shape
    N = W["A"].shape[1]
    A = _f64(W["A"])
    z = x.reshape(B * T, P) @ _f64(W["W_in"])
    z[:, :P] += _f64(W["b_dt"])
    z = np.ascontiguousarray(z)
    tg = _f64(target)
    sb = np.ascontiguousarray([r[0] for r in rows], dtype=np.int64)
    stt = np.ascontiguousarray([r[1] for r in rows], dtype=np.int64)
    out = np.empty((len(rows), P + 2 * N))
    pi = ctypes.POINTER(_I64)
    lib.sel_dz_rows(B, T, P, N, 0 if Tbar is None else int(Tbar), _p(x), _p(A), _p(z), _p(tg), len(rows),
                    sb.ctypes.data_as(pi), stt.ctypes.data_as(pi), _p(out))
    return out


def stack_forward(layers: list, xhat: np.ndarray) -> list:
    """Forward through a residual stack of selective layers ([AS] What carries the argument:
    y^K = y^0 + sum_k ytilde^k; layer 1 reads the input, layer k >= 2 the residual stream
    normalised to unit root-mean-square per token, as the diagonal stack does).  Returns the
    per-layer states, each with y; layers k >= 2 also hold r_in."""
    from .oracle import normalize
    states = []
    y_prev = _f64(xhat)
    for k, W in enumerate(layers):
        if k == 0:
            st = forward(W, y_prev)
        else:
            x, r = normalize(y_prev)
            st = forward(W, x, y_prev)
            st["r_in"] = r
        states.append(st)
        y_prev = st["y"]
    return states


def stack_grad(layers: list, xhat: np.ndarray, target: np.ndarray, Tbar=None, mode: int = AGGREGATED) -> dict:
    """Loss and per-layer gradients of the selective stack ([AS] Core claim, Proposition 3):
    layer k is seeded with its total cotangent gy^k, and gy^{k-1} = gy^k + J_k^T dxhat^k
    through the normalisation (layer 1's input gradient is returned as gx)."""
    from .oracle import normalize_vjp
    states = stack_forward(layers, xhat)
    loss, gy = loss_and_cotangent(states[-1]["y"], target)
    grads = [None] * len(layers)
    seeds = [None] * len(layers)
    count = 0
    for k in range(len(layers) - 1, -1, -1):
        seeds[k] = gy
        gk = grad(layers[k], states[k], gy, Tbar, mode)
        grads[k] = gk
        count += gk["vjp_count"]
        dx = gk["dxhat"]
        if k > 0:
            dx = normalize_vjp(states[k]["xhat"], states[k]["r_in"], dx)
        gy = gy + dx
    return dict(loss=loss, states=states, grads=grads, gy=seeds, gx=gy, vjp_count=count)
