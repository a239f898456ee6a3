"""Python side of the fp64 oracle: builds and calls ``adj_oracle.c``, runs the stack.

TEST INFRASTRUCTURE ONLY: the product never imports this module.

Source: the review page "Adjoint sharding for very long context training of state
space models" (pith.science), cited as [AS].

Stack semantics ([AS] What carries the argument: residual identity
y^K = y^0 + sum_k ytilde^k; Core claim: Proposition 3; Load-bearing premise: the
layers read "normalized inputs"):
  y^0 = xhat^1 = the input; for k >= 2 the layer input is the normalised residual
  stream xhat^k = y^{k-1} / r^{k-1}, r = sqrt(mean_p (y^{k-1}_p)^2 + EPS) per token;
  y^k = y^{k-1} + ytilde^k(xhat^k).
  L = sum_{b,t} 1/2 ||y^K_t - target_t||^2, gy^K = y^K - target.
  Layer k's VJP sums are seeded with its total cotangent gy^k = dL/dy^k, and
  gy^{k-1} = gy^k + J_k^T dxhat^k (the residual path plus the layer's input path,
  J_k = dxhat^k/dy^{k-1}: dy = (dxhat - xhat mean_p(xhat dxhat)) / r; J_1 = identity).
  ``cotangent="top"`` instead seeds every layer with gy^K, holding the layer
  inputs fixed -- the other reading of Proposition 3, kept for comparison.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

LITERAL = 0
AGGREGATED = 1
EPS = 1e-6      # normalisation epsilon of the stacked layer inputs

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "adj_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liborc.so")
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile adj_oracle.c with gcc into oracle/_build/liborc.so (with OpenMP when the
    compiler has it; the results do not depend on the thread count)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        base = ["gcc", "-O3", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        if subprocess.call(base[:1] + ["-fopenmp"] + base[1:], stderr=subprocess.DEVNULL) != 0:
            subprocess.check_call(base)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.orc_layer_forward.argtypes = [_I64] * 4 + [_D] * 12
    lib.orc_layer_forward.restype = None
    lib.orc_layer_grad.argtypes = [_I64] * 5 + [ctypes.c_int] + [_D] * 16
    lib.orc_layer_grad.restype = _I64
    lib.orc_threads.argtypes = [ctypes.c_int]
    lib.orc_threads.restype = ctypes.c_int
    return lib


def use_library(path):
    """Point the oracle at another build of adj_oracle.c (None restores the default).

    Used only by the mutation tests, which compile deliberately broken copies."""
    global _lib
    _lib = None if path is None else _bind(path)


def _load():
    global _lib
    if _lib is None:
        lib = _bind(build())
        _lib = lib
    return _lib


def threads(n: int = 0) -> int:
    """Set the oracle's thread count (n > 0) and return the count in use."""
    return int(_load().orc_threads(int(n)))


def _p(x):
    return x.ctypes.data_as(_D)


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def layer_forward(W: dict, xhat: np.ndarray, xres=None) -> dict:
    """One layer forward in fp64.  xhat [B,T,P] (layer input), xres [B,T,P] (residual
    input, default xhat); returns a, u, c, h [B,T,N] and y = xres + ytilde [B,T,P]."""
    lib = _load()
    xhat = _f64(xhat)
    xr = None if xres is None else _f64(xres)
    B, T, P = xhat.shape
    N = W["W_a"].shape[1]
    Wa, WB, Wc, ba, Wo = (_f64(W[k]) for k in ("W_a", "W_B", "W_c", "b_a", "W_o"))
    a, u, c, h = (np.empty((B, T, N)) for _ in range(4))
    y = np.empty((B, T, P))
    lib.orc_layer_forward(B, T, P, N, _p(Wa), _p(WB), _p(Wc), _p(ba), _p(Wo), _p(xhat),
                          None if xr is None else _p(xr), _p(a), _p(u), _p(c), _p(h), _p(y))
    return dict(a=a, u=u, c=c, h=h, y=y, xhat=xhat)


def layer_grad(W: dict, st: dict, gy: np.ndarray, Tbar=None, mode: int = AGGREGATED) -> dict:
    """Adjoint-sharding gradient of one layer for the cotangent gy = dL/dy (fp64).

    st holds the layer's forward states (xhat, a, c, h).  Tbar None = full adjoint.
    Returns dW_a, dW_B, dW_c [P,N], db_a [N], dW_o [N,P], dxhat [B,T,P] (input path
    only), mu [B,T,N] (sum over t of the adjoint vectors) and the VJP pair count.
    """
    lib = _load()
    xhat, a, c, h = (_f64(st[k]) for k in ("xhat", "a", "c", "h"))
    gy = _f64(gy)
    B, T, P = xhat.shape
    N = a.shape[2]
    Wa, WB, Wc, Wo = (_f64(W[k]) for k in ("W_a", "W_B", "W_c", "W_o"))
    dWa, dWB, dWc = (np.empty((P, N)) for _ in range(3))
    dba = np.empty((N,))
    dWo = np.empty((N, P))
    dx = np.empty((B, T, P))
    mu = np.empty((B, T, N))
    count = lib.orc_layer_grad(B, T, P, N, 0 if Tbar is None else int(Tbar), mode,
                               _p(Wa), _p(WB), _p(Wc), _p(Wo), _p(xhat), _p(a), _p(c), _p(h),
                               _p(gy), _p(dWa), _p(dWB), _p(dWc), _p(dba), _p(dWo), _p(dx), _p(mu))
    return dict(dW_a=dWa, dW_B=dWB, dW_c=dWc, db_a=dba, dW_o=dWo, dxhat=dx, mu=mu, vjp_count=int(count))


def normalize(y: np.ndarray):
    """xhat = y / r, r = sqrt(mean_p y_p^2 + EPS) per token.  Returns (xhat, r[...,1])."""
    r = np.sqrt(np.mean(y * y, axis=-1, keepdims=True) + EPS)
    return y / r, r


def normalize_vjp(xhat: np.ndarray, r: np.ndarray, dxhat: np.ndarray) -> np.ndarray:
    """Cotangent of y for xhat = y / r: (dxhat - xhat mean_p(xhat dxhat)) / r."""
    return (dxhat - xhat * np.mean(xhat * dxhat, axis=-1, keepdims=True)) / r


def stack_forward(layers: list, xhat: np.ndarray) -> list:
    """Forward through the residual stack; returns the per-layer states (each with y)."""
    states = []
    y_prev = _f64(xhat)
    for k, W in enumerate(layers):
        if k == 0:
            st = layer_forward(W, y_prev)
        else:
            x, r = normalize(y_prev)
            st = layer_forward(W, x, y_prev)
            st["r_in"] = r
        states.append(st)
        y_prev = st["y"]
    return states


def loss_and_cotangent(y: np.ndarray, target: np.ndarray):
    """L = sum 1/2 ||y - target||^2 and gy = y - target (fp64)."""
    r = _f64(y) - _f64(target)
    return 0.5 * float(np.sum(r * r)), r


def stack_grad(layers: list, xhat: np.ndarray, target: np.ndarray, Tbar=None,
               mode: int = AGGREGATED, cotangent: str = "total") -> dict:
    """Loss and per-layer gradients of the residual stack (Proposition 3 reading above).

    Returns dict(loss, states, grads=[per layer dict], gy=[cotangent seeding each layer],
    gx = dL/dxhat^1 (total reading), vjp_count).
    """
    states = stack_forward(layers, xhat)
    loss, gy = loss_and_cotangent(states[-1]["y"], target)
    gy_top = gy
    grads = [None] * len(layers)
    seeds = [None] * len(layers)
    count = 0
    for k in range(len(layers) - 1, -1, -1):
        seed = gy if cotangent == "total" else gy_top
        seeds[k] = seed
        gk = layer_grad(layers[k], states[k], seed, Tbar, mode)
        grads[k] = gk
        count += gk["vjp_count"]
        if cotangent == "total":
            dx = gk["dxhat"]
            if k > 0:
                dx = normalize_vjp(states[k]["xhat"], states[k]["r_in"], dx)
            gy = gy + dx
    return dict(loss=loss, states=states, grads=grads, gy=seeds, gx=gy, vjp_count=count)
