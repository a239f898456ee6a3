"""Independent checks for the selective-layer oracle: step-by-step BPTT, per-term
truncated BPTT, complex-step and central finite differences (NumPy, fp64 / complex128).

TEST INFRASTRUCTURE ONLY.  Written separately from ``sel_oracle.c``: ordinary
reverse-mode differentiation through time with a running dL/dh, the way
backpropagation computes the gradient that the review page "Adjoint sharding for very
long context training of state space models" ([AS]) says adjoint sharding reproduces
exactly ([AS] The reading; If this is right).

Layer (the pages' general form h_t = A_t h_{t-1} + B_t xhat_t, y_t = C_t h_t, [AS]
Circularity Check, assumptions, in its selective reading): z = xhat W_in + [b_dt,0,0],
dt = softplus(z[:P]), B_t = z[P:P+N], C_t = z[P+N:], Abar = exp(dt A),
h_t = Abar h_{t-1} + dt B_t xhat_t, y_t = xres_t + sum_n C_t,n h_t,pn;
L = sum 1/2 ||y - target||^2.  Stacks: layer 1 reads the input (xres = the input),
layer k >= 2 reads y^{k-1} scaled to unit root-mean-square per token (xres = y^{k-1}).
"""
from __future__ import annotations

import numpy as np

PARAMS = ("W_in", "b_dt", "A")


def _softplus(z):
    return np.log(1.0 + np.exp(z))


EPS = 1e-6


def forward(W, xhat, dtype=np.float64, xres=None):
    """Forward pass storing every intermediate; float64 or complex128."""
    x = np.asarray(xhat, dtype=dtype)
    xr = x if xres is None else np.asarray(xres, dtype=dtype)
    Win, bdt, A = (np.asarray(W[k], dtype=dtype) for k in PARAMS)
    P, N = A.shape
    z = x @ Win
    z[..., :P] += bdt
    dt = _softplus(z[..., :P])
    Bt, Ct = z[..., P:P + N], z[..., P + N:]
    Ab = np.exp(dt[..., :, None] * A)                       # [B,T,P,N]
    u = dt[..., :, None] * Bt[..., None, :] * x[..., :, None]
    h = np.zeros_like(u)
    prev = np.zeros_like(u[:, 0])
    for t in range(x.shape[1]):
        prev = Ab[:, t] * prev + u[:, t]
        h[:, t] = prev
    y = xr + np.einsum("btn,btpn->btp", Ct, h)
    return dict(x=x, z=z, dt=dt, Bt=Bt, Ct=Ct, Ab=Ab, h=h, y=y, A=A, Win=Win)


def loss(W, xhat, target, dtype=np.float64):
    c = forward(W, xhat, dtype)
    d = c["y"] - np.asarray(target, dtype=dtype)
    return 0.5 * np.sum(d * d), c


def _param_grads(c, ddt, dB, dC, dA, dxd):
    P = c["A"].shape[0]
    sig = 1.0 / (1.0 + np.exp(-c["z"][..., :P]))
    dz = np.concatenate([ddt * sig, dB, dC], axis=-1)
    x = c["x"]
    dW = np.einsum("btq,btj->qj", x, dz)
    dx = dxd + np.einsum("btj,pj->btp", dz, c["Win"])   # xhat's input path: the input term, the projection
    return dict(dW_in=dW, db_dt=dz[..., :P].sum(axis=(0, 1)), dA=dA, dz=dz, dxhat=dx)


def backward(c, gy, Tbar=None):
    """Gradient for the cotangent gy.  Tbar None: ordinary BPTT with one running dL/dh.
    Tbar = W: per-term truncated BPTT -- for every t, the loss term at t is backpropagated
    through its own W most recent steps only."""
    x, dt, Bt, Ct, Ab, h, A = (c[k] for k in ("x", "dt", "Bt", "Ct", "Ab", "h", "A"))
    Bn, T, P = x.shape
    gy = np.asarray(gy)
    ddt = np.zeros_like(dt)
    dB = np.zeros_like(Bt)
    dxd = np.zeros_like(x)
    dC = np.einsum("btp,btpn->btn", gy, h)
    dA = np.zeros_like(A)

    def step(i, dh):   # the VJP of step i for the cotangent dh on h_i; returns dh on h_{i-1}
        nonlocal dA
        hp = h[:, i - 1] if i > 0 else np.zeros_like(h[:, 0])
        dAb = dh * hp
        ddt[:, i] += np.einsum("bpn,bpn->bp", dAb, A[None] * Ab[:, i])
        dA = dA + np.einsum("bpn,bp->pn", dAb * Ab[:, i], dt[:, i])
        ddt[:, i] += np.einsum("bpn,bn->bp", dh, Bt[:, i]) * x[:, i]
        dB[:, i] += np.einsum("bpn,bp->bn", dh, dt[:, i] * x[:, i])
        dxd[:, i] += np.einsum("bpn,bn->bp", dh, Bt[:, i]) * dt[:, i]
        return Ab[:, i] * dh

    if Tbar is None or Tbar >= T:
        dh_next = np.zeros_like(h[:, 0])
        for t in range(T - 1, -1, -1):
            dh = gy[:, t, :, None] * Ct[:, t, None, :] + dh_next
            dh_next = step(t, dh)
    else:
        for t in range(T):
            dh = gy[:, t, :, None] * Ct[:, t, None, :]
            for i in range(t, max(-1, t - Tbar), -1):
                dh = step(i, dh)
    return _param_grads(c, ddt, dB, dC, dA, dxd)


def bptt_grad(W, xhat, target, Tbar=None):
    L, c = loss(W, xhat, target)
    return backward(c, c["y"] - np.asarray(target), Tbar)


def stack_loss(layers, xhat, target, dtype=np.float64):
    """Forward through the stack (normalised inputs for layers k >= 2); returns L and the caches."""
    y = np.asarray(xhat, dtype=dtype)
    caches = []
    for k, W in enumerate(layers):
        if k == 0:
            c = forward(W, y, dtype)
        else:
            r = np.sqrt(np.sum(y * y, axis=-1, keepdims=True) / y.shape[-1] + EPS)
            c = forward(W, y / r, dtype, xres=y)
            c["r"] = r
        caches.append(c)
        y = c["y"]
    d = y - np.asarray(target, dtype=dtype)
    return 0.5 * np.sum(d * d), caches


def stack_bptt_grad(layers, xhat, target, Tbar=None):
    """Per-layer gradients of the stack: each layer backpropagated (ordinary or per-term
    truncated BPTT) with its total cotangent, which then passes to the layer below through
    the residual and, by the chain rule written out, through the normalisation."""
    L, caches = stack_loss(layers, xhat, target)
    gy = caches[-1]["y"] - np.asarray(target)
    out = [None] * len(layers)
    for k in range(len(layers) - 1, -1, -1):
        g = backward(caches[k], gy, Tbar)
        out[k] = g
        dx = g["dxhat"]
        if k > 0:
            c = caches[k]
            xh, r = c["x"], c["r"]
            # xhat = y / r, r = sqrt(mean y^2 + eps): dy = dx / r - y (sum dx y) / (P r^3)
            y = xh * r
            dx = dx / r - y * np.sum(dx * y, axis=-1, keepdims=True) / (y.shape[-1] * r ** 3)
        gy = gy + dx
    return out


def stack_complex_step_grad(layers, xhat, target, k, name, step=1e-30):
    """Layer k's derivative of L with respect to parameter `name` by the complex step."""
    base = np.asarray(layers[k][name], dtype=np.float64)
    g = np.empty_like(base)
    for idx in np.ndindex(base.shape):
        Lc = [{q: np.asarray(W[q], dtype=np.complex128) for q in PARAMS} for W in layers]
        Lc[k][name] = Lc[k][name].copy()
        Lc[k][name][idx] += 1j * step
        L, _ = stack_loss(Lc, xhat, target, dtype=np.complex128)
        g[idx] = L.imag / step
    return g


def complex_step_grad(W, xhat, target, step=1e-30):
    """Every parameter's derivative by the complex step Im L(theta + i s e_k) / s."""
    out = {}
    for k in PARAMS:
        base = np.asarray(W[k], dtype=np.float64)
        g = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            Wc = {q: np.asarray(W[q], dtype=np.complex128) for q in PARAMS}
            Wc[k] = Wc[k].copy()
            Wc[k][idx] += 1j * step
            L, _ = loss(Wc, xhat, target, dtype=np.complex128)
            g[idx] = L.imag / step
        out[k] = g
    return out


def central_diff_grad(W, xhat, target, rel_step=1e-5):
    out = {}
    for k in PARAMS:
        base = np.asarray(W[k], dtype=np.float64)
        g = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            s = rel_step * max(1.0, abs(base[idx]))
            Wp = {q: np.asarray(W[q], dtype=np.float64).copy() for q in PARAMS}
            Wm = {q: np.asarray(W[q], dtype=np.float64).copy() for q in PARAMS}
            Wp[k][idx] += s
            Wm[k][idx] -= s
            g[idx] = (loss(Wp, xhat, target)[0] - loss(Wm, xhat, target)[0]) / (2 * s)
        out[k] = g
    return out
