"""Independent checks for the oracle: step-by-step BPTT, per-term truncated BPTT,
complex-step and central finite differences (NumPy, fp64 / complex128).

TEST INFRASTRUCTURE ONLY.  Written separately from ``adj_oracle.c``: ordinary
reverse-mode differentiation through time with a running dL/dh, the way
backpropagation computes the gradient that the review page "Adjoint sharding for
very long context training of state space models" ([AS]) says adjoint sharding
reproduces exactly ([AS] The reading; If this is right, 4th bullet).

Model and stack: [AS] Assumptions (Sec. 3.1 SSM dynamics, Sec. 3.2 residual
structure), diagonal selective form a = sigmoid(x W_a + b_a), u = x W_B,
c = x W_c, h_t = a_t h_{t-1} + u_t, y^k = y^{k-1} + (c h) W_o with y^0 the input;
layer 1 reads the input, layer k >= 2 reads y^{k-1} scaled to unit root-mean-square
per token ([AS] Load-bearing premise: "normalized inputs"; EPS below).
"""
from __future__ import annotations

import numpy as np

PARAMS = ("W_a", "W_B", "W_c", "b_a", "W_o")
EPS = 1e-6


def forward(layers, xhat, dtype=np.float64):
    """Forward pass storing every intermediate; works for float64 and complex128."""
    y_prev = np.asarray(xhat, dtype=dtype)
    cache = []
    for li, W in enumerate(layers):
        Wa, WB, Wc, ba, Wo = (np.asarray(W[k], dtype=dtype) for k in PARAMS)
        if li == 0:
            x, rms = y_prev, None
        else:
            rms = np.sqrt(np.sum(y_prev * y_prev, axis=-1, keepdims=True) / y_prev.shape[-1] + EPS)
            x = y_prev / rms
        z = x @ Wa + ba
        a = 1.0 / (1.0 + np.exp(-z))
        u = x @ WB
        c = x @ Wc
        h = np.zeros_like(u)
        prev = np.zeros_like(u[:, 0])
        for t in range(x.shape[1]):
            prev = a[:, t] * prev + u[:, t]
            h[:, t] = prev
        y = y_prev + (c * h) @ Wo
        cache.append(dict(x=x, a=a, u=u, c=c, h=h, y=y, y_in=y_prev, rms=rms))
        y_prev = y
    return cache


def loss(layers, xhat, target, dtype=np.float64):
    y = forward(layers, xhat, dtype)[-1]["y"]
    r = y - np.asarray(target, dtype=dtype)
    return 0.5 * np.sum(r * r)


def backward(layers, cache, gy_top, Tbar=None):
    """Reverse-mode through the stack.

    Tbar None: ordinary BPTT with one running dL/dh_t per layer.
    Tbar given: per-loss-term truncated BPTT -- for each token t the direct
    cotangent of h_t (g_t c_t) is propagated back through at most Tbar-1
    transitions, separately for every t (brute force, O(T Tbar N)).  The
    cotangent handed to the layer below is gy + dxhat of the truncated layer
    gradient (a per-layer truncation).
    Returns (per-layer grads, dL/dxhat^1).
    """
    gy = np.array(gy_top, dtype=np.float64)
    grads = [None] * len(layers)
    for k in range(len(layers) - 1, -1, -1):
        W = layers[k]
        Wa, WB, Wc, Wo = (np.asarray(W[n], dtype=np.float64) for n in ("W_a", "W_B", "W_c", "W_o"))
        st = cache[k]
        x, a, c, h = st["x"], st["a"], st["c"], st["h"]
        Bn, T, _ = x.shape
        g = gy @ Wo.T                      # d L / d (c h)
        dWo = np.einsum("btn,btp->np", c * h, gy)
        dc = g * h
        dh_direct = g * c                 # d l_t / d h_t through y_t only
        dh = np.zeros_like(dh_direct)     # total dL/dh_t (full) or its truncated sum
        if Tbar is None:
            run = np.zeros_like(dh_direct[:, 0])
            for t in range(T - 1, -1, -1):
                run = dh_direct[:, t] + run
                dh[:, t] = run
                run = run * a[:, t]       # through h_t = a_t h_{t-1} + u_t to h_{t-1}
        else:
            for t in range(T):
                seed = dh_direct[:, t]
                for step in range(Tbar):
                    i = t - step
                    if i < 0:
                        break
                    dh[:, i] += seed
                    seed = seed * a[:, i]
        hprev = np.concatenate([np.zeros_like(h[:, :1]), h[:, :-1]], axis=1)
        du = dh
        dz = dh * hprev * a * (1.0 - a)
        grads[k] = dict(
            W_a=np.einsum("btp,btn->pn", x, dz), W_B=np.einsum("btp,btn->pn", x, du),
            W_c=np.einsum("btp,btn->pn", x, dc), b_a=dz.sum(axis=(0, 1)), W_o=dWo,
            mu=dh,
        )
        dx = dz @ Wa.T + du @ WB.T + dc @ Wc.T
        if st["rms"] is not None:
            # through x = y_in / rms(y_in): d y_in = dx / rms - y_in (y_in . dx) / (P rms^3)
            yi, rms = st["y_in"], st["rms"]
            dx = dx / rms - yi * np.sum(yi * dx, axis=-1, keepdims=True) / (yi.shape[-1] * rms ** 3)
        gy = gy + dx
    return grads, gy


def bptt_grad(layers, xhat, target, Tbar=None):
    cache = forward(layers, xhat)
    r = cache[-1]["y"] - np.asarray(target, dtype=np.float64)
    grads, gx = backward(layers, cache, r, Tbar)
    return dict(loss=0.5 * float(np.sum(r * r)), grads=grads, gx=gx)


def complex_step_grad(layers, xhat, target, step=1e-30):
    """dL/dtheta for every parameter by the complex-step derivative Im L(theta + i s e)/s.

    sigmoid is analytic, so this is exact up to rounding (no subtraction).
    """
    out = []
    for k, W in enumerate(layers):
        gk = {}
        for name in PARAMS:
            base = np.asarray(W[name], dtype=np.float64)
            g = np.empty(base.shape)
            for idx in np.ndindex(base.shape):
                pert = base.astype(np.complex128)
                pert[idx] += 1j * step
                lay = [dict(L) for L in layers]
                lay[k] = dict(W)
                lay[k][name] = pert
                g[idx] = loss(lay, xhat, target, dtype=np.complex128).imag / step
            gk[name] = g
        out.append(gk)
    return out


def central_diff_grad(layers, xhat, target, rel_step=1e-3):
    """dL/dtheta by the fourth-order central difference
    (8(f(+h) - f(-h)) - (f(+2h) - f(-2h))) / (12 h), h = rel_step * max(1, |theta|)."""
    out = []
    for k, W in enumerate(layers):
        gk = {}
        for name in PARAMS:
            base = np.asarray(W[name], dtype=np.float64)
            g = np.empty(base.shape)
            for idx in np.ndindex(base.shape):
                hstep = rel_step * max(1.0, abs(base[idx]))
                vals = []
                for m in (1, -1, 2, -2):
                    pert = base.copy()
                    pert[idx] += m * hstep
                    lay = [dict(L) for L in layers]
                    lay[k] = dict(W)
                    lay[k][name] = pert
                    vals.append(loss(lay, xhat, target))
                g[idx] = (8.0 * (vals[0] - vals[1]) - (vals[2] - vals[3])) / (12.0 * hstep)
            gk[name] = g
        out.append(gk)
    return out
