"""Drivers of one general selective layer and of a residual stack of them: device buffers
and the libadj.so call sequence.
PyTorch provides device memory and the stream; every arithmetic step runs in the
library's kernels.

Layer (the review page "Adjoint sharding for very long context training of state space
models" [AS], Circularity Check, assumptions: h_t = A_t h_{t-1} + B_t xhat_t,
y_t = C_t h_t, in its selective reading; include/adj.h states it in full).  One step:
  adj_sel_fwd          z = xhat W_in; h; y = xhat + sum_n C h
  adj_loss_mse         gy = y - target, L = sum 1/2 ||y - target||^2
  adj_sel_bwd          dz (the cotangent of z) and dA, full or truncated window
                       ([AS] Core claim, Proposition 2 and its truncation)
  adj_sel_param_grad   dW_in = xhat^T dz, db_dt = sum_t dz[:, :P]
"""
from __future__ import annotations

import numpy as np
import torch

from . import lib
from .stack import _dev_bf16, _dev_f32


class SelLayer:
    """Buffers for one selective-layer shape.  x_bf16: xhat and W_in stored as bf16 (and
    dz, the parameter GEMM's operand, as bf16)."""

    def __init__(self, B, T, P, N, x_bf16=False, device="cuda", Tbar=None):
        self.B, self.T, self.P, self.N = B, T, P, N
        self.x_bf16 = x_bf16
        self.device = torch.device(device)
        dt = lib.BF16 if x_bf16 else lib.F32
        self.dims = lib.dims(B, T, P, N, dt, dt)
        xt = torch.bfloat16 if x_bf16 else torch.float32
        dev = self.device
        zeros = lambda *s, dtype=torch.float32: torch.zeros(*s, dtype=dtype, device=dev)  # noqa: E731
        ZW = P + 2 * N
        self.x = zeros(B, T, P, dtype=xt)
        self.target = zeros(B, T, P)
        self.W_in = zeros(P, ZW, dtype=xt)
        self.b_dt = zeros(P)
        self.A = zeros(P, N)
        self.z = zeros(B, T, ZW)
        self.h = zeros(B, T, P, N)
        self.y = zeros(B, T, P)
        self.gy = zeros(B, T, P)
        self.dz = zeros(B, T, ZW, dtype=xt)
        self.dA = zeros(P, N)
        self.dW_in = zeros(P, ZW)
        self.db_dt = zeros(P)
        self.loss = torch.zeros(1, dtype=torch.float64, device=dev)
        tb = 0 if Tbar is None else int(Tbar)
        need = max(lib.workspace_bytes(self.dims, lib.OP_SEL_FWD), lib.workspace_bytes(self.dims, lib.OP_SEL_BWD, tb),
                   lib.workspace_bytes(self.dims, lib.OP_SEL_BWD, 0), lib.workspace_bytes(self.dims, lib.OP_SEL_PARAM),
                   lib.workspace_bytes(self.dims, lib.OP_LOSS))
        if need == 0:
            raise ValueError("unsupported selective-layer sizes or window")
        self.ws_bytes = int(need)
        self.ws = torch.zeros(self.ws_bytes // 4 + 64, dtype=torch.int32, device=dev)
        self.w = lib.sel_weights(self.W_in, self.b_dt, self.A)

    def load(self, inputs: dict):
        """Copy seeded host inputs (synth.make_sel_inputs) to the device."""
        dev = self.device
        put = _dev_bf16 if self.x_bf16 else _dev_f32
        self.x.copy_(put(inputs["xhat"], dev))
        self.target.copy_(_dev_f32(inputs["target"], dev))
        self.W_in.copy_(put(inputs["W_in"], dev))
        self.b_dt.copy_(_dev_f32(inputs["b_dt"], dev))
        self.A.copy_(_dev_f32(inputs["A"], dev))

    def forward(self, stream=None):
        lib.sel_fwd(self.dims, self.w, self.x, self.z, self.h, self.y, self.ws, self.ws_bytes, stream)

    def loss_grad(self, stream=None):
        lib.loss_mse(self.dims, self.y, self.target, self.gy, self.loss, self.ws, self.ws_bytes, stream)

    def backward(self, Tbar=None, stream=None, accumulate=False):
        lib.sel_bwd(self.dims, self.w, self.x, self.z, self.h, self.gy, Tbar, self.dz, self.dA, self.ws,
                    self.ws_bytes, stream)
        lib.sel_param_grad(self.dims, self.x, self.dz, self.dW_in, self.db_dt, int(accumulate), self.ws,
                           self.ws_bytes, stream)

    def step(self, Tbar=None, stream=None):
        self.forward(stream)
        self.loss_grad(stream)
        self.backward(Tbar, stream)

    def capture(self, Tbar=None):
        """A CUDA graph of one step on these buffers."""
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self.step(Tbar)
        torch.cuda.current_stream(self.device).wait_stream(side)
        with torch.cuda.graph(g):
            self.step(Tbar)
        return g

    def status(self, stream=None) -> int:
        return lib.stream_status(self.ws, stream)

    def grads_numpy(self):
        return dict(W_in=self.dW_in.double().cpu().numpy(), b_dt=self.db_dt.double().cpu().numpy(),
                    A=self.dA.double().cpu().numpy())


class SelStack:
    """A residual stack of K selective layers ([AS] What carries the argument: y^K = y^0 +
    sum_k ytilde^k; Load-bearing premise: normalised layer inputs).  One step:
      for k = 1..K: adj_rms_norm(y^{k-1})   xhat^k = y^{k-1} / r   (k >= 2; xhat^1 = input)
                    adj_sel_fwd(k)          z^k, h^k; y^k = y^{k-1} + sum_n C h (y^1: input + ...)
      adj_loss_mse                          gy^K = y^K - target, L
      for k = K..1: adj_sel_bwd(k)          dz, dA^k and (k >= 2) the input term and row dots
                    adj_sel_param_grad(k)   dW_in^k, db_dt^k and (k >= 2) gy^{k-1} through the
                                            projection, the input term and the normalisation
    x_bf16: xhat^k and W_in^k stored as bf16 (and dz)."""

    def __init__(self, B, T, P, N, K, x_bf16=False, device="cuda", Tbar=None):
        self.B, self.T, self.P, self.N, self.K = B, T, P, N, K
        self.x_bf16 = x_bf16
        self.device = torch.device(device)
        dt = lib.BF16 if x_bf16 else lib.F32
        self.dims = lib.dims(B, T, P, N, dt, dt)
        xt = torch.bfloat16 if x_bf16 else torch.float32
        dev = self.device
        zeros = lambda *s, dtype=torch.float32: torch.zeros(*s, dtype=dtype, device=dev)  # noqa: E731
        ZW = P + 2 * N
        self.x = [zeros(B, T, P, dtype=xt) for _ in range(K)]     # layer inputs xhat^k
        self.r = [zeros(B, T) for _ in range(K - 1)]               # rms of y^k, the next layer's input
        self.z = [zeros(B, T, ZW) for _ in range(K)]
        self.h = [zeros(B, T, P, N) for _ in range(K)]
        self.y = [zeros(B, T, P) for _ in range(K)]                # the residual stream y^k
        self.target = zeros(B, T, P)
        self.gy = [zeros(B, T, P), zeros(B, T, P)]
        cols = lib.sel_rowdot_cols(self.dims)
        if cols == 0:
            raise ValueError("unsupported selective-layer sizes")
        self.gadd = zeros(B, T, P) if K > 1 else None
        self.rowdot = zeros(B * T, cols) if K > 1 else None
        self.dz = zeros(B, T, ZW, dtype=xt)
        self.loss = torch.zeros(1, dtype=torch.float64, device=dev)
        self.W_in = [zeros(P, ZW, dtype=xt) for _ in range(K)]
        self.b_dt = [zeros(P) for _ in range(K)]
        self.A = [zeros(P, N) for _ in range(K)]
        self.dW_in = [zeros(P, ZW) for _ in range(K)]
        self.db_dt = [zeros(P) for _ in range(K)]
        self.dA = [zeros(P, N) for _ in range(K)]
        tb = 0 if Tbar is None else int(Tbar)
        need = max(lib.workspace_bytes(self.dims, lib.OP_SEL_FWD), lib.workspace_bytes(self.dims, lib.OP_SEL_BWD, tb),
                   lib.workspace_bytes(self.dims, lib.OP_SEL_BWD, 0), lib.workspace_bytes(self.dims, lib.OP_SEL_PARAM),
                   lib.workspace_bytes(self.dims, lib.OP_LOSS))
        if need == 0:
            raise ValueError("unsupported selective-layer sizes or window")
        self.ws_bytes = int(need)
        self.ws = torch.zeros(self.ws_bytes // 4 + 64, dtype=torch.int32, device=dev)
        self.w = [lib.sel_weights(self.W_in[k], self.b_dt[k], self.A[k]) for k in range(K)]

    def load(self, inputs: dict):
        """Copy seeded host inputs (synth.make_sel_stack_inputs) to the device."""
        dev = self.device
        put = _dev_bf16 if self.x_bf16 else _dev_f32
        self.x[0].copy_(put(inputs["xhat"], dev))
        self.target.copy_(_dev_f32(inputs["target"], dev))
        for k, W in enumerate(inputs["layers"]):
            self.W_in[k].copy_(put(W["W_in"], dev))
            self.b_dt[k].copy_(_dev_f32(W["b_dt"], dev))
            self.A[k].copy_(_dev_f32(W["A"], dev))

    def forward(self, stream=None):
        for k in range(self.K):
            xres = None
            if k > 0:
                lib.rms_norm(self.dims, self.y[k - 1], self.x[k], self.r[k - 1], stream)
                xres = self.y[k - 1]
            lib.sel_fwd(self.dims, self.w[k], self.x[k], self.z[k], self.h[k], self.y[k], self.ws, self.ws_bytes,
                        stream, xres=xres)

    def loss_grad(self, stream=None):
        lib.loss_mse(self.dims, self.y[-1], self.target, self.gy[0], self.loss, self.ws, self.ws_bytes, stream)

    def backward(self, Tbar=None, stream=None, accumulate=False):
        """Layer K down to 1; afterwards seed(0) holds layer 1's total cotangent."""
        cur = 0
        for k in range(self.K - 1, -1, -1):
            gy = self.gy[cur]
            inp = k > 0
            r = self.r[k - 1] if inp else None
            gadd = self.gadd if inp else None
            rowdot = self.rowdot if inp else None
            lib.sel_bwd(self.dims, self.w[k], self.x[k], self.z[k], self.h[k], gy, Tbar, self.dz, self.dA[k], self.ws,
                        self.ws_bytes, stream, r=r, gadd=gadd, rowdot=rowdot)
            lib.sel_param_grad(self.dims, self.x[k], self.dz, self.dW_in[k], self.db_dt[k], int(accumulate), self.ws,
                               self.ws_bytes, stream, w=self.w[k] if inp else None, r=r, gadd=gadd, rowdot=rowdot,
                               gy_prev=self.gy[1 - cur] if inp else None)
            cur = 1 - cur
        self._seed0 = self.gy[1 - cur]

    def seed0(self):
        """Layer 1's total cotangent dL/dy^1 from the last backward."""
        return self._seed0

    def step(self, Tbar=None, stream=None):
        self.forward(stream)
        self.loss_grad(stream)
        self.backward(Tbar, stream)

    def capture(self, Tbar=None):
        """A CUDA graph of one step on these buffers."""
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self.step(Tbar)
        torch.cuda.current_stream(self.device).wait_stream(side)
        with torch.cuda.graph(g):
            self.step(Tbar)
        return g

    def status(self, stream=None) -> int:
        return lib.stream_status(self.ws, stream)

    def grads_numpy(self, k):
        return dict(W_in=self.dW_in[k].double().cpu().numpy(), b_dt=self.db_dt[k].double().cpu().numpy(),
                    A=self.dA[k].double().cpu().numpy())
