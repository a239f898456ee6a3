"""Driver of one general selective layer: device buffers and the libadj.so call sequence.
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
