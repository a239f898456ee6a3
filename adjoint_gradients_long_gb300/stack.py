"""Stack driver: sequences the libadj.so calls for a residual stack of diagonal
selective SSM layers on one GPU.  PyTorch provides device memory and the stream;
every arithmetic step runs in the library's kernels.

Order of one gradient step ([AS] = review page "Adjoint sharding for very long
context training of state space models"; [AS] Referee Report on Algorithm 1 for
the stored states, Core claim for Propositions 2 and 3, Load-bearing premise for
the normalised layer inputs):
  for k = 1..K: adj_rms_norm(y^{k-1})      xhat^k = y^{k-1} / r^{k-1}   (k >= 2; xhat^1 = input)
                adj_fwd_scan(k)            stores a^k, c^k, h^k; y^k = y^{k-1} + ytilde^k
  adj_loss_mse                             gy^K = y^K - target, L
  for k = K..1: adj_bwd_{full,trunc}(k)    VJP seeds D_a, D_u, D_c, E of layer k (k >= 2: and
                                           the row dots dz = xhat . dxhat)
                adj_param_grad(k)          dW_in^k, db_a^k, dW_o^k and (k >= 2)
                                           gy^{k-1} = gy^k + J^T dxhat^k through the normalisation
"""
from __future__ import annotations

import numpy as np
import torch

from . import lib
from .synth import bf16_bits


def _dev_f32(x, device):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)


def _dev_bf16(x, device):
    bits = torch.from_numpy(bf16_bits(np.ascontiguousarray(x, np.float32)).view(np.int16))
    return bits.to(device).view(torch.bfloat16)


class AdjStack:
    """Device buffers and call sequence for one workload shape.

    x_bf16: GEMM operands (xhat, W_in, W_o) stored as bf16; d_bf16: VJP seeds stored as bf16.
    """

    def __init__(self, B, T, P, N, K, x_bf16=False, d_bf16=False, device="cuda", Tbar=None):
        self.B, self.T, self.P, self.N, self.K = B, T, P, N, K
        self.x_bf16, self.d_bf16 = x_bf16, d_bf16
        self.device = torch.device(device)
        xd = lib.BF16 if x_bf16 else lib.F32
        dd = lib.BF16 if d_bf16 else lib.F32
        self.dims = lib.dims(B, T, P, N, xd, dd)
        xt = torch.bfloat16 if x_bf16 else torch.float32
        dt = torch.bfloat16 if d_bf16 else torch.float32
        dev = self.device
        z = lambda *s, dtype=torch.float32: torch.zeros(*s, dtype=dtype, device=dev)  # noqa: E731
        # per-layer stored states and outputs
        self.x = [z(B, T, P, dtype=xt) for _ in range(K)]    # layer inputs xhat^k (GEMM operands)
        self.r = [z(B, T) for _ in range(K - 1)]              # rms of y^k for the next layer's input
        self.a = [z(B, T, N) for _ in range(K)]
        self.c = [z(B, T, N) for _ in range(K)]
        self.h = [z(B, T, N) for _ in range(K)]
        self.y = [z(B, T, P) for _ in range(K)]                # fp32 residual stream y^k
        self.target = z(B, T, P)
        self.D = [z(B, T, N, dtype=dt) for _ in range(4)]     # D_a, D_u, D_c, E
        self.gy = [z(B, T, P), z(B, T, P)]
        # bf16 layers: the cotangents rounded to bf16, the operand their backward GEMMs read
        self.gy_x = [z(B, T, P, dtype=torch.bfloat16), z(B, T, P, dtype=torch.bfloat16)] if x_bf16 else [None, None]
        # per token and 128-channel group: xhat . dxhat of a normalised layer input
        self.dz = z(B * T, (N + 127) // 128) if K > 1 else None
        self.loss = torch.zeros(1, dtype=torch.float64, device=dev)
        self.W_in = [z(P, 3 * N, dtype=xt) for _ in range(K)]
        self.b_a = [z(N) for _ in range(K)]
        self.W_o = [z(N, P, dtype=xt) for _ in range(K)]
        self.dW_in = [z(P, 3 * N) for _ in range(K)]
        self.db_a = [z(N) for _ in range(K)]
        self.dW_o = [z(N, P) for _ in range(K)]
        tb = Tbar if Tbar is not None else T
        need = max(lib.workspace_bytes(self.dims, op, max(1, tb)) for op in
                   (lib.OP_FWD, lib.OP_BWD_FULL, lib.OP_BWD_TRUNC, lib.OP_PARAM, lib.OP_LOSS))
        self.ws_bytes = int(need)
        self.ws = torch.zeros(self.ws_bytes // 4 + 64, dtype=torch.int32, device=dev)
        self.w = [None] * K

    # ------------------------------------------------------------------ inputs
    def layer_input(self, k):
        return self.x[k]

    def load(self, inputs: dict):
        """Copy seeded host inputs (synth.make_inputs) to the device."""
        dev = self.device
        put = _dev_bf16 if self.x_bf16 else _dev_f32
        self.x[0].copy_(put(inputs["xhat"], dev))
        self.target.copy_(_dev_f32(inputs["target"], dev))
        for k, W in enumerate(inputs["layers"]):
            W_in = np.concatenate([W["W_a"], W["W_B"], W["W_c"]], axis=1)
            self.W_in[k].copy_(put(W_in, dev))
            self.b_a[k].copy_(_dev_f32(W["b_a"], dev))
            self.W_o[k].copy_(put(W["W_o"], dev))
        self._bind_weights()

    def _bind_weights(self):
        self.w = [lib.weights(self.W_in[k], self.b_a[k], self.W_o[k]) for k in range(self.K)]

    # ------------------------------------------------------------------ calls
    def forward(self, stream=None):
        for k in range(self.K):
            xres = None
            if k > 0:
                lib.rms_norm(self.dims, self.y[k - 1], self.x[k], self.r[k - 1], stream)
                xres = self.y[k - 1]
            lib.fwd_scan(self.dims, self.w[k], self.x[k], xres, self.a[k], self.c[k], self.h[k],
                         self.y[k], None, self.ws, self.ws_bytes, stream)

    def loss_grad(self, stream=None):
        lib.loss_mse(self.dims, self.y[-1], self.target, self.gy[0], self.loss, self.ws, self.ws_bytes, stream,
                     gy_x=self.gy_x[0])

    def backward(self, Tbar=None, stream=None, accumulate=False, on_layer=None):
        """Adjoint pass and parameter gradients, layer K down to 1.  Tbar None = full."""
        cur = 0
        for k in range(self.K - 1, -1, -1):
            gy = self.gy[cur]
            Da, Du, Dc, E = self.D
            dz = self.dz if k > 0 else None
            gx = self.gy_x[cur]
            if Tbar is None:
                lib.bwd_full(self.dims, self.w[k], self.a[k], self.c[k], self.h[k], gy, Da, Du, Dc, E,
                             self.ws, self.ws_bytes, stream, dz=dz, gy_x=gx)
            else:
                lib.bwd_trunc(self.dims, self.w[k], self.a[k], self.c[k], self.h[k], gy, Da, Du, Dc, E, Tbar,
                              self.ws, self.ws_bytes, stream, dz=dz, gy_x=gx)
            if on_layer is not None:
                on_layer(k, self)
            # k >= 1: gy^{k-1} = gy^k + J^T dxhat^k through the normalised input, in the
            # input-gradient GEMM's epilogue
            gp = self.gy[1 - cur] if k > 0 else None
            lib.param_grad(self.dims, self.w[k], self.x[k], Da, Du, Dc, E, gy, self.dW_in[k],
                           self.db_a[k], self.dW_o[k], gp, None, int(accumulate), self.ws, self.ws_bytes, stream,
                           r=self.r[k - 1] if k > 0 else None, dz=dz, gy_x=gx,
                           gy_prev_x=self.gy_x[1 - cur] if k > 0 else None)
            cur = 1 - cur

    def step(self, Tbar=None, stream=None):
        self.forward(stream)
        self.loss_grad(stream)
        self.backward(Tbar, stream)

    def capture(self, Tbar=None):
        """A CUDA graph of one step on these buffers (``replay()`` reruns it): the library
        calls enqueue only kernels and memsets on the current stream, so the whole step
        captures, and a replay skips the per-call host work and launch gaps."""
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self.step(Tbar)                 # one eager step first: lazy initialisation off the capture
        torch.cuda.current_stream(self.device).wait_stream(side)
        with torch.cuda.graph(g):
            self.step(Tbar)
        return g

    def status(self, stream=None) -> int:
        return lib.stream_status(self.ws, stream)

    # ------------------------------------------------------------------ results
    def grads_numpy(self, k):
        N = self.N
        dW_in = self.dW_in[k].double().cpu().numpy()
        return dict(W_a=dW_in[:, :N], W_B=dW_in[:, N:2 * N], W_c=dW_in[:, 2 * N:],
                    b_a=self.db_a[k].double().cpu().numpy(), W_o=self.dW_o[k].double().cpu().numpy())
