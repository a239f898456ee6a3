"""Stack driver: sequences the libadj.so calls for a residual stack of diagonal
selective SSM layers on one GPU.  PyTorch provides device memory and the stream;
every arithmetic step runs in the library's kernels.

Order of one gradient step ([AS] = review page "Adjoint sharding for very long
context training of state space models"; [AS] Referee Report on Algorithm 1 for
the stored states, Core claim for Propositions 2 and 3):
  for k = 1..K: adj_fwd_scan(k)            stores a^k, c^k, h^k; y^k = xhat^{k+1}
  adj_loss_mse                             gy^K = y^K - target, L
  for k = K..1: adj_bwd_{full,trunc}(k)    VJP seeds D_a, D_u, D_c, E of layer k
                adj_param_grad(k)          dW_in^k, db_a^k, dW_o^k and gy^{k-1}
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
        self.x = [z(B, T, P, dtype=xt)]                       # GEMM operand of layer k
        self.a = [z(B, T, N) for _ in range(K)]
        self.c = [z(B, T, N) for _ in range(K)]
        self.h = [z(B, T, N) for _ in range(K)]
        self.y = [z(B, T, P) for _ in range(K)]                # fp32 residual stream y^k
        for _ in range(K - 1):
            self.x.append(z(B, T, P, dtype=xt) if x_bf16 else None)
        self.target = z(B, T, P)
        self.D = [z(B, T, N, dtype=dt) for _ in range(4)]     # D_a, D_u, D_c, E
        self.gy = [z(B, T, P), z(B, T, P)]
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
        return self.x[k] if (k == 0 or self.x_bf16) else self.y[k - 1]

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
            y_x = self.x[k + 1] if (self.x_bf16 and k + 1 < self.K) else None
            xres = self.y[k - 1] if k > 0 else None
            lib.fwd_scan(self.dims, self.w[k], self.layer_input(k), xres, self.a[k], self.c[k], self.h[k],
                         self.y[k], y_x, self.ws, self.ws_bytes, stream)

    def loss_grad(self, stream=None):
        lib.loss_mse(self.dims, self.y[-1], self.target, self.gy[0], self.loss, self.ws, self.ws_bytes, stream)

    def backward(self, Tbar=None, stream=None, accumulate=False, on_layer=None):
        """Adjoint pass and parameter gradients, layer K down to 1.  Tbar None = full."""
        cur = 0
        for k in range(self.K - 1, -1, -1):
            gy = self.gy[cur]
            Da, Du, Dc, E = self.D
            if Tbar is None:
                lib.bwd_full(self.dims, self.w[k], self.a[k], self.c[k], self.h[k], gy, Da, Du, Dc, E,
                             self.ws, self.ws_bytes, stream)
            else:
                lib.bwd_trunc(self.dims, self.w[k], self.a[k], self.c[k], self.h[k], gy, Da, Du, Dc, E, Tbar,
                              self.ws, self.ws_bytes, stream)
            if on_layer is not None:
                on_layer(k, self)
            gy_prev = self.gy[1 - cur] if k > 0 else None
            lib.param_grad(self.dims, self.w[k], self.layer_input(k), Da, Du, Dc, E, gy, self.dW_in[k],
                           self.db_a[k], self.dW_o[k], gy_prev, int(accumulate), self.ws, self.ws_bytes, stream)
            cur = 1 - cur

    def step(self, Tbar=None, stream=None):
        self.forward(stream)
        self.loss_grad(stream)
        self.backward(Tbar, stream)

    def status(self, stream=None) -> int:
        return lib.stream_status(self.ws, stream)

    # ------------------------------------------------------------------ results
    def grads_numpy(self, k):
        N = self.N
        dW_in = self.dW_in[k].double().cpu().numpy()
        return dict(W_a=dW_in[:, :N], W_B=dW_in[:, N:2 * N], W_c=dW_in[:, 2 * N:],
                    b_a=self.db_a[k].double().cpu().numpy(), W_o=self.dW_o[k].double().cpu().numpy())
