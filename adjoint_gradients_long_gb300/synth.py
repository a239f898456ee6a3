"""Seeded synthetic inputs for the diagonal selective SSM adjoint-gradient workloads.

This module only draws random numbers and rounds them to the storage type a
consumer reads; it holds none of the method's arithmetic.  Both the CPU oracle
(through the tests) and the CUDA path (through the tests and the benchmark) are
fed from here, so the two always see bit-identical values.

Workloads (sizes, distributions and windows follow the problem statement of
"Adjoint sharding for very long context training of state space models",
Section 3.1 model form; the initialisation is the one the workload list fixes):

  ssm1_p16   1 layer, P=16,  N=8,   T=256,     B=1, fp32, full window
  ssm1_p128  1 layer, P=128, N=256, T=16384,   B=4, fp32, full and Tbar=2048
  ssm8_p512  8 layers, P=512, N=256, T=65536,  B=1, bf16 GEMM operands, Tbar=4096
  ssm1_1m    1 layer, P=256, N=256, T=2^20,    B=1, bf16 GEMM operands, b_a=4,
             Tbar=4096 and full
  ssm4_p2048 4 layers, P=2048, N=256, T=131072, B=1, bf16 GEMM operands, Tbar=8192

General selective layer (one layer; per channel p the step dt = softplus(z_p), the
decay exp(dt A_pn), input-dependent B_t, C_t):

  sel1_p16   P=16,   N=8,  T=256,   B=1, fp32,                 full and Tbar=64
  sel1_p64   P=64,   N=16, T=2048,  B=2, fp32,                 full and Tbar=256
  sel1_p1024 P=1024, N=16, T=65536, B=1, bf16 GEMM operands,   Tbar=8192 and full

Every tensor is drawn in token chunks of CHUNK tokens from its own counter-keyed
PCG64 stream (seed, tensor id, batch row, chunk index), so any token range of a
workload can be regenerated on its own and equals the same slice of the whole.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

CHUNK = 4096

# tensor stream ids
_S_XHAT, _S_TARGET = 1, 2
_S_WA, _S_WB, _S_WC, _S_WO = 11, 12, 13, 14
_S_WDT, _S_BDT, _S_A = 21, 22, 23


@dataclasses.dataclass(frozen=True)
class Workload:
    key: str
    index: int          # 1-based position in the workload list
    K: int              # residual layers
    P: int              # model width
    N: int              # state size
    T: int              # tokens per sequence
    B: int              # sequences
    x_dtype: str        # "f32" or "bf16": GEMM operand storage (xhat, W_in, W_o, D, E)
    windows: tuple      # truncation windows to evaluate; None = full adjoint
    wa_var: float       # W_a ~ N(0, wa_var / P)
    b_a: float          # gate bias, a ~ sigmoid(b_a)

    @property
    def seed(self) -> int:
        return 1000 + self.index


WORKLOADS = {
    "ssm1_p16": Workload("ssm1_p16", 1, 1, 16, 8, 256, 1, "f32", (None,), 0.01, 3.0),
    "ssm1_p128": Workload("ssm1_p128", 2, 1, 128, 256, 16384, 4, "f32", (None, 2048), 0.01, 3.0),
    "ssm8_p512": Workload("ssm8_p512", 3, 8, 512, 256, 65536, 1, "bf16", (4096,), 0.01, 3.0),
    "ssm1_1m": Workload("ssm1_1m", 4, 1, 256, 256, 1 << 20, 1, "bf16", (4096, None), 0.01, 4.0),
    "ssm4_p2048": Workload("ssm4_p2048", 5, 4, 2048, 256, 131072, 1, "bf16", (8192,), 1.0, 3.0),
}


def workload(key_or_index) -> Workload:
    if isinstance(key_or_index, int):
        for w in WORKLOADS.values():
            if w.index == key_or_index:
                return w
        raise KeyError(key_or_index)
    return WORKLOADS[key_or_index]


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + (((u >> 16) & 1) + np.uint32(0x7FFF))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-representable."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    if np.any(u & np.uint32(0xFFFF)):
        raise ValueError("values are not bf16-representable; call round_bf16 first")
    return (u >> 16).astype(np.uint16)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def _tokens(seed: int, stream: int, B: int, t0: int, t1: int, width: int) -> np.ndarray:
    out = np.empty((B, t1 - t0, width), np.float32)
    for b in range(B):
        c0, c1 = t0 // CHUNK, (t1 + CHUNK - 1) // CHUNK
        for c in range(c0, c1):
            blk = _rng(seed, stream, b, c).standard_normal((CHUNK, width), dtype=np.float32)
            lo, hi = max(t0, c * CHUNK), min(t1, (c + 1) * CHUNK)
            out[b, lo - t0:hi - t0] = blk[lo - c * CHUNK:hi - c * CHUNK]
    return out


def make_layer_weights(w: Workload, k: int, P: Optional[int] = None, N: Optional[int] = None,
                       seed: Optional[int] = None) -> dict:
    """Weights of layer k (0-based): W_a, W_B, W_c [P,N], b_a [N], W_o [N,P], float32."""
    P = w.P if P is None else P
    N = w.N if N is None else N
    seed = w.seed if seed is None else seed
    sd = np.float32(1.0 / np.sqrt(P))
    W_a = _rng(seed, _S_WA, k).standard_normal((P, N), dtype=np.float32) * np.float32(np.sqrt(w.wa_var / P))
    W_B = _rng(seed, _S_WB, k).standard_normal((P, N), dtype=np.float32) * sd
    W_c = _rng(seed, _S_WC, k).standard_normal((P, N), dtype=np.float32) * sd
    W_o = _rng(seed, _S_WO, k).standard_normal((N, P), dtype=np.float32) * sd
    b_a = np.full((N,), w.b_a, np.float32)
    if w.x_dtype == "bf16":
        W_a, W_B, W_c, W_o = (round_bf16(m) for m in (W_a, W_B, W_c, W_o))
    return dict(W_a=W_a, W_B=W_B, W_c=W_c, b_a=b_a, W_o=W_o)


def make_inputs(w, T: Optional[int] = None, B: Optional[int] = None, P: Optional[int] = None,
                N: Optional[int] = None, K: Optional[int] = None, t0: int = 0,
                seed: Optional[int] = None) -> dict:
    """Inputs of a workload, optionally resized (T, B, P, N, K) or restricted to tokens [t0, t0+T).

    Returns dict(xhat [B,T,P], target [B,T,P], layers=[weights per layer]) in float32; for
    bf16 workloads xhat and the weight matrices hold bf16-representable values.
    """
    if not isinstance(w, Workload):
        w = workload(w)
    T = w.T if T is None else T
    B = w.B if B is None else B
    P = w.P if P is None else P
    N = w.N if N is None else N
    K = w.K if K is None else K
    seed = w.seed if seed is None else seed
    xhat = _tokens(seed, _S_XHAT, B, t0, t0 + T, P)
    target = _tokens(seed, _S_TARGET, B, t0, t0 + T, P)
    if w.x_dtype == "bf16":
        xhat = round_bf16(xhat)
    layers = [make_layer_weights(w, k, P, N, seed) for k in range(K)]
    return dict(xhat=xhat, target=target, layers=layers, workload=w, T=T, B=B, P=P, N=N, K=K)


@dataclasses.dataclass(frozen=True)
class SelWorkload:
    """A workload of the general selective layer (one layer)."""
    key: str
    P: int              # channels
    N: int              # states per channel
    T: int              # tokens per sequence
    B: int              # sequences
    x_dtype: str        # "f32" or "bf16": GEMM operand storage (xhat, W_in, dz)
    windows: tuple      # truncation windows; None = full adjoint
    seed: int


SEL_WORKLOADS = {
    "sel1_p16": SelWorkload("sel1_p16", 16, 8, 256, 1, "f32", (None, 64), 2001),
    "sel1_p64": SelWorkload("sel1_p64", 64, 16, 2048, 2, "f32", (None, 256), 2002),
    "sel1_p1024": SelWorkload("sel1_p1024", 1024, 16, 65536, 1, "bf16", (8192, None), 2003),
}


def make_sel_inputs(w, T: Optional[int] = None, B: Optional[int] = None, P: Optional[int] = None,
                    N: Optional[int] = None, t0: int = 0, seed: Optional[int] = None) -> dict:
    """Inputs of a selective-layer workload, optionally resized or restricted to tokens
    [t0, t0+T).  float32 arrays: xhat, target [B,T,P] ~ N(0,1); W_in [P, P+2N] = [W_dt ~
    N(0, 0.25/P) | W_B ~ N(0, 1/P) | W_C ~ N(0, 1/P)]; b_dt [P] ~ U[-7, -2.3] (so the step
    softplus(b_dt) spans about 1e-3 .. 1e-1); A [P,N] = -(n+1) U[0.8, 1.2].  bf16 workloads
    hold bf16-representable xhat and W_in."""
    if not isinstance(w, SelWorkload):
        w = SEL_WORKLOADS[w]
    T = w.T if T is None else T
    B = w.B if B is None else B
    P = w.P if P is None else P
    N = w.N if N is None else N
    seed = w.seed if seed is None else seed
    xhat = _tokens(seed, _S_XHAT, B, t0, t0 + T, P)
    target = _tokens(seed, _S_TARGET, B, t0, t0 + T, P)
    if w.x_dtype == "bf16":
        xhat = round_bf16(xhat)
    return dict(xhat=xhat, target=target, **_sel_weights(seed, P, N, w.x_dtype), workload=w, T=T, B=B, P=P, N=N)


def _sel_weights(seed: int, P: int, N: int, x_dtype: str) -> dict:
    W_dt = _rng(seed, _S_WDT).standard_normal((P, P), dtype=np.float32) * np.float32(0.5 / np.sqrt(P))
    W_B = _rng(seed, _S_WB).standard_normal((P, N), dtype=np.float32) * np.float32(1.0 / np.sqrt(P))
    W_C = _rng(seed, _S_WC).standard_normal((P, N), dtype=np.float32) * np.float32(1.0 / np.sqrt(P))
    W_in = np.ascontiguousarray(np.concatenate([W_dt, W_B, W_C], axis=1))
    b_dt = _rng(seed, _S_BDT).uniform(-7.0, -2.3, size=P).astype(np.float32)
    A = (-(np.arange(N, dtype=np.float32) + 1.0)[None, :]
         * _rng(seed, _S_A).uniform(0.8, 1.2, size=(P, N)).astype(np.float32)).astype(np.float32)
    if x_dtype == "bf16":
        W_in = round_bf16(W_in)
    return dict(W_in=W_in, b_dt=b_dt, A=A)


def make_sel_stack_inputs(w, K: int, T: Optional[int] = None, B: Optional[int] = None, P: Optional[int] = None,
                          N: Optional[int] = None, t0: int = 0, seed: Optional[int] = None) -> dict:
    """A residual stack of K selective layers: the input, target and layer 1's weights of
    make_sel_inputs, and layer k's (k >= 2) weights drawn the same way from the seed
    seed + 1000 (k - 1).  layers: a list of K dicts W_in, b_dt, A."""
    d = make_sel_inputs(w, T, B, P, N, t0, seed)
    s0 = d["workload"].seed if seed is None else seed
    layers = [dict(W_in=d["W_in"], b_dt=d["b_dt"], A=d["A"])]
    for k in range(1, K):
        layers.append(_sel_weights(s0 + 1000 * k, d["P"], d["N"], d["workload"].x_dtype))
    d["layers"] = layers
    d["K"] = K
    return d
