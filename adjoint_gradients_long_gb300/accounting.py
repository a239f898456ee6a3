"""Storage and traffic accounting for the adjoint-sharding path (host-side arithmetic only).

``paper_state_values`` is the stored-state count of the review page "Adjoint
sharding for very long context training of state space models" (Referee Report,
major comment on Section 4.5): storing {A_t, C_t, h_t, y_t} for T tokens and K
layers costs T K (2N + P) + T P values.  ``stored_bytes`` is what this library
actually keeps per layer: a, c, h in fp32 plus the layer input xhat.  For comparison
(the page's central claim is a memory saving over backpropagation, Referee Report major
comment 3), ``bptt_saved_bytes`` counts what reverse-mode differentiation of the same
stack must save, and ``checkpoint_saved_bytes`` the peak with activation checkpointing.
"""
from __future__ import annotations


def paper_state_values(T: int, K: int, N: int, P: int) -> int:
    """Section 4.5 stored-value count T K (2N + P) + T P."""
    return T * K * (2 * N + P) + T * P


def stored_bytes(B: int, T: int, K: int, N: int, P: int, x_bytes: int) -> int:
    """Bytes this library keeps between the forward and the backward pass: per layer and
    token, a, c, h (3N fp32) and the layer input xhat (P values of x_bytes each)."""
    return B * T * K * (3 * N * 4 + P * x_bytes)


def bptt_saved_bytes(B: int, T: int, K: int, N: int, P: int, x_bytes: int) -> int:
    """Bytes reverse-mode differentiation of the same stack keeps from the forward pass when
    every operation saves only what its own derivative reads, per layer and token:
    the layer input xhat (the three input projections' weight gradients, P values of
    x_bytes), the gate a (the sigmoid's derivative and the recurrence's dh_{t-1}), the state
    h (h_{t-1} for the recurrence's da_t, h_t for the product c . h), c (the product), and the
    product c . h (the output projection's weight gradient): 4N fp32 values."""
    return B * T * K * (4 * N * 4 + P * x_bytes)


def checkpoint_saved_bytes(B: int, T: int, K: int, N: int, P: int, x_bytes: int, segment: int = 0) -> int:
    """Peak bytes kept by reverse-mode differentiation with activation checkpointing (the
    input of every segment-th layer is kept; a segment's activations are recomputed during
    the backward pass and held only while it is differentiated): the kept fp32 residual
    streams (P values a token each) plus one segment's saved bytes.  segment defaults to the
    integer nearest sqrt(K)."""
    s = segment if segment > 0 else max(1, int(round(K ** 0.5)))
    kept = -(-K // s) * B * T * P * 4
    return kept + bptt_saved_bytes(B, T, min(s, K), N, P, x_bytes)


def step_bytes(P: int, N: int, x_bytes: int, d_bytes: int, window: bool, stacked: bool) -> dict:
    """Algorithmic HBM bytes per token per layer of each call of the library as built
    (inputs read once, outputs written once, workspace round trips included)."""
    fwd = {
        "proj_in": P * x_bytes + 3 * N * 4,           # read xhat; write a, c, u
        "fwd_scan": 2 * N * 4 + N * 4,                # read a, u; write h
        "proj_out": 2 * N * 4 + P * x_bytes + P * 4 + (P * 2 if x_bytes == 2 else 0),
    }
    bwd = {
        "cot_proj": P * 4 + N * 4,                    # read gy; write g
        "bwd_scan": 4 * N * 4 + 4 * N * d_bytes,      # read g, c, a, h; write D_a, D_u, D_c, E
    }
    if window:
        bwd["win_scan"] = 3 * N * 4 + N * 4           # read g, c, a; write R
        bwd["bwd_scan"] += N * 4                      # read R
    par = {
        "param_grad": P * x_bytes + 3 * N * d_bytes + N * d_bytes + P * 4,
        "colsum": N * d_bytes,
    }
    if stacked:
        par["input_grad"] = 3 * N * d_bytes + P * 4 + P * 4
    return {"fwd": fwd, "bwd": bwd, "param": par}


def stack_buffer_bytes(B: int, T: int, K: int, N: int, P: int, x_bytes: int, d_bytes: int) -> dict:
    """Device bytes of every buffer the stack driver (stack.AdjStack) allocates, by group,
    workspace excluded: what one gradient step of the library needs besides its scratch.
      states    a, c, h per layer (fp32) and the layer inputs xhat (x_bytes), r per stacked layer
      streams   the fp32 residual stream y per layer, the target, two cotangent buffers gy
                (and, with bf16 GEMM operands, their two bf16 copies)
      seeds     D_a, D_u, D_c, E (d_bytes) and the row dots dz of a normalised input
      params    W_in, b_a, W_o per layer (x_bytes; b_a fp32) and their fp32 gradients
      loss      one fp64 value"""
    bt = B * T
    states = K * bt * (3 * N * 4 + P * x_bytes) + (K - 1) * bt * 4
    streams = K * bt * P * 4 + bt * P * 4 + 2 * bt * P * 4 + (2 * bt * P * 2 if x_bytes == 2 else 0)
    seeds = 4 * bt * N * d_bytes + (bt * ((N + 127) // 128) * 4 if K > 1 else 0)
    params = K * (P * 3 * N * x_bytes + N * 4 + N * P * x_bytes) + K * (P * 3 * N + N + N * P) * 4
    # allocations: x, a, c, h, y per layer; r per stacked layer; target, two gy, loss; four
    # seeds; dz; W_in, b_a, W_o and their gradients per layer
    count = 5 * K + (K - 1) + 4 + 4 + (1 if K > 1 else 0) + 6 * K + (2 if x_bytes == 2 else 0)
    return {"states": states, "streams": streams, "seeds": seeds, "params": params, "loss": 8, "buffers": count}
