"""CPU fp64 oracle for the adjoint-sharding gradient path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
import this package.  It shares no code with the CUDA library or its binding.
"""
from .oracle import (  # noqa: F401
    AGGREGATED, EPS, LITERAL, build, normalize, normalize_vjp, layer_forward, layer_grad, loss_and_cotangent,
    stack_forward, stack_grad, threads, use_library,
)
