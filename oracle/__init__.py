"""Plain CPU float64 oracle for causal attention forward, backward (with the GProj
bf16 emulation) and backward-over-backward.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import or run anything in this
package.  The library's product path never does, and this package imports nothing
from the library: the two share no code.  Inputs come from ``workloads`` (seeded
random draws only, no attention arithmetic).

Parity status of each function: all are pinned by tests that do not re-use the
oracle's own formulas (brute force, finite differences, symbolic differentiation,
closed-form special cases and invariants); see ``tests/test_oracle_pins.py``.
"""
from .attention import (  # noqa: F401
    backward, backward_all, backward_bf16_dS, backward_cols, backward_rows, bf16_round, bob,
    bob_all, bob_bf16_dS, bob_bf16_dS_all, bob_col_pass, bob_cols, bob_row_pass, bob_rows, default_scale, forward, forward_all,
    forward_online, forward_rows, hidden, scores, Segments, SegmentsBatch, softmax_rows, Window,
)
