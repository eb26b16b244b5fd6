"""Float64 CPU oracle for the fused attention-KL divergence.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may call it.  It shares no code with the CUDA library.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` against closed forms, invariants, brute force on
tiny inputs, finite differences and independent library routines.  No
function is "parity unpinned".
"""

from .streamkl_oracle import (  # noqa: F401
    visible_mask,
    forward,
    forward_head,
    forward_rows,
    forward_online,
    forward_two_pass,
    backward,
    backward_head,
    backward_dq_rows,
    backward_dk_keys,
    loss,
    MODE_P2,
    MODE_P1,
)
