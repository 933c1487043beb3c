"""CPU oracle for the fa_fwd attention forward pass and its backward pass.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its cpu_baseline leg and its
``--impl reference`` arm) may import this package. The CUDA path in
``flashattention_fa_fwd_gb300`` never imports it, and it imports nothing from
that package: the two share no code.

Modules
-------
attention
    The plain definition of attention, materialised in float64 with numpy
    (``attention``, ``attention_rows``). This is what every parity test
    compares the CUDA kernels against.
backward
    The gradients dQ, dK, dV of that definition for an output gradient dO,
    with P rebuilt from the forward's log-sum-exp (``attention_bwd``).
online
    A step-by-step model of the streaming (online) softmax recurrence in the
    pages' notation (m, l, acc, alpha), with switches that plant the mistakes
    the pages warn about. Tests use it to show that the parity checks catch
    those mistakes; it is never used as a parity reference.

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
the pages print, closed forms, invariants and pure-Python brute force.
"""

from .attention import attention, attention_rows, flop_count  # noqa: F401
from .backward import attention_bwd, bwd_flop_count  # noqa: F401
from .online import online_attention_row, online_softmax_trace  # noqa: F401
