"""fp64 CPU oracle for fused linear cross-entropy.

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import or run it. It shares no code with the CUDA path.

* :mod:`oracle.flce_oracle` -- the streaming fp64 definition (forward,
  backward, sampled rows).
* :mod:`oracle.brute` -- pure-Python brute force on tiny inputs: materialised
  logits, explicit softmax, forward quantities only.
"""
from . import flce_oracle  # noqa: F401
from .flce_oracle import backward, final_logits, forward, row_weights  # noqa: F401
