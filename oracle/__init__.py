"""fp64 CPU oracle for the attention backward pass (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The CUDA path never does.
"""
from .attn_oracle import (allowed_mask, delta_from_output, head_backward, head_forward,
                          mha_backward, mha_forward)

__all__ = ["allowed_mask", "delta_from_output", "head_backward", "head_forward",
           "mha_backward", "mha_forward"]
