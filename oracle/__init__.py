"""CPU oracle for fused scaled-dot-product attention (forward and backward).

TEST INFRASTRUCTURE, NOT PART OF THE LIBRARY. Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import anything here. The CUDA library shares no
code, header, table or helper with this package, and neither imports the
other; the only thing both sides consume is the seeded input generator in
``scaled_dot_product_07_gb300.workloads``, which holds none of the method's
arithmetic.

Everything is float64 numpy on the host, one (batch, head) at a time, with
the full score matrix materialised.

Pins (tests that tie the oracle to something other than itself) live in
``tests/test_oracle.py``; every function here is pinned there.
"""

from .philox import keep_mask, keep_mask_head, keep_threshold, philox4x32_10, uniform_words
from .sdpa import default_scale, head_backward, head_forward, sdpa_bwd, sdpa_fwd

__all__ = [
    "philox4x32_10", "keep_threshold", "uniform_words", "keep_mask_head", "keep_mask",
    "default_scale", "head_forward", "head_backward", "sdpa_fwd", "sdpa_bwd",
]
