"""CPU oracle for the decode-time sparse-SwiGLU MoE layer (``moe_oracle``) and for the
expert activation tracking and expert cache (``eam_oracle``).

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, fp64 restatement of what
the method computes, written to be checked by eye against the pages it cites.  It
shares no code with the CUDA library and imports nothing from it.  Only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import it; the product path never does.

Parity pins: every function here is pinned by CPU tests (hand-worked closed-form
fixtures under ``tests/golden/``, closed forms worked by hand in ``tests/test_eam.py``,
library routines for special cases, brute force on tiny inputs and invariants).  No
function is "parity unpinned".
"""

from .moe_oracle import (  # noqa: F401
    GROUP,
    quantize_int2,
    dequantize_int2,
    route_topk,
    expert_up,
    sparse_swiglu_expert,
    quantile_threshold,
    rmsnorm,
    moe_layer,
    silu,
)
