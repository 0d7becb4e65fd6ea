"""moe_route_topk_noalloc (static scratch, no workspace) against moe_route_topk,
through the C ABI (marked gpu).  The file name sorts last so that it also runs
after every other test has used the device.

Both entry points launch the same router kernel on the same inputs, so the
expert indices and counts must be equal and the weights equal within 2e-6 (the
router test tolerance).  Consecutive calls share the static scratch: the cases
below run back to back, from one token (one CTA) to the multi-CTA hand-off of two
or more tokens (one CTA per token, the last one to finish found with the scratch's
counter, which must start at zero), up to the stated maximum of B * k pairs.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ses = pytest.importorskip("sparse_expert_swiglu_gb300")
from sparse_expert_swiglu_gb300 import synth  # noqa: E402
from sparse_expert_swiglu_gb300._lib import MoeError, ROUTE_NOALLOC_MAX_PAIRS  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ses.build_library()
    ses.lib()


def _same(a, b):
    idx_a, w_a, cnt_a = (t.cpu().numpy() for t in a)
    idx_b, w_b, cnt_b = (t.cpu().numpy() for t in b)
    assert np.array_equal(idx_a, idx_b)
    assert np.array_equal(cnt_a, cnt_b)
    np.testing.assert_allclose(w_a, w_b, rtol=0, atol=2e-6)


CASES = [(1, 4096, 8, 2, True), (64, 4096, 8, 2, True), (1024, 2048, 64, 2, False),
         (3, 256, 256, 8, True)]


def test_noalloc_matches_workspace_router_twice_in_a_row():
    for rep in range(2):
        for i, (B, d, E, k, renorm) in enumerate(CASES):
            assert B * k <= ROUTE_NOALLOC_MAX_PAIRS
            x = synth.tokens(B, d, 40 + 10 * rep + i).cuda()
            wr = synth.router(d, E, 40 + 10 * rep + i).cuda()
            got = ses.route_topk_noalloc(x, wr, k, renorm)
            ref = ses.route_topk(x, wr, k, renorm)
            torch.cuda.synchronize()
            _same(got, ref)


def test_noalloc_rejects_more_pairs_than_its_scratch():
    B, d, E, k = 1024, 256, 8, 4  # 4096 pairs > 2048
    x = synth.tokens(B, d, 3).cuda()
    wr = synth.router(d, E, 3).cuda()
    with pytest.raises(MoeError) as err:
        ses.route_topk_noalloc(x, wr, k, True)
    assert err.value.status == -4
    # the scratch is still usable afterwards
    x1, wr1 = x[:8].contiguous(), wr
    _same(ses.route_topk_noalloc(x1, wr1, 2, True), ses.route_topk(x1, wr1, 2, True))
