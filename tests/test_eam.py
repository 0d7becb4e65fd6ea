"""Expert activation tracking, PredictEAM and the expert cache ("MOE-INFINITY: Efficient
MoE Inference on Personal Machines with Sparsity-Aware Expert Cache", sec. 4.3, 4.5,
4.7 Algorithm 1, appendix B.1).

The oracle is pinned to closed forms derived by hand from the pages' definitions on a
2-layer, 3-expert example; the library's host implementation is then compared with the
oracle bit for bit (integer counts, exact sums, the same double operations), on that
example and on seeded synthetic request traces.  None of this needs a GPU, except the
last test, which builds a request EAM from the router kernel's per-expert counts.
"""

import math

import numpy as np
import pytest

from oracle import eam_oracle as eo

A = np.array([[1, 0, 0], [0, 2, 0]], dtype=np.int32)
B = np.array([[0, 1, 0], [0, 0, 3]], dtype=np.int32)
C = np.array([[0, 2, 0], [0, 0, 1]], dtype=np.int32)
CUR0 = np.array([[1, 0, 0], [0, 0, 0]], dtype=np.int32)  # layer 0 routed, layer 1 not yet
CUR1 = np.array([[1, 0, 0], [0, 1, 0]], dtype=np.int32)

# Hand-derived values (sec. 4.5 definitions):
#   d(CUR0, A) = 1 - 1/sqrt(5)                  (a.b = 1, |CUR0| = 1, |A| = sqrt 5)
#   d(CUR0, B) = 1                              (orthogonal)
#   PredictEAM(CUR0, layer 0, 1 match): A's rows normalised: [1,0,0] x 1, [0,1,0] x (1 - 1/2)
#   PredictEAM(CUR0, layer 0, 2 matches): A + B = [[1,1,0],[0,2,3]] -> [.5,.5,0] x 1, [0,.4,.6] x .5
#   PredictEAM(CUR1, layer 1, 1 match): A nearest (1 - 3/sqrt 10 < 1); [1,0,0] x (1 + 1/2), [0,1,0] x 1
PINS = [
    (CUR0, 0, 1, [[1.0, 0.0, 0.0], [0.0, 0.5, 0.0]]),
    (CUR0, 0, 2, [[0.5, 0.5, 0.0], [0.0, 0.2, 0.3]]),
    (CUR1, 1, 1, [[1.5, 0.0, 0.0], [0.0, 1.0, 0.0]]),
]


def _oracle_ab():
    o = eo.Eamc(2, 3, 2)
    o.insert(A)
    o.insert(B)
    return o


def test_oracle_cosine_distance_closed_forms():
    assert eo.cosine_distance(CUR0, A) == pytest.approx(1 - 1 / math.sqrt(5), abs=1e-15)
    assert eo.cosine_distance(CUR0, B) == 1.0
    assert eo.cosine_distance(CUR1, A) == pytest.approx(1 - 3 / math.sqrt(10), abs=1e-15)
    assert eo.cosine_distance(A, A) == pytest.approx(0.0, abs=1e-15)
    assert eo.cosine_distance(3 * A, A) == pytest.approx(0.0, abs=1e-15)  # scale-free
    assert eo.cosine_distance(np.zeros((2, 3), np.int32), A) == 1.0


@pytest.mark.parametrize("cur,layer,n,expected", PINS)
def test_oracle_predict_closed_forms(cur, layer, n, expected):
    np.testing.assert_allclose(eo.predict(_oracle_ab(), cur, layer, n), expected, rtol=0, atol=1e-15)


def test_oracle_predict_row_sums_are_the_proximity_factor():
    rng = np.random.default_rng(0)
    o = eo.Eamc(6, 8, 5)
    for _ in range(5):
        o.insert(rng.integers(0, 4, size=(6, 8)))
    for layer in range(6):
        p = eo.predict(o, rng.integers(0, 3, size=(6, 8)), layer, 3)
        for i in range(6):
            assert p[i].sum() == pytest.approx(1 - (i - layer) / 6, abs=1e-12)


def test_oracle_cache_and_replacement_closed_forms():
    # capacity 2 filled by (0,0), (1,2); request (1,1) at layer 1 with CUR1: priorities
    # (1.5 + 1e-3)/1.5 * 1 for (0,0) and (0 + 1e-3)/1 * 0.5 for (1,2): (1,2) goes
    o = _oracle_ab()
    c = eo.ExpertCache(2, 2, 3)
    assert c.lookup(o, CUR1, 0, 0, 1, 1e-3) == (False, None)
    assert c.lookup(o, CUR1, 1, 2, 1, 1e-3) == (False, None)
    assert c.lookup(o, CUR1, 1, 1, 1, 1e-3) == (False, (1, 2))
    assert c.lookup(o, CUR1, 0, 0, 1, 1e-3) == (True, None)
    assert c.items == [(0, 0), (1, 1)]
    # full EAMC {A, B}: C is nearest to B (1 - 5/sqrt 50 against 1), so B's slot is reused
    assert eo.cosine_distance(C, B) == pytest.approx(1 - 5 / math.sqrt(50), abs=1e-15)
    assert o.insert(C) == 1
    assert [e.tolist() for e in o.entries] == [A.tolist(), C.tolist()]


def test_oracle_cache_lru_free_of_prediction_when_eps_dominates():
    # an empty EAMC predicts nothing: every priority is eps * (1 - layer/L), so the
    # cached expert of the deepest layer goes first (ties: the earliest inserted)
    o = eo.Eamc(4, 2, 3)
    c = eo.ExpertCache(3, 4, 2)
    z = np.zeros((4, 2), np.int32)
    for key in [(0, 0), (3, 1), (3, 0)]:
        c.lookup(o, z, key[0], key[1], 1, 1e-4)
    assert c.lookup(o, z, 1, 1, 1, 1e-4) == (False, (3, 1))


# ---------------------------------------------------------------- library vs oracle

def test_library_matches_the_pins():
    import sparse_expert_swiglu_gb300 as ses
    e = ses.EAMC(2, 3, 2)
    assert e.insert(A) == 0 and e.insert(B) == 1 and len(e) == 2
    idx, dist = e.match(CUR0, 2)
    assert idx.tolist() == [0, 1]
    assert dist[0] == eo.cosine_distance(CUR0, A) and dist[1] == 1.0
    for cur, layer, n, expected in PINS:
        got = e.predict(cur, layer, n)
        assert np.array_equal(got, eo.predict(_oracle_ab(), cur, layer, n))
        np.testing.assert_allclose(got, expected, rtol=0, atol=1e-15)
    c = ses.ExpertCache(2, 2, 3)
    assert c.lookup(e, CUR1, 0, 0, 1, 1e-3) == (False, None)
    assert c.lookup(e, CUR1, 1, 2, 1, 1e-3) == (False, None)
    assert c.lookup(e, CUR1, 1, 1, 1, 1e-3) == (False, (1, 2))
    assert c.lookup(e, CUR1, 0, 0, 1, 1e-3) == (True, None)
    assert c.contents() == [(0, 0), (1, 1)]
    assert e.insert(C) == 1
    assert e.entry(0).tolist() == A.tolist() and e.entry(1).tolist() == C.tolist()


def _requests(rng, n_req, L, E, iters):
    """Synthetic decode traces: every request prefers a few experts per layer (the
    skew within a request that the pages describe), drawn from one of a few groups."""
    groups = [rng.dirichlet(np.full(E, 0.3), size=L) for _ in range(4)]
    out = []
    for _ in range(n_req):
        pref = groups[rng.integers(len(groups))]
        it = []
        for _ in range(iters):
            ieam = np.zeros((L, E), np.int32)
            for i in range(L):
                for j in rng.choice(E, size=2, replace=False, p=pref[i]):
                    ieam[i, j] += 1
            it.append(ieam)
        out.append(it)
    return out


@pytest.mark.parametrize("L,E,cap,n_match", [(8, 8, 6, 1), (32, 8, 20, 3), (4, 64, 5, 2)])
def test_library_matches_oracle_on_traces(L, E, cap, n_match):
    import sparse_expert_swiglu_gb300 as ses
    rng = np.random.default_rng(L * 1000 + E)
    reqs = _requests(rng, 3 * cap, L, E, 6)
    lib_c, orc_c = ses.EAMC(L, E, cap), eo.Eamc(L, E, cap)
    lib_k, orc_k = ses.ExpertCache(L * 2, L, E), eo.ExpertCache(L * 2, L, E)
    n_evict = 0
    for r in reqs:
        ream_l = np.zeros((L, E), np.int32)
        ream_o = np.zeros((L, E), np.int32)
        for ieam in r:
            for i in range(L):
                ses.eam_add_counts(ream_l, i, ieam[i])
                eo.add_counts(ream_o, i, ieam[i])
                # the layer's experts requested from the cache as the layer runs
                for j in np.nonzero(ieam[i])[0]:
                    got = lib_k.lookup(lib_c, ream_l, i, int(j), n_match, 1e-4)
                    want = orc_k.lookup(orc_c, ream_o, i, int(j), n_match, 1e-4)
                    assert got == want
                    n_evict += got[1] is not None
            assert np.array_equal(ream_l, ream_o)
        if len(orc_c.entries) == cap:
            idx, dist = lib_c.match(ream_l, n_match)
            oi, od = eo.nearest(orc_c.entries, ream_o, n_match)
            assert idx.tolist() == oi and dist.tolist() == od
            for layer in (0, L // 2, L - 1):
                assert np.array_equal(lib_c.predict(ream_l, layer, n_match),
                                      eo.predict(orc_c, ream_o, layer, n_match))
        assert lib_c.insert(ream_l) == orc_c.insert(ream_o)
    assert lib_k.contents() == orc_k.items
    for i in range(cap):
        assert lib_c.entry(i).tolist() == orc_c.entries[i].tolist()
    assert n_evict > 0


def test_library_argument_checks():
    import sparse_expert_swiglu_gb300 as ses
    lib = ses.lib()
    assert lib.moe_eamc_bytes(0, 8, 4) == 0 and lib.moe_expert_cache_bytes(0) == 0
    e = ses.EAMC(2, 3, 2)
    with pytest.raises(ses.MoeError):
        e.predict(CUR0, 2, 1)  # layer out of range
    with pytest.raises(ses.MoeError):
        e.entry(0)  # empty
    with pytest.raises(ValueError):
        e.insert(np.zeros((3, 3), np.int32))
    c = ses.ExpertCache(2, 2, 3)
    with pytest.raises(ses.MoeError):
        c.lookup(ses.EAMC(3, 3, 2), CUR0, 0, 0)  # EAMC of another shape
    with pytest.raises(ses.MoeError):
        c.lookup(e, CUR0, 0, 3)  # expert out of range
    assert lib.moe_eamc_size(None) < 0


@pytest.mark.gpu
def test_request_eam_from_router_counts():
    """A request EAM built from the router kernel's per-expert counts (one row per MoE
    layer and iteration) equals the counts of the oracle's top-k choices."""
    import torch
    import sparse_expert_swiglu_gb300 as ses
    from oracle import moe_oracle as orc
    from sparse_expert_swiglu_gb300 import synth
    L, E, k, d, B = 4, 8, 2, 1024, 6
    routers = [synth.router(d, E, 500, layer=i).cuda() for i in range(L)]
    ream = np.zeros((L, E), np.int32)
    ref = np.zeros((L, E), np.int32)
    for it in range(3):
        x = synth.tokens(B, d, 600 + it).cuda()
        for i in range(L):
            _, _, counts = ses.route_topk(x, routers[i], k, renorm=True)
            ses.eam_add_counts(ream, i, counts.cpu().numpy())
            idx, _, _ = orc.route_topk(x.cpu().numpy(), routers[i].cpu().numpy(), k, True)
            eo.add_counts(ref, i, np.bincount(idx.ravel(), minlength=E))
    assert np.array_equal(ream, ref)
    assert ream.sum() == 3 * L * B * k
    torch.cuda.synchronize()


def test_library_matches_oracle_on_random_shapes():
    """Random shapes, capacities, match counts and request sequences (hypothesis):
    the library's slots, matches, predictions and cache decisions equal the oracle's."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")
    import sparse_expert_swiglu_gb300 as ses

    @hyp.settings(max_examples=40, deadline=None)
    @hyp.given(L=st.integers(1, 6), E=st.integers(1, 9), cap=st.integers(1, 5),
               n_match=st.integers(1, 4), seed=st.integers(0, 2 ** 31 - 1))
    def run(L, E, cap, n_match, seed):
        rng = np.random.default_rng(seed)
        lib_c, orc_c = ses.EAMC(L, E, cap), eo.Eamc(L, E, cap)
        lib_k, orc_k = ses.ExpertCache(max(1, L), L, E), eo.ExpertCache(max(1, L), L, E)
        for _ in range(2 * cap + 2):
            m = rng.integers(0, 4, size=(L, E)).astype(np.int32)
            layer = int(rng.integers(L))
            assert np.array_equal(lib_c.predict(m, layer, n_match), eo.predict(orc_c, m, layer, n_match))
            idx, dist = lib_c.match(m, n_match)
            oi, od = eo.nearest(orc_c.entries, m, n_match)
            assert idx.tolist() == oi and dist.tolist() == od
            for _ in range(3):
                e = int(rng.integers(E))
                assert lib_k.lookup(lib_c, m, layer, e, n_match, 1e-4) == \
                    orc_k.lookup(orc_c, m, layer, e, n_match, 1e-4)
            assert lib_c.insert(m) == orc_c.insert(m)
        assert lib_k.contents() == orc_k.items

    run()
