"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each oracle function is checked against at least one of: a hand-worked closed-form
fixture under tests/golden/ (with its citation), a library routine that a special
case reduces to, brute force on tiny inputs, or an invariant of the method.  The
mutation tests at the end plant plausible mistakes in the oracle and check that a
pin catches each of them.
"""

import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from tests.conftest import load_golden

F16 = np.float16


def _h(a):
    return np.asarray(a, dtype=np.float64).astype(F16)


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def test_route_golden():
    g = load_golden("route_topk.json")
    for case in g["cases"]:
        idx, w, logits = orc.route_topk(_h(g["x"]), _h(g["w_router"]), case["k"], bool(case["renorm"]))
        assert idx.tolist() == case["idx"]
        if case["w"] is not None:
            for row, exp in enumerate(case["w"]):
                if exp is not None:
                    np.testing.assert_allclose(w[row], exp, rtol=0, atol=1e-15)


def _topk_by_rank_count(logits, k):
    """Brute force: expert e is in the top-k iff fewer than k experts beat it,
    where e' beats e if its logit is larger or equal with a lower index."""
    E = logits.size
    chosen = []
    for e in range(E):
        beaten_by = sum(1 for o in range(E) if logits[o] > logits[e] or (logits[o] == logits[e] and o < e))
        if beaten_by < k:
            chosen.append((beaten_by, e))
    return [e for _, e in sorted(chosen)]


@pytest.mark.parametrize("E,k", [(4, 1), (8, 2), (16, 6), (64, 6)])
def test_route_bruteforce(E, k):
    rng = np.random.default_rng(E * 10 + k)
    B, d = 6, 32
    # small integers make exact ties common
    x = rng.integers(-2, 3, size=(B, d)).astype(F16)
    wr = rng.integers(-1, 2, size=(d, E)).astype(F16)
    idx, w, logits = orc.route_topk(x, wr, k, True)
    for b in range(B):
        assert idx[b].tolist() == _topk_by_rank_count(logits[b], k)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_route_softmax_special_cases():
    """k = E with renorm is the library softmax over all logits; renorm=False is
    the full softmax read at the chosen experts."""
    from scipy.special import softmax
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 64)).astype(F16)
    wr = (0.5 * rng.standard_normal((64, 8))).astype(F16)
    idx, w, logits = orc.route_topk(x, wr, 8, True)
    full = softmax(logits, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, idx.astype(np.int64), axis=1), rtol=1e-13, atol=0)
    idx2, w2, _ = orc.route_topk(x, wr, 2, False)
    np.testing.assert_allclose(w2, np.take_along_axis(full, idx2.astype(np.int64), axis=1), rtol=1e-13, atol=0)
    # logits are x . W_r (not the transpose): compare with the library matmul
    np.testing.assert_allclose(logits, x.astype(np.float64) @ wr.astype(np.float64), rtol=0, atol=0)


# ---------------------------------------------------------------------------
# INT2 quantiser
# ---------------------------------------------------------------------------

def _golden_quant_matrix():
    g = load_golden("int2_quant.json")
    cols, qcols = [], []
    for c in g["columns"]:
        reps = 64 // len(c["pattern"])
        cols.append(np.tile(np.asarray(c["pattern"], np.float64), reps))
        qcols.append(np.tile(np.asarray(c["q_pattern"]), reps))
    return g, np.stack(cols, axis=1).astype(F16), np.stack(qcols, axis=1)


def test_quant_golden():
    g, w, q_exp = _golden_quant_matrix()
    q, s, z = orc.quantize_int2(w)
    assert q.tolist() == q_exp.tolist()
    assert s.astype(np.float64)[0].tolist() == [c["scale"] for c in g["columns"]]
    assert z.astype(np.float64)[0].tolist() == [c["zero"] for c in g["columns"]]
    deq = orc.dequantize_int2(q, s, z)
    # degenerate column: dequantisation returns the constant exactly
    assert np.all(deq[:, 1] == w[:, 1].astype(np.float64))
    # grid column: the values on the grid {-0.25, 0, 0.25, 0.5} come back exactly,
    # the half-way values go to the even code
    w0 = w[:, 0].astype(np.float64)
    on_grid = np.isin(w0, [-0.25, 0.0, 0.25, 0.5])
    assert np.all(deq[on_grid, 0] == w0[on_grid])
    assert np.all(np.abs(deq[~on_grid, 0] - w0[~on_grid]) == 0.125)


def test_quant_random_properties():
    rng = np.random.default_rng(11)
    d, f = 256, 96
    w = (0.02 * rng.standard_normal((d, f))).astype(F16)
    q, s, z = orc.quantize_int2(w)
    assert q.dtype == np.uint8 and q.max() <= 3
    deq = orc.dequantize_int2(q, s, z)
    sg = np.repeat(s.astype(np.float64), 64, axis=0)
    zg = np.repeat(z.astype(np.float64), 64, axis=0)
    # rounding to the nearest code: error at most half a step, plus the fp16 rounding of zero
    bound = sg * (0.5 + 2.0 ** -10 * (1.0 + np.abs(zg)))
    assert np.all(np.abs(deq - w.astype(np.float64)) <= bound)
    # the group minimum and maximum land on the end codes
    qg = q.reshape(d // 64, 64, f)
    assert np.all(qg.min(axis=1) == 0) and np.all(qg.max(axis=1) == 3)
    # scale is the fp16 rounding of (max - min) / 3
    wg = w.astype(np.float64).reshape(d // 64, 64, f)
    np.testing.assert_allclose(s.astype(np.float64), (wg.max(1) - wg.min(1)) / 3, rtol=2.0 ** -10, atol=0)


def test_dequant_definition():
    q = np.array([[0], [3]] * 32, dtype=np.uint8)
    s = np.array([[0.5]], dtype=F16)
    z = np.array([[1.25]], dtype=F16)
    deq = orc.dequantize_int2(q, s, z)
    assert deq[0, 0] == 0.5 * (0 - 1.25) and deq[1, 0] == 0.5 * (3 - 1.25)


# ---------------------------------------------------------------------------
# sparse SwiGLU expert
# ---------------------------------------------------------------------------

def _golden_expert():
    g = load_golden("sparse_expert.json")
    return g, _h(g["x"]), _h(g["w_gate"]), np.asarray(g["w_up"], np.float64), _h(g["w_down"])


def test_expert_golden():
    g, x, wg, wu, wd = _golden_expert()
    for case in g["cases"]:
        y, v, mask = orc.sparse_swiglu_expert(x, wg, wu, wd, case["t"])
        assert mask.tolist() == case["mask"]
        np.testing.assert_allclose(y, case["y"], rtol=1e-14, atol=1e-12)


def _rand_expert(d, f, seed, n=3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, d)).astype(F16)
    wg = (0.2 * rng.standard_normal((d, f))).astype(F16)
    wu = (0.2 * rng.standard_normal((d, f))).astype(F16)
    wd = (0.2 * rng.standard_normal((f, d))).astype(F16)
    q, s, z = orc.quantize_int2(wu)
    return x, wg, orc.dequantize_int2(q, s, z), wd


def test_expert_t0_is_dense_swiglu_library():
    """t = 0 keeps every non-zero column: the result is the dense SwiGLU expert,
    here computed with torch's silu and matmul in fp64."""
    x, wg, wu, wd = _rand_expert(128, 96, 1)
    y, v, mask = orc.sparse_swiglu_expert(x, wg, wu, wd, 0.0)
    assert mask.all()
    tx = torch.from_numpy(x.astype(np.float64))
    ref = (torch.nn.functional.silu(tx @ torch.from_numpy(wg.astype(np.float64)))
           * (tx @ torch.from_numpy(wu))) @ torch.from_numpy(wd.astype(np.float64))
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_expert_tinf_is_exact_zero():
    x, wg, wu, wd = _rand_expert(64, 64, 2)
    y, v, mask = orc.sparse_swiglu_expert(x, wg, wu, wd, math.inf)
    assert not mask.any()
    assert np.all(y == 0) and not np.any(np.signbit(y))


def test_expert_gate_zero_gives_zero():
    x, wg, wu, wd = _rand_expert(64, 64, 3)
    y, _, _ = orc.sparse_swiglu_expert(x, np.zeros_like(wg), wu, wd, 0.1)
    assert np.all(y == 0)


def test_expert_linear_in_down():
    x, wg, wu, wd = _rand_expert(64, 64, 4)
    y1, _, _ = orc.sparse_swiglu_expert(x, wg, wu, wd, 0.3)
    y2, _, _ = orc.sparse_swiglu_expert(x, wg, wu, 2 * wd.astype(np.float64), 0.3)
    np.testing.assert_allclose(y2, 2 * y1, rtol=1e-13, atol=1e-13)


def test_expert_kept_count_monotone():
    x, wg, wu, wd = _rand_expert(64, 128, 5)
    prev = None
    for t in [0.0, 0.1, 0.2, 0.5, 1.0, 2.0, 1e9]:
        _, _, mask = orc.sparse_swiglu_expert(x, wg, wu, wd, t)
        kept = mask.sum()
        assert prev is None or kept <= prev
        prev = kept


def test_expert_bruteforce_loops():
    """Scalar loops over every (token, column, input) on tiny shapes."""
    rng = np.random.default_rng(6)
    n, d, f = 2, 5, 7
    x = rng.standard_normal((n, d)).astype(F16)
    wg = rng.standard_normal((d, f)).astype(F16)
    wu = rng.standard_normal((d, f))
    wd = rng.standard_normal((f, d)).astype(F16)
    t = 0.8
    y, _, _ = orc.sparse_swiglu_expert(x, wg, wu, wd, t)
    for b in range(n):
        out = [0.0] * d
        for i in range(f):
            vi = sum(float(x[b, k]) * wu[k, i] for k in range(d))
            if not abs(vi) > t:
                continue
            gi = sum(float(x[b, k]) * float(wg[k, i]) for k in range(d))
            hi = gi / (1.0 + math.exp(-gi)) * vi
            for c in range(d):
                out[c] += hi * float(wd[i, c])
        np.testing.assert_allclose(y[b], out, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# threshold calibration, RMSNorm
# ---------------------------------------------------------------------------

def test_quantile_golden():
    g = load_golden("quantile.json")
    for pct, t in g["cases"]:
        assert orc.quantile_threshold(np.asarray(g["v"], np.float64), pct) == t


@pytest.mark.parametrize("pct", [1, 37, 50, 70, 90, 99, 100])
def test_quantile_is_inverted_cdf(pct):
    rng = np.random.default_rng(pct)
    v = rng.standard_normal(1001)
    exp = np.quantile(np.abs(v), pct / 100.0, method="inverted_cdf")
    assert orc.quantile_threshold(v, pct) == exp


def test_rmsnorm_closed_form():
    np.testing.assert_allclose(orc.rmsnorm(np.array([[3.0, 4.0]])),
                               [[3 / math.sqrt(12.5 + 1e-6), 4 / math.sqrt(12.5 + 1e-6)]], rtol=1e-15)
    y = np.random.default_rng(0).standard_normal((3, 256)) * 7
    r = orc.rmsnorm(y, eps=0.0)
    np.testing.assert_allclose(np.mean(r * r, axis=1), 1.0, rtol=1e-13)


# ---------------------------------------------------------------------------
# MoE layer
# ---------------------------------------------------------------------------

def _golden_layer():
    g = load_golden("moe_layer.json")

    def ex(e):
        return dict(w_gate=_h(e["w_gate"]), w_up_deq=np.asarray(e["w_up"], np.float64),
                    w_down=_h(e["w_down"]), thr=e["thr"])
    return g, [ex(e) for e in g["experts"]], [ex(e) for e in g["shared"]]


def test_layer_golden():
    g, experts, shared = _golden_layer()
    x, wr = _h(g["x"]), _h(g["w_router"])
    y, info = orc.moe_layer(x, wr, experts, 2, True)
    assert info["idx"].tolist() == g["idx"]
    np.testing.assert_allclose(info["w"], g["w"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(y, g["y_routed_only"], rtol=1e-14)
    y, _ = orc.moe_layer(x, wr, experts, 2, True, shared=shared)
    np.testing.assert_allclose(y, g["y_with_shared"], rtol=1e-14)
    y, _ = orc.moe_layer(x, wr, experts, 2, True, shared=shared, rmsnorm_out=True)
    np.testing.assert_allclose(y, g["y_with_shared_rmsnorm"], rtol=1e-14)


def _rand_layer(E, d, f, seed):
    rng = np.random.default_rng(seed)
    exps = []
    for e in range(E):
        x0, wg, wu, wd = _rand_expert(d, f, seed * 100 + e, n=1)
        exps.append(dict(w_gate=wg, w_up_deq=wu, w_down=wd, thr=0.4))
    wr = (0.3 * rng.standard_normal((d, E))).astype(F16)
    x = rng.standard_normal((5, d)).astype(F16)
    return x, wr, exps


def test_layer_k_equals_E_is_softmax_mixture():
    x, wr, exps = _rand_layer(4, 64, 64, 7)
    y, info = orc.moe_layer(x, wr, exps, 4, True)
    from scipy.special import softmax
    p = softmax(x.astype(np.float64) @ wr.astype(np.float64), axis=1)
    ref = np.zeros_like(y)
    for e, ex in enumerate(exps):
        ye, _, _ = orc.sparse_swiglu_expert(x, ex["w_gate"], ex["w_up_deq"], ex["w_down"], ex["thr"])
        ref += p[:, e:e + 1] * ye
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_layer_tokens_independent():
    """Each token's output depends only on that token: permuting the batch
    permutes the outputs."""
    x, wr, exps = _rand_layer(8, 64, 64, 8)
    y, _ = orc.moe_layer(x, wr, exps, 2, True)
    perm = np.array([3, 0, 4, 1, 2])
    yp, _ = orc.moe_layer(x[perm], wr, exps, 2, True)
    np.testing.assert_allclose(yp, y[perm], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by a pin above
# ---------------------------------------------------------------------------

def _expert_golden_passes():
    try:
        test_expert_golden()
        return True
    except AssertionError:
        return False


def test_mutation_sigmoid_instead_of_silu(monkeypatch):
    monkeypatch.setattr(orc, "silu", lambda a: 1.0 / (1.0 + np.exp(-np.asarray(a, np.float64))))
    assert not _expert_golden_passes()


def test_mutation_silu_sign(monkeypatch):
    monkeypatch.setattr(orc, "silu", lambda a: np.asarray(a, np.float64) / (1.0 + np.exp(np.asarray(a, np.float64))))
    assert not _expert_golden_passes()


def test_mutation_non_strict_mask(monkeypatch):
    real = orc.sparse_swiglu_expert

    def mutant(x, wg, wu, wd, t, mask=None):
        v = np.asarray(x, np.float64) @ np.asarray(wu, np.float64)
        return real(x, wg, wu, wd, t, mask=np.abs(v) >= t)
    monkeypatch.setattr(orc, "sparse_swiglu_expert", mutant)
    assert not _expert_golden_passes()


def test_mutation_transposed_down(monkeypatch):
    real = orc.sparse_swiglu_expert
    monkeypatch.setattr(orc, "sparse_swiglu_expert",
                        lambda x, wg, wu, wd, t, mask=None: real(x, wg, wu, np.asarray(wd)[:, ::-1], t, mask))
    assert not _expert_golden_passes()


def test_mutation_zero_sign_in_quantiser(monkeypatch):
    real = orc.dequantize_int2
    monkeypatch.setattr(orc, "dequantize_int2", lambda q, s, z: real(q, s, -np.asarray(z)))
    with pytest.raises(AssertionError):
        test_quant_golden()


def test_mutation_floor_instead_of_rint(monkeypatch):
    class NpFloor:
        def __getattr__(self, name):
            return np.floor if name == "rint" else getattr(np, name)
    monkeypatch.setattr(orc, "np", NpFloor())
    with pytest.raises(AssertionError):
        test_quant_golden()


def test_mutation_router_tie_break(monkeypatch):
    real = orc.route_topk

    def mutant(x, wr, k, renorm=True):
        # ties go to the higher index: reverse the expert order and map back
        E = np.asarray(wr).shape[1]
        idx, w, logits = real(x, np.asarray(wr)[:, ::-1], k, renorm)
        return (E - 1 - idx).astype(np.int32), w, logits[:, ::-1]
    monkeypatch.setattr(orc, "route_topk", mutant)
    with pytest.raises(AssertionError):
        test_route_golden()


def test_layer_additive_over_column_slices():
    """Every kept intermediate column contributes its own term h_i W^down[i, :] to an
    expert's output (steps 3 and 4 of Algorithm 1), so a layer's output (before the
    RMSNorm) is the sum of the layers whose experts keep only one slice of the columns
    each; the reference arm of the bench times one slice per step."""
    rng = np.random.default_rng(21)
    d, f, E, k = 128, 96, 4, 2
    x = rng.standard_normal((3, d)).astype(np.float16)
    wr = (rng.standard_normal((d, E)) * 0.1).astype(np.float16)
    experts = [dict(w_gate=rng.standard_normal((d, f)) * 0.05, w_up_deq=rng.standard_normal((d, f)) * 0.05,
                    w_down=rng.standard_normal((f, d)) * 0.05, thr=0.1) for _ in range(E)]
    y_full, _ = orc.moe_layer(x, wr, experts, k, True)
    total = np.zeros_like(y_full)
    for c in np.array_split(np.arange(f), 5):
        sl = [dict(w_gate=ex["w_gate"][:, c], w_up_deq=ex["w_up_deq"][:, c], w_down=ex["w_down"][c, :],
                   thr=ex["thr"]) for ex in experts]
        y, _ = orc.moe_layer(x, wr, sl, k, True)
        total += y
    np.testing.assert_allclose(total, y_full, rtol=0, atol=1e-14)
