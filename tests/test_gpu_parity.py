"""CUDA path vs the fp64 oracle, through the C ABI (marked gpu).

Inputs come from the seeded generator and are handed to both sides; thresholds are
computed by the oracle from calibration tokens.  Every comparison follows the band
rule of tests/parity.py.
"""

from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from tests import parity

pytestmark = pytest.mark.gpu

ses = pytest.importorskip("sparse_expert_swiglu_gb300")
from sparse_expert_swiglu_gb300 import synth  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ses.build_library()
    ses.lib()


def _np16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


# ---------------------------------------------------------------------------
# INT2 pack: bit-exact against the oracle's quantiser
# ---------------------------------------------------------------------------

def _pack_check(w_up: torch.Tensor):
    d, f = w_up.shape
    packed = ses.pack_int2_up(w_up.cuda().contiguous())
    q, s, z = ses.unpack_int2_up(packed, d, f)
    q_ref, s_ref, z_ref = orc.quantize_int2(_np16(w_up))
    assert np.array_equal(_np16(q), q_ref)
    # fp16 values equal (a zero point of -0 and +0 are the same value)
    assert np.array_equal(_np16(s).astype(np.float64), s_ref.astype(np.float64))
    assert np.array_equal(_np16(z).astype(np.float64), z_ref.astype(np.float64))
    # re-packing the same weights gives the same bytes
    assert torch.equal(packed, ses.pack_int2_up(w_up.cuda().contiguous()))


@pytest.mark.parametrize("d,f", [(256, 512), (768, 208), (4096, 1024), (64, 16)])
def test_pack_random(d, f):
    _pack_check(synth.normal_f16((d, f), 0.02, 7, d + f))


def test_pack_golden_and_degenerate():
    from tests.test_oracle_pins import _golden_quant_matrix
    _, w, q_exp = _golden_quant_matrix()
    w = np.concatenate([w, np.zeros((64, 13), np.float16)], axis=1)  # f = 16, an all-zero group too
    _pack_check(torch.from_numpy(w))
    q, _, _ = ses.unpack_int2_up(ses.pack_int2_up(torch.from_numpy(w).cuda()), 64, 16)
    assert np.array_equal(_np16(q)[:, :3], q_exp)


def test_pack_wide_range():
    # groups with large offsets, tiny spreads and sign mixes
    rng = np.random.default_rng(3)
    base = rng.uniform(-1000, 1000, size=(1, 64)).astype(np.float32)
    spread = 10.0 ** rng.uniform(-6, 2, size=(1, 64)).astype(np.float32)
    w = (base + spread * rng.standard_normal((512, 64)).astype(np.float32)).astype(np.float16)
    _pack_check(torch.from_numpy(w))


# ---------------------------------------------------------------------------
# router
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,d,E,k,renorm", [(1, 4096, 8, 2, True), (32, 4096, 8, 2, True),
                                            (64, 2048, 64, 6, True), (5, 256, 4, 1, False),
                                            (7, 512, 16, 3, False), (3, 256, 256, 8, True)])
def test_route_matches_oracle(B, d, E, k, renorm):
    x = synth.tokens(B, d, 11)
    wr = synth.router(d, E, 11)
    idx, w, cnt = ses.route_topk(x.cuda(), wr.cuda(), k, renorm)
    idx, w, cnt = _np16(idx), _np16(w), _np16(cnt)
    idx_ref, w_ref, logits = orc.route_topk(_np16(x), _np16(wr), k, renorm)
    S = np.abs(_np16(x).astype(np.float64)) @ np.abs(_np16(wr).astype(np.float64))
    ok, n_band = parity.route_band(logits, S, idx, k)
    assert ok and n_band == 0
    # weights: the oracle's softmax at the kernel's experts
    for b in range(B):
        l = logits[b, idx[b]] if renorm else logits[b]
        p = np.exp(l - l.max())
        p /= p.sum()
        exp = p if renorm else p[idx[b]]
        np.testing.assert_allclose(w[b], exp, rtol=0, atol=2e-6)
    assert np.array_equal(cnt, np.bincount(idx.ravel(), minlength=E))


def test_route_exact_ties():
    """Small integers make exact ties; fp32 sums of them are exact, so the kernel must
    apply the same tie-break (lower index first) as the oracle, with no band."""
    rng = np.random.default_rng(5)
    for E, k in [(8, 2), (16, 6), (64, 6), (12, 3)]:
        B, d = 16, 256
        x = rng.integers(-2, 3, size=(B, d)).astype(np.float16)
        wr = rng.integers(-1, 2, size=(d, E)).astype(np.float16)
        idx, _, _ = ses.route_topk(torch.from_numpy(x).cuda(), torch.from_numpy(wr).cuda(), k, True)
        idx_ref, _, _ = orc.route_topk(x, wr, k, True)
        assert np.array_equal(_np16(idx), idx_ref)


# ---------------------------------------------------------------------------
# one expert
# ---------------------------------------------------------------------------

class OracleExpert:
    def __init__(self, w_up, gate_t, down):
        self.q, self.s, self.z = orc.quantize_int2(_np16(w_up))
        self.w_up_deq = orc.dequantize_int2(self.q, self.s, self.z)
        self.w_gate = _np16(gate_t).T
        self.w_down = _np16(down)

    def thr(self, xcal, pct):
        return np.float32(orc.quantile_threshold(orc.expert_up(xcal, self.w_up_deq), pct))


@pytest.mark.parametrize("d,f,n", [(256, 512, 1), (256, 512, 4), (256, 512, 9), (768, 208, 3),
                                   (768, 208, 17), (2048, 1408, 8), (512, 4096, 2)])
@pytest.mark.parametrize("pct", [0, 50, 90, 101])
def test_expert_matches_oracle(d, f, n, pct):
    E, e = 3, 1
    de = synth.experts(E, d, f, 21)
    x = synth.tokens(n, d, 21)
    ox = OracleExpert(de.w_up[e], de.gate_t[e], de.down[e])
    xcal = _np16(synth.calibration_tokens(64, d, 21))
    t = np.float32(math.inf) if pct == 101 else ox.thr(xcal, pct)
    thr = torch.full((E,), float(t), dtype=torch.float32)
    ex = ses.Experts.from_dense(de.w_up.cuda(), de.gate_t.cuda(), de.down.cuda(), thr.cuda())
    y, dbg = ses.expert_sparse_swiglu(x.cuda(), ex, e, debug=True)
    y = _np16(y)
    v_gpu = _np16(dbg["v"])[:, 0]
    m_gpu = parity.unpack_mask(_np16(dbg["mask"])[:, 0], f)
    xs = _np16(x)
    v_ref = orc.expert_up(xs, ox.w_up_deq)
    S = parity.up_magnitude(xs, ox.q, ox.s, ox.z)
    assert parity.check_v(v_gpu, v_ref, S) <= parity.TAU
    bad, n_band = parity.check_mask(m_gpu, v_ref, S, float(t))
    assert bad == 0
    y_ref, _, _ = orc.sparse_swiglu_expert(xs, ox.w_gate, ox.w_up_deq, ox.w_down, float(t), mask=m_gpu)
    if pct == 101:
        assert not m_gpu.any()
        assert np.all(y.view(np.uint16) == 0)  # exactly +0
    max_abs, rel = parity.check_y(y, y_ref)
    assert max_abs <= parity.Y_MAX_ABS
    assert rel <= parity.Y_REL_L2 or np.linalg.norm(y_ref) == 0


def test_expert_deterministic():
    d, f, n = 768, 208, 9
    de = synth.experts(2, d, f, 5)
    thr = torch.tensor([0.3, 0.3], dtype=torch.float32).cuda()
    ex = ses.Experts.from_dense(de.w_up.cuda(), de.gate_t.cuda(), de.down.cuda(), thr)
    x = synth.tokens(n, d, 5).cuda()
    ws = ses.Workspace(ses.expert_workspace_bytes(n, d, f))
    y1 = ses.expert_sparse_swiglu(x, ex, 0, ws=ws).clone()
    y2 = ses.expert_sparse_swiglu(x, ex, 0, ws=ws)
    assert torch.equal(y1, y2)
    assert ws.status() == 0


def test_expert_empty_batch():
    d, f = 256, 512
    de = synth.experts(1, d, f, 5)
    ex = ses.Experts.from_dense(de.w_up.cuda(), de.gate_t.cuda(), de.down.cuda(),
                                torch.zeros(1, dtype=torch.float32).cuda())
    y = ses.expert_sparse_swiglu(torch.empty((0, d), dtype=torch.float16, device="cuda"), ex, 0)
    assert y.shape == (0, d)


# ---------------------------------------------------------------------------
# whole layer
# ---------------------------------------------------------------------------

# Decisions a case may have the band excuse: inside the fp32 rounding band of the boundary
# and taken differently by the kernel and the oracle.  The band itself is wide (about 0.3 %
# of mask decisions lie in it: S counts |z| times the group's sum of |x|), but the kernel's
# error is far below its half-width, so excused decisions stay below 1e-4 of all of them
# (at least a few are allowed), and at most one top-k choice in 16 tokens.
def band_bounds(B, n_mask_decisions):
    return max(2, B // 16), max(4, int(1e-4 * n_mask_decisions))


def check_layer(xs, wrs, k, renorm, rmsnorm, y, dbg, thr_r, thr_s, oracle_expert, shared, f,
                expect_zero=False):
    """The layer's outputs against the oracle on the same input: routing (band rule), weights,
    every v within the rounding band, masks exact outside it, band counts within bounds, y
    within the tolerance after the oracle takes the kernel's band decisions."""
    B = xs.shape[0]
    E = thr_r.shape[0]
    idx_ref, _, logits = orc.route_topk(xs, wrs, k, renorm)
    S_route = np.abs(xs.astype(np.float64)) @ np.abs(wrs.astype(np.float64))
    y = _np16(y)
    idx_gpu = _np16(dbg["topk_idx"])
    w_gpu = _np16(dbg["topk_w"])
    ok, n_band_route = parity.route_band(logits, S_route, idx_gpu, k)
    assert ok
    # oracle weights at the kernel's experts
    w_at = np.empty((B, k))
    for b in range(B):
        l = logits[b, idx_gpu[b]] if renorm else logits[b]
        p = np.exp(l - l.max())
        p /= p.sum()
        w_at[b] = p if renorm else p[idx_gpu[b]]
    np.testing.assert_allclose(w_gpu, w_at, rtol=0, atol=2e-6)
    v_all = _np16(dbg["v"])
    m_all = parity.unpack_mask(_np16(dbg["mask"]), f)
    masks = {}
    experts_o = [None] * E
    n_band_mask, n_excused, n_decisions = 0, 0, 0
    worst_v = 0.0
    for e in sorted(set(idx_gpu.ravel().tolist())):
        rows, cols = np.nonzero(idx_gpu == e)
        order = np.argsort(rows, kind="stable")
        toks, slots = rows[order], cols[order]
        ox = oracle_expert("r", e)
        v_ref = orc.expert_up(xs[toks], ox.w_up_deq)
        S = parity.up_magnitude(xs[toks], ox.q, ox.s, ox.z)
        worst_v = max(worst_v, parity.check_v(v_all[toks, slots], v_ref, S))
        bad, nb = parity.check_mask(m_all[toks, slots], v_ref, S, float(thr_r[e]))
        assert bad == 0
        n_band_mask += nb
        n_excused += parity.mask_excused(m_all[toks, slots], v_ref, S, float(thr_r[e]))
        n_decisions += v_ref.size
        masks[("r", e)] = m_all[toks, slots]
        experts_o[e] = dict(w_gate=ox.w_gate, w_up_deq=ox.w_up_deq, w_down=ox.w_down, thr=float(thr_r[e]))
    shared_o = []
    for s_ in range(shared):
        ox = oracle_expert("s", s_)
        v_ref = orc.expert_up(xs, ox.w_up_deq)
        S = parity.up_magnitude(xs, ox.q, ox.s, ox.z)
        worst_v = max(worst_v, parity.check_v(v_all[:, k + s_], v_ref, S))
        bad, nb = parity.check_mask(m_all[:, k + s_], v_ref, S, float(thr_s[s_]))
        assert bad == 0
        n_band_mask += nb
        n_excused += parity.mask_excused(m_all[:, k + s_], v_ref, S, float(thr_s[s_]))
        n_decisions += v_ref.size
        masks[("s", s_)] = m_all[:, k + s_]
        shared_o.append(dict(w_gate=ox.w_gate, w_up_deq=ox.w_up_deq, w_down=ox.w_down, thr=float(thr_s[s_])))
    assert worst_v <= parity.TAU
    route_max, mask_max = band_bounds(B, n_decisions)
    print(f"band: routing choices excused {n_band_route} of {B} tokens; mask decisions in the band "
          f"{n_band_mask}, excused {n_excused}, of {n_decisions}; worst |v - v_ref| / S {worst_v:.2e}")
    assert n_band_route <= route_max, (n_band_route, route_max)
    assert n_excused <= mask_max, (n_excused, mask_max)
    y_ref, _ = orc.moe_layer(xs, wrs, experts_o, k, renorm, shared=shared_o,
                             rmsnorm_out=rmsnorm, route=(idx_gpu, w_at), masks=masks)
    max_abs, rel = parity.check_y(y, y_ref)
    if expect_zero:
        assert np.all(y.view(np.uint16) == 0)
    assert max_abs <= parity.Y_MAX_ABS, max_abs
    assert rel <= parity.Y_REL_L2 or np.linalg.norm(y_ref) == 0, rel
    kept = m_all[:, :k].mean() if B else 0.0
    return dict(max_abs=max_abs, rel=rel, band_mask=n_band_mask, excused_mask=n_excused, band_route=n_band_route,
                worst_v=worst_v, kept=float(kept), decisions=n_decisions)


def run_layer_case(d, f, E, k, B, shared, pcts, seed, ncal=64, renorm=True, rmsnorm=False,
                   gen_device="cpu", interleave=False, host_rows=False, oracle_cache=None):
    dev = gen_device
    de = synth.experts(E, d, f, seed, device=dev)
    ds = synth.experts(shared, d, f, seed, device=dev, kind=1) if shared else None
    wr = synth.router(d, E, seed, device=dev)
    x = synth.tokens(B, d, seed, device=dev)
    xs, wrs = _np16(x), _np16(wr)
    xcal = _np16(synth.calibration_tokens(ncal, d, seed, device=dev))
    idx_ref, _, _ = orc.route_topk(xs, wrs, k, renorm)
    cache = {} if oracle_cache is None else oracle_cache

    def oracle_expert(kind, e):
        key = (seed, d, f, kind, e)
        if key not in cache:
            src = de if kind == "r" else ds
            cache[key] = OracleExpert(src.w_up[e], src.gate_t[e], src.down[e])
        return cache[key]

    routed_used = sorted(set(idx_ref.ravel().tolist()))
    ex_gpu = ses.Experts.from_dense(de.w_up.to("cuda"), de.gate_t.to("cuda"), de.down.to("cuda"),
                                    torch.zeros(E, dtype=torch.float32, device="cuda"),
                                    interleave=interleave)
    sh_gpu = None
    if shared:
        sh_gpu = ses.Experts.from_dense(ds.w_up.to("cuda"), ds.gate_t.to("cuda"), ds.down.to("cuda"),
                                        torch.zeros(shared, dtype=torch.float32, device="cuda"),
                                        interleave=interleave)
    if host_rows:
        # gate/down rows in page-locked host memory; thresholds shared with ex_gpu/sh_gpu
        layer = ses.Layer(wr.to("cuda"), ex_gpu.to_host_rows(), k, renorm,
                          sh_gpu.to_host_rows() if shared else None)
        ws = ses.Workspace(ses.layer_host_rows_workspace_bytes(layer, B))
        decode = ses.layer_decode_host_rows
    else:
        layer = ses.Layer(wr.to("cuda"), ex_gpu, k, renorm, sh_gpu)
        ws = ses.Workspace(ses.layer_workspace_bytes(layer, B))
        decode = ses.layer_decode
    results = []
    for pct in pcts:
        thr_r = np.zeros(E, np.float32)
        for e in routed_used:
            thr_r[e] = math.inf if pct == 101 else oracle_expert("r", e).thr(xcal, pct)
        thr_s = np.zeros(shared, np.float32)
        for s in range(shared):
            thr_s[s] = math.inf if pct == 101 else oracle_expert("s", s).thr(xcal, pct)
        ex_gpu.thr.copy_(torch.from_numpy(thr_r))
        if shared:
            sh_gpu.thr.copy_(torch.from_numpy(thr_s))
        y, dbg = decode(x.to("cuda"), layer, rmsnorm=rmsnorm, ws=ws, debug=True)
        assert ws.status() == 0
        r = check_layer(xs, wrs, k, renorm, rmsnorm, y, dbg, thr_r, thr_s, oracle_expert, shared, f,
                        expect_zero=(pct == 101 and not shared))
        results.append(dict(pct=pct, **r))
    return results


def test_layer_tiny():
    """d=256, f=512, E=8, top-2, 4 tokens; thresholds from 256 calibration tokens."""
    run_layer_case(256, 512, 8, 2, 4, 0, [0, 50, 90, 101], seed=0, ncal=256)


def test_layer_tiny_rmsnorm_and_full_softmax():
    run_layer_case(256, 512, 8, 2, 4, 0, [50], seed=1, ncal=256, renorm=False, rmsnorm=True)


def test_layer_ragged_with_shared():
    """d=768 (a partial 512-superblock), f=208 (13 column tiles, mask words ragged),
    9 tokens (a group of 8 and a group of 1), one shared expert."""
    run_layer_case(768, 208, 4, 2, 9, 1, [0, 50, 101], seed=2)


@pytest.mark.parametrize("B,pcts", [(20, [0, 50, 101]), (64, [50])])
def test_layer_batched_ragged_with_shared(B, pcts):
    """The batched path (16 to 64 tokens) on a ragged layer: d=768 (a partial 512-input
    superblock, 3 slices of 256), f=208 (13 column tiles: an odd number, so the last mask
    word is half written; 4 row tiles of 64 with a short last one), 4 experts top-2 (up to
    64 tokens per expert), one shared expert serving every token."""
    run_layer_case(768, 208, 4, 2, B, 1, pcts, seed=21)


def test_layer_batched_d2048_shared():
    """The batched path at d = 2048 (one 2048-column chunk over 16 warps), f = 1408 as in
    DeepSeek-V2-Lite, 8 routed experts top-2 and 2 shared experts, 32 tokens (8 per routed
    expert on average, 32 per shared expert: two groups of 16)."""
    run_layer_case(2048, 1408, 8, 2, 32, 2, [0, 90], seed=23, gen_device="cuda")


def test_layer_batched_reproducible():
    """The batched path sums in fixed orders: two calls give identical bits."""
    d, f, E, k, B = 1024, 512, 8, 2, 32
    de = synth.experts(E, d, f, 22)
    ex = ses.Experts.from_dense(de.w_up.cuda(), de.gate_t.cuda(), de.down.cuda(),
                                torch.full((E,), 0.05, dtype=torch.float32).cuda(), interleave=True)
    layer = ses.Layer(synth.router(d, E, 22).cuda(), ex, k)
    assert ses.layer_path(layer, B) == "batched"
    x = synth.tokens(B, d, 22).cuda()
    ws = ses.Workspace(ses.layer_workspace_bytes(layer, B))
    y1 = ses.layer_decode(x, layer, ws=ws, rmsnorm=True).clone()
    y2 = ses.layer_decode(x, layer, ws=ws, rmsnorm=True)
    assert torch.equal(y1, y2)
    assert ws.status() == 0


def test_layer_deepseek_v2_lite_shape():
    """d=2048, f=1408, 64 routed experts top-6, 2 shared experts."""
    run_layer_case(2048, 1408, 64, 6, 8, 2, [0, 50, 90], seed=3, gen_device="cuda")


def test_layer_mixtral_8x7b_b1():
    """d=4096, f=14336, 8 experts top-2, one decode token, 0/50/70/90% thresholds."""
    run_layer_case(4096, 14336, 8, 2, 1, 0, [0, 50, 70, 90], seed=4, gen_device="cuda")


def test_layer_mixtral_8x7b_batch8():
    run_layer_case(4096, 14336, 8, 2, 8, 0, [70], seed=5, gen_device="cuda")


def test_layer_mixtral_8x7b_batch3():
    """Three tokens: a pair through the two-kernel decode path, then the third token
    through the one-kernel layer, on one workspace."""
    run_layer_case(4096, 14336, 8, 2, 3, 0, [70], seed=7, gen_device="cuda")


def test_layer_general_path_3_tokens():
    """Three tokens with 128 routed experts (more than the decode paths route): the
    general path, groups of at most 3 tokens on the tensor-core gather with the 4-row x
    buffer."""
    run_layer_case(1024, 512, 128, 2, 3, 0, [0, 70], seed=17)


def test_layer_deepseek_v2_lite_pairs():
    """Four tokens of the DeepSeek-V2-Lite shape (64 routed experts top-6, 2 shared):
    two pairs through the two-kernel decode path, each pair's routing, v and masks
    written at its tokens."""
    run_layer_case(2048, 1408, 64, 6, 4, 2, [0, 90], seed=18, gen_device="cuda")


def test_workspace_shared_across_token_counts():
    """One workspace (sized for the largest call) used by calls with 4, 1, 2, 8 and 3
    tokens in turn: every result equals that of a call on a fresh workspace, up to the
    order of the decode paths' fp32 additions."""
    d, f, E, k = 1024, 512, 8, 2
    de = synth.experts(E, d, f, 19, device="cuda")
    ex = ses.Experts.from_dense(de.w_up, de.gate_t, de.down, torch.full((E,), 0.05, device="cuda"))
    layer = ses.Layer(synth.router(d, E, 19, device="cuda"), ex, k, True)
    counts = [4, 1, 2, 8, 3]
    paths = [ses.layer_path(layer, B) for B in counts]
    assert paths == ["decode_pairs", "decode_fused", "decode", "general", "decode_pairs"], paths
    shared_ws = ses.Workspace(max(ses.layer_workspace_bytes(layer, B) for B in counts))
    for i, B in enumerate(counts):
        x = synth.tokens(B, d, 190 + i, device="cuda")
        y_shared = ses.layer_decode(x, layer, rmsnorm=True, ws=shared_ws)
        y_fresh = ses.layer_decode(x, layer, rmsnorm=True, ws=ses.Workspace(ses.layer_workspace_bytes(layer, B)))
        torch.cuda.synchronize()
        assert shared_ws.status() == 0
        assert _same_up_to_sum_order(y_shared, y_fresh), (B, paths[i])


_BIG_ORACLE = {}


@pytest.fixture(scope="module", autouse=True)
def _drop_big_oracle():
    yield
    _BIG_ORACLE.clear()


@pytest.mark.parametrize("B", [16, 32])
def test_layer_mixtral_8x7b_batch_sweep(B):
    """The Mixtral-8x7B batch sweep's largest batches (70 %): 16 tokens on the general path,
    32 tokens (8 per expert) on the batched path; one set of experts for both."""
    run_layer_case(4096, 14336, 8, 2, B, 0, [70], seed=8, gen_device="cuda", oracle_cache=_BIG_ORACLE)


@pytest.mark.parametrize("B", [16, 32, 64])
def test_layer_deepseek_v2_lite_batches(B):
    """DeepSeek-V2-Lite shape (64 experts top-6, 2 shared experts) at 16, 32 and 64 tokens,
    0 % and 90 % (16 and 32 tokens on the general path, 64 on the batched path)."""
    run_layer_case(2048, 1408, 64, 6, B, 2, [0, 90], seed=9, gen_device="cuda", oracle_cache=_BIG_ORACLE)


def test_stack_mixtral_8x22b_spot_checks():
    """56 layers of the Mixtral-8x22B shape (d = 6144, f = 16384, 8 experts top-2), one token,
    70 % thresholds, each layer fed the RMS-normalised output of the one before it on the GPU
    (layers are generated one at a time); layers 0, 27 and 55 are checked against the oracle
    on the GPU's own input to that layer."""
    d, f, E, k, L, seed = 6144, 16384, 8, 2, 56, 77
    spots = (0, 27, 55)
    x = synth.tokens(1, d, seed, device="cuda")
    xcal = synth.calibration_tokens(64, d, seed, device="cuda")
    cws = ses.Workspace(ses.expert_workspace_bytes(64, d, f))
    ws = None
    for l in range(L):
        de = synth.experts(E, d, f, seed, device="cuda", layer=l)
        wr = synth.router(d, E, seed, device="cuda", layer=l)
        ex = ses.Experts.from_dense(de.w_up, de.gate_t, de.down,
                                    torch.full((E,), float("inf"), dtype=torch.float32, device="cuda"),
                                    interleave=True)
        # 70 % thresholds from the library's own v over the calibration tokens (set-up only:
        # the oracle check uses the same thresholds)
        thr = torch.zeros(E, dtype=torch.float32, device="cuda")
        for e in range(E):
            _, cd = ses.expert_sparse_swiglu(xcal, ex, e, ws=cws, debug=True)
            a = torch.sort(cd["v"].abs().flatten()).values
            thr[e] = a[(70 * a.numel() + 99) // 100 - 1]
        ex.thr.copy_(thr)
        layer = ses.Layer(wr, ex, k, True)
        if ws is None:
            ws = ses.Workspace(ses.layer_workspace_bytes(layer, 1))
        y, dbg = ses.layer_decode(x, layer, rmsnorm=True, ws=ws, debug=True)
        assert ws.status() == 0
        if l in spots:
            cache = {}

            def oracle_expert(kind, e, de=de):
                if e not in cache:
                    cache[e] = OracleExpert(de.w_up[e], de.gate_t[e], de.down[e])
                return cache[e]

            r = check_layer(_np16(x), _np16(wr), k, True, True, y, dbg, _np16(thr), np.zeros(0, np.float32),
                            oracle_expert, 0, f)
            print(f"layer {l}: {r}")
        x = y.clone()
        del de, ex, layer, dbg, y
        torch.cuda.empty_cache()


def test_layer_wide_hidden_general_path():
    """d = 6144 with five tokens: the general path's gather with 24 consumer warps (groups of
    at most 2 tokens on the CUDA cores, the 800-thread build)."""
    run_layer_case(6144, 1024, 8, 2, 5, 0, [0, 70], seed=75, gen_device="cuda", rmsnorm=True)


def test_layer_mixtral_8x22b_shape_b2():
    """d=6144, f=16384, two tokens (the decode path), RMSNorm output."""
    run_layer_case(6144, 16384, 8, 2, 2, 0, [70], seed=6, gen_device="cuda", rmsnorm=True)


# One or two tokens with 8, 16 or 32 routed experts take the fused decode kernel
# (routing, up projection, mask, gathered rows and sums in one kernel).

@pytest.mark.parametrize("B", [1, 2])
def test_decode_tiny(B):
    """d=256 (one partial superblock of 4 groups), f=512, E=8, top-2."""
    run_layer_case(256, 512, 8, 2, B, 0, [0, 50, 90, 101], seed=20 + B, ncal=256)


def test_decode_rmsnorm_and_full_softmax():
    run_layer_case(512, 512, 8, 2, 2, 0, [50], seed=23, ncal=256, renorm=False, rmsnorm=True)


def test_decode_ragged_with_shared():
    """d=768 (a partial superblock), f=208 (13 column tiles), two tokens, one shared expert."""
    run_layer_case(768, 208, 8, 2, 2, 1, [0, 50, 101], seed=24)


@pytest.mark.parametrize("E,k,shared,d,f", [(16, 4, 0, 1024, 704), (32, 8, 2, 2048, 1408)])
def test_decode_wider_routing(E, k, shared, d, f):
    run_layer_case(d, f, E, k, 2, shared, [0, 70], seed=25 + k, gen_device="cuda")


@pytest.mark.parametrize("B", [1, 2])
def test_decode_wide_hidden(B):
    """d = 6144 (Mixtral-8x22B width) on the decode path: one unit lane of 12 superblock
    warps in the up kernel, 24 gather warps."""
    run_layer_case(6144, 1024, 8, 2, B, 0, [0, 70], seed=70 + B, gen_device="cuda", rmsnorm=(B == 2))


@pytest.mark.parametrize("B", [1, 2])
def test_decode_deepseek_v2_lite(B):
    """DeepSeek-V2-Lite shape (64 routed experts, top-6, 2 shared experts, d = 2048,
    f = 1408) on the decode path: the router's 8-chunk reduction and two experts per
    lane in its top-k."""
    run_layer_case(2048, 1408, 64, 6, B, 2, [0, 50, 90], seed=60 + B, gen_device="cuda")


def test_decode_mixtral_8x7b_b2():
    run_layer_case(4096, 14336, 8, 2, 2, 0, [50, 90], seed=30, gen_device="cuda", rmsnorm=True)


@pytest.mark.parametrize("B", [1, 2, 5, 8])
def test_layer_interleaved_gate_down(B):
    """gate and down rows interleaved in one buffer (one read per kept column), on the
    decode path (1 or 2 tokens), in pairs (5 tokens) and on the general path (8 tokens),
    with a shared expert."""
    assert ses.Experts.from_dense(*[torch.zeros(s, dtype=torch.float16, device="cuda")
                                    for s in [(1, 256, 16), (1, 16, 256), (1, 16, 256)]],
                                  torch.zeros(1, device="cuda"), interleave=True).interleaved
    run_layer_case(1024, 352, 8, 2, B, 1, [0, 70], seed=40 + B, interleave=True)


def test_layer_path_selection():
    """One or two tokens with 8/16/32/64 routed experts take a decode path: one kernel for
    one token up to d = 4096, else two kernels up to d = 6144; three or four such tokens
    (up to six, or four with more than 16 routed experts) go through it in pairs; other
    shapes take the general path."""
    def layer(d, f, E):
        de = synth.experts(E, d, f, 50)
        ex = ses.Experts.from_dense(de.w_up.cuda(), de.gate_t.cuda(), de.down.cuda(),
                                    torch.zeros(E, dtype=torch.float32).cuda())
        return ses.Layer(synth.router(d, E, 50).cuda(), ex, 2)
    small = layer(1024, 256, 8)
    assert ses.layer_path(small, 1) == "decode_fused"
    assert ses.layer_path(small, 2) == "decode"
    # three to six tokens: two at a time through the decode path
    assert ses.layer_path(small, 3) == "decode_pairs"
    assert ses.layer_path(small, 6) == "decode_pairs"
    assert ses.layer_path(small, 7) == "general"
    assert ses.layer_path(layer(6144, 256, 8), 4) == "decode_pairs"
    assert ses.layer_path(layer(1024, 256, 128), 3) == "general"
    # with more than 16 routed experts only up to four tokens go in pairs
    assert ses.layer_path(layer(1024, 256, 64), 4) == "decode_pairs"
    assert ses.layer_path(layer(1024, 256, 64), 5) == "general"
    assert ses.layer_path(layer(1024, 256, 64), 1) == "decode_fused"
    assert ses.layer_path(layer(1024, 256, 128), 1) == "general"
    assert ses.layer_path(layer(4096, 256, 8), 1) == "decode_fused"
    assert ses.layer_path(layer(4096, 256, 8), 2) == "decode"
    assert ses.layer_path(layer(6144, 256, 8), 1) == "decode"
    assert ses.layer_path(layer(6400, 256, 8), 1) == "general"
    # 16 to 64 tokens with d <= 4096 and at least 6 tokens per routed expert on average:
    # the batched path
    assert ses.layer_path(small, 8) == "general"
    assert ses.layer_path(small, 16) == "general"
    assert ses.layer_path(small, 24) == "batched"
    assert ses.layer_path(small, 32) == "batched"
    assert ses.layer_path(small, 64) == "batched"
    assert ses.layer_path(small, 65) == "general"
    assert ses.layer_path(layer(6144, 256, 8), 16) == "general"


def _same_up_to_sum_order(a, b):
    """Equal up to the order of the fp32 additions: the decode path adds the CTAs'
    shares of y in a varying order.  A reordered sum of n terms differs by at most about
    n * 2^-24 times the terms' magnitude (1e-4 of max |y| covers the 152-share sum with
    margin), and the fp16 rounding after it can add one ulp of the value."""
    a32, b32 = a.float(), b.float()
    ulp = torch.clamp(torch.maximum(a32.abs(), b32.abs()), min=2.0 ** -14) * 2.0 ** -10
    tol = ulp + 1e-4 * float(b32.abs().max())
    diff = (a32 - b32).abs()
    ok = bool((diff <= tol).all())
    if not ok:
        i = int(torch.argmax(diff - tol))
        print("worst", i, float(a32.view(-1)[i]), float(b32.view(-1)[i]), float(tol.view(-1)[i]))
    return ok


@pytest.mark.parametrize("B", [1, 2])
def test_decode_host_rows(B):
    """FloE's on-the-fly setting: gate and down rows in page-locked host memory, only the
    kept rows fetched (up kernel, fetch kernel, gather kernel); one shared expert,
    interleaved rows for one token, separate buffers for two."""
    run_layer_case(1024, 352, 8, 2, B, 1, [0, 70, 101], seed=80 + B, interleave=(B == 1), host_rows=True)


def test_decode_host_rows_mixtral_8x7b():
    """Host-resident rows at the Mixtral-8x7B layer size (d = 4096, f = 14336)."""
    run_layer_case(4096, 14336, 8, 2, 1, 0, [70], seed=90, gen_device="cuda", interleave=True,
                   host_rows=True)


def test_decode_host_rows_match_device_rows():
    """The host-rows call gives the device-rows result up to the order of the fp32
    additions (DeepSeek-V2-Lite shape, two tokens, RMSNorm); layer_decode refuses host
    rows, and shapes off the decode path are unsupported."""
    d, f, E, k, ns = 2048, 1408, 64, 6, 2
    de, ds = synth.experts(E, d, f, 95, device="cuda"), synth.experts(ns, d, f, 95, device="cuda", kind=1)
    thr = lambda n: torch.full((n,), 0.02, dtype=torch.float32, device="cuda")  # noqa: E731
    ex = ses.Experts.from_dense(de.w_up, de.gate_t, de.down, thr(E), interleave=True)
    sh = ses.Experts.from_dense(ds.w_up, ds.gate_t, ds.down, thr(ns))
    wr = synth.router(d, E, 95, device="cuda")
    dev_layer = ses.Layer(wr, ex, k, True, sh)
    host_layer = ses.Layer(wr, ex.to_host_rows(), k, True, sh.to_host_rows())
    assert host_layer.routed.rows_on_host and host_layer.routed.interleaved
    x = synth.tokens(2, d, 95, device="cuda")
    y_dev = ses.layer_decode(x, dev_layer, rmsnorm=True)
    ws = ses.Workspace(ses.layer_host_rows_workspace_bytes(host_layer, 2))
    y_host = ses.layer_decode_host_rows(x, host_layer, rmsnorm=True, ws=ws)
    assert ws.status() == 0
    assert _same_up_to_sum_order(y_host, y_dev)
    with pytest.raises(ValueError):
        ses.layer_decode(x, host_layer)
    x5 = synth.tokens(5, d, 96, device="cuda")
    with pytest.raises(ses.MoeError):
        ses.layer_decode_host_rows(x5, host_layer)


def test_decode_host_rows_refuses_partly_registered_rows():
    """Host rows whose buffer is page-locked only in part (its first half registered): the
    call checks that the last byte of each row buffer is registered in the same mapping and
    refuses with MOE_ERR_INVALID_ARG, before anything is enqueued."""
    d, f, E, k = 1024, 352, 8, 2
    de = synth.experts(E, d, f, 97)
    ex = ses.Experts.from_dense(de.w_up.cuda(), de.gate_t.cuda(), de.down.cuda(),
                                torch.full((E,), 0.05, dtype=torch.float32).cuda())
    gate_h = de.gate_t.clone()  # pageable
    down_h = de.down.clone().pin_memory()
    cudart = torch.cuda.cudart()
    nbytes = gate_h.numel() * gate_h.element_size()
    assert int(cudart.cudaHostRegister(gate_h.data_ptr(), nbytes // 2, 0)) == 0
    try:
        host = ses.Experts(ex.up_packed, gate_h, down_h, ex.thr)
        assert host.rows_on_host and gate_h.is_pinned()
        layer = ses.Layer(synth.router(d, E, 97).cuda(), host, k)
        x = synth.tokens(1, d, 97).cuda()
        with pytest.raises(ses.MoeError) as err:
            ses.layer_decode_host_rows(x, layer)
        assert err.value.status == -1
        torch.cuda.synchronize()
    finally:
        assert int(cudart.cudaHostUnregister(gate_h.data_ptr())) == 0


def test_wait_timeout_is_reported_and_the_context_stays_usable():
    """A bounded wait that runs out (a barrier nothing completes, 20 rounds of at most
    about 1 ms) records MOE_ERR_TIMEOUT, which moe_get_status returns once and clears;
    a layer then runs on the same stream and workspace and gives the result it gave
    before."""
    d, f, E, k = 1024, 512, 8, 2
    de = synth.experts(E, d, f, 33)
    ex = ses.Experts.from_dense(de.w_up.cuda(), de.gate_t.cuda(), de.down.cuda(),
                                torch.full((E,), 0.05, dtype=torch.float32).cuda())
    layer = ses.Layer(synth.router(d, E, 33).cuda(), ex, k)
    x = synth.tokens(2, d, 33).cuda()
    ws = ses.Workspace(ses.layer_workspace_bytes(layer, 2))
    y0 = ses.layer_decode(x, layer, ws=ws)
    assert ws.status() == 0
    lib = ses.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.moe_selftest_wait_timeout(ws.ptr(), ws.nbytes, 20, stream) == 0
    assert ws.status() == -6  # MOE_ERR_TIMEOUT
    assert ws.status() == 0   # read once, then cleared
    y1 = ses.layer_decode(x, layer, ws=ws)
    assert ws.status() == 0
    assert _same_up_to_sum_order(y1, y0)
    assert lib.moe_selftest_wait_timeout(ws.ptr(), ws.nbytes, 0, stream) == -1


@pytest.mark.parametrize("B", [1, 2])
def test_decode_up_projection_repeatable(B):
    """v = x W~^up is formed in a fixed order on the decode path, so calls in a row must
    give identical bits.  At the Mixtral-8x7B shape (two unit lanes sharing the packed-strip
    ring) this catches a strip read before its copy landed: a parity wait on a ring stage
    cannot tell a phase from the one two back, so no lane may skip a phase of a stage."""
    d, f, E, k = 4096, 14336, 8, 2
    de = synth.experts(E, d, f, 30, device="cuda")
    ex = ses.Experts.from_dense(de.w_up, de.gate_t, de.down, torch.full((E,), 0.9, device="cuda"),
                                interleave=True)
    del de
    layer = ses.Layer(synth.router(d, E, 30, device="cuda"), ex, k, True)
    x = synth.tokens(B, d, 30, device="cuda")
    ws = ses.Workspace(ses.layer_workspace_bytes(layer, B))
    _, dbg = ses.layer_decode(x, layer, rmsnorm=True, ws=ws, debug=True)
    v0, m0 = dbg["v"].clone(), dbg["mask"].clone()
    differ = 0
    for _ in range(300):
        _, dbg = ses.layer_decode(x, layer, rmsnorm=True, ws=ws, debug=True)
        differ += int(not (torch.equal(dbg["v"], v0) and torch.equal(dbg["mask"], m0)))
    assert ws.status() == 0
    assert differ == 0, f"{differ} of 300 calls gave a different v or mask"


def test_prefetch_hook_leaves_results_unchanged():
    """The inter-expert prefetch hook only moves the predicted experts' packed up
    projections into L2: v and the masks are bit-identical with and without it, y agrees up
    to the order of its fp32 additions, also when the prefetch runs on a second stream
    beside the layer, with repeated, out-of-range and negative ids, and with a byte cap."""
    d, f, E, k = 4096, 2048, 8, 2
    de = synth.experts(E, d, f, 32, device="cuda")
    ex = ses.Experts.from_dense(de.w_up, de.gate_t, de.down, torch.full((E,), 0.5, device="cuda"),
                                interleave=True)
    del de
    layer = ses.Layer(synth.router(d, E, 32, device="cuda"), ex, k, True)
    x = synth.tokens(1, d, 32, device="cuda")
    ws = ses.Workspace(ses.layer_workspace_bytes(layer, 1))
    y0, dbg = ses.layer_decode(x, layer, rmsnorm=True, ws=ws, debug=True)
    y0, v0, m0 = y0.clone(), dbg["v"].clone(), dbg["mask"].clone()
    assert int(dbg["mask"].ne(0).sum()) > 0
    idx, _, _ = ses.route_topk(x, layer.w_router, k)
    junk = torch.tensor([-1, E, 3, 3, 1000, int(idx[0, 0])], dtype=torch.int32, device="cuda")
    per = ses.packed_bytes(d, f)

    def check():
        y, dbg = ses.layer_decode(x, layer, rmsnorm=True, ws=ws, debug=True)
        assert torch.equal(dbg["v"], v0) and torch.equal(dbg["mask"], m0)
        assert _same_up_to_sum_order(y, y0)

    for ids, cap in [(idx, 0), (junk, 0), (torch.arange(E, dtype=torch.int32, device="cuda"), 3 * per),
                     (idx, per - 1), (idx[:0], 0)]:
        ses.prefetch_experts(ex, ids, max_bytes=cap)
        check()
    # beside the layer, on a second stream
    side = torch.cuda.Stream()
    for _ in range(5):
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            ses.prefetch_experts(ex, torch.arange(E, dtype=torch.int32, device="cuda"))
        check()
        torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert ws.status() == 0


def test_nonfinite_tokens_keep_expert_ids_valid():
    """A token with NaN or infinite entries (an overflow upstream) must not become an
    invalid expert index: every router ranks a NaN logit as -inf, so each token's k
    experts stay k distinct valid ones on all three paths, and the layer finishes with a
    clean status (its output for such a token is not finite, as the oracle's would be)."""
    for d, f, E, k, B, path in [(1024, 512, 8, 2, 1, "decode_fused"), (1024, 512, 8, 2, 2, "decode"),
                                (1024, 512, 8, 2, 3, "decode_pairs"), (256, 512, 8, 2, 8, "general")]:
        de = synth.experts(E, d, f, 33, device="cuda")
        ex = ses.Experts.from_dense(de.w_up, de.gate_t, de.down, torch.full((E,), 0.05, device="cuda"))
        layer = ses.Layer(synth.router(d, E, 33, device="cuda"), ex, k, True)
        assert ses.layer_path(layer, B) == path
        x = synth.tokens(B, d, 33, device="cuda")
        x[0] = float("nan")
        if B > 1:
            x[1, 5] = float("inf")
            x[1, 6] = -float("inf")
        for idx in (ses.route_topk(x, layer.w_router, k)[0], ses.route_topk_noalloc(x, layer.w_router, k)[0]):
            idx = idx.cpu()
            assert int(idx.min()) >= 0 and int(idx.max()) < E
            assert all(len(set(row.tolist())) == k for row in idx)
        ws = ses.Workspace(ses.layer_workspace_bytes(layer, B))
        y, dbg = ses.layer_decode(x, layer, rmsnorm=False, ws=ws, debug=True)
        idx = dbg["topk_idx"].cpu()
        assert int(idx.min()) >= 0 and int(idx.max()) < E
        assert all(len(set(row.tolist())) == k for row in idx)
        assert ws.status() == 0
        if B > 2:
            # the other tokens are unaffected on the general path (own groups or exact sums)
            assert torch.isfinite(y[2:].float()).all()


def test_decode_repeated_calls_share_the_workspace():
    """Many calls in a row on one workspace (the decode kernels reset their accumulator
    and counters) give the same output up to the order of the fp32 additions."""
    d, f, E, k = 1024, 512, 8, 2
    de = synth.experts(E, d, f, 31)
    ex = ses.Experts.from_dense(de.w_up.cuda(), de.gate_t.cuda(), de.down.cuda(),
                                torch.full((E,), 0.05, dtype=torch.float32).cuda())
    layer = ses.Layer(synth.router(d, E, 31).cuda(), ex, k)
    x = synth.tokens(1, d, 31).cuda()
    ws = ses.Workspace(ses.layer_workspace_bytes(layer, 1))
    y0 = ses.layer_decode(x, layer, ws=ws, rmsnorm=True).clone()
    for _ in range(20):
        assert _same_up_to_sum_order(ses.layer_decode(x, layer, ws=ws, rmsnorm=True), y0)
    assert ws.status() == 0


def test_decode_workspace_shared_across_shapes():
    """One workspace serving layers of different widths and one or two tokens in turn:
    every call matches the same call on a fresh workspace (the accumulator of a wider
    earlier call must not leak into a later one)."""
    layers = []
    for i, (d, f) in enumerate([(1024, 512), (2048, 768)]):
        de = synth.experts(8, d, f, 60 + i)
        ex = ses.Experts.from_dense(de.w_up.cuda(), de.gate_t.cuda(), de.down.cuda(),
                                    torch.full((8,), 0.05, dtype=torch.float32).cuda(), interleave=True)
        layers.append(ses.Layer(synth.router(d, 8, 60 + i).cuda(), ex, 2))
    nbytes = max(ses.layer_workspace_bytes(lay, B) for lay in layers for B in (1, 2))
    ws = ses.Workspace(nbytes)
    for rep in range(3):
        for li, lay in enumerate(layers):
            for B in (2, 1):
                assert ses.layer_path(lay, B) == ("decode_fused" if B == 1 else "decode")
                x = synth.tokens(B, lay.w_router.shape[0], 70 + 4 * rep + 2 * li + B).cuda()
                got = ses.layer_decode(x, lay, ws=ws, rmsnorm=(B == 1)).clone()
                fresh = ses.Workspace(ses.layer_workspace_bytes(lay, B))
                ref = ses.layer_decode(x, lay, ws=fresh, rmsnorm=(B == 1))
                assert _same_up_to_sum_order(got, ref), (rep, li, B)
                assert fresh.status() == 0
    assert ws.status() == 0


def test_layer_deterministic_and_status():
    d, f, E, k, B = 768, 208, 4, 2, 9
    de = synth.experts(E, d, f, 9)
    ex = ses.Experts.from_dense(de.w_up.cuda(), de.gate_t.cuda(), de.down.cuda(),
                                torch.full((E,), 0.2, dtype=torch.float32).cuda())
    layer = ses.Layer(synth.router(d, E, 9).cuda(), ex, k)
    x = synth.tokens(B, d, 9).cuda()
    ws = ses.Workspace(ses.layer_workspace_bytes(layer, B))
    y1 = ses.layer_decode(x, layer, ws=ws).clone()
    y2 = ses.layer_decode(x, layer, ws=ws)
    assert torch.equal(y1, y2)
    assert ws.status() == 0
