"""fp64 CPU oracle of the decode-time MoE layer with FloE-style sparse SwiGLU experts.

TEST INFRASTRUCTURE ONLY (see the package docstring): imported by the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``, never by the
product path.  Plain numpy; every floating-point result is computed in fp64 from
the fp16 input bits, except the INT2 quantiser, whose fp32 arithmetic decides
integer codes and is therefore done in the same fp32 IEEE operations the kernel
uses.

Sources (page title, section):
  [FloE]  "FloE: On-the-Fly MoE Inference on Memory-constrained GPU" (xllm-io paper
          review): sec. 三 "MoE 专家前向计算" (the SwiGLU expert formula),
          "混合压缩策略" (gate/down sparsified, up projection INT2),
          "双稀疏预测器 / Intra-expert Predictor" (the reused up projection predicts
          the mask), "系统协同优化 / Algorithm 1: Efficient Sparse Kernel" and its
          optimisation list (transposed W^down, only selected columns loaded,
          SiLU fused with the elementwise product).
  [MoE-Lightning] "MoE-Lightning: High-Throughput MoE Inference on
          Memory-constrained GPUs", sec. 三 "MoE 模型架构" (a gating network picks
          the top-k experts of every token).
  [MoE-Infinity] "MOE-INFINITY: Efficient MoE Inference on Personal Machines with
          Sparsity-Aware Expert Cache", sec. A3 background (router per MoE layer;
          Mixtral-8x7B: 8 experts, 2 selected per token).

Where the pages are silent the plainest reading is taken; each such reading is
stated in the docstring of the function that makes it.
"""

from __future__ import annotations

import numpy as np

# Rows of W^up (input features) that share one INT2 scale and zero point.
GROUP = 64


def _f64(a) -> np.ndarray:
    return np.asarray(a).astype(np.float64)


def silu(a):
    """SiLU(a) = a / (1 + exp(-a)), fp64 ([FloE] sec. 三, expert formula)."""
    a = _f64(a)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


# ---------------------------------------------------------------------------
# INT2 up projection ([FloE] "混合压缩策略": W^up is stored quantised, Q(.))
# ---------------------------------------------------------------------------

def quantize_int2(w_up):
    """Quantise W^up [d, f] (fp16) to 2-bit codes with one fp16 (scale, zero) per
    (64-row group, column).

    The pages name the scheme only as INT2 Q(.) of the up projection.  Reading
    (asymmetric min/max per group, fp16 scale and zero point), per group G and
    column j, every operation in fp32 with IEEE round-to-nearest-even:
        scale = fp16( (max_G w - min_G w) / 3 );  if that fp16 is 0, scale = 1
        zero  = fp16( clamp(-min_G w / scale, -65504, 65504) )
        q     = clamp( rint( w / scale + zero ), 0, 3 )      (rint: half to even)
    and the dequantised weight is scale * (q - zero), exact in fp64.

    Returns (q uint8 [d, f], scale fp16 [d/64, f], zero fp16 [d/64, f]).
    """
    w = np.asarray(w_up)
    if w.dtype != np.float16 or w.ndim != 2:
        raise TypeError("w_up must be a 2-D float16 array")
    d, f = w.shape
    if d % GROUP:
        raise ValueError("d must be a multiple of 64")
    if not np.all(np.isfinite(w)):
        raise ValueError("w_up must be finite")
    wg = w.astype(np.float32).reshape(d // GROUP, GROUP, f)
    w_max = wg.max(axis=1)
    w_min = wg.min(axis=1)
    scale = ((w_max - w_min) / np.float32(3.0)).astype(np.float16)
    scale[scale == 0] = np.float16(1.0)
    scale32 = scale.astype(np.float32)
    zero32 = np.clip(-w_min / scale32, np.float32(-65504.0), np.float32(65504.0))
    zero = zero32.astype(np.float16)
    t = wg / scale32[:, None, :] + zero.astype(np.float32)[:, None, :]
    q = np.clip(np.rint(t), 0, 3).astype(np.uint8).reshape(d, f)
    return q, scale, zero


def dequantize_int2(q, scale, zero):
    """W~^up[k, j] = scale[k // 64, j] * (q[k, j] - zero[k // 64, j]), fp64 (exact)."""
    s = np.repeat(_f64(scale), GROUP, axis=0)
    z = np.repeat(_f64(zero), GROUP, axis=0)
    return s * (_f64(q) - z)


# ---------------------------------------------------------------------------
# Router ([MoE-Lightning] sec. 三; [MoE-Infinity] A3 background)
# ---------------------------------------------------------------------------

def route_topk(x, w_router, k, renorm=True):
    """Softmax top-k routing of every token.

    logits = x . W_r   (x [B, d] fp16, W_r [d, E] fp16; fp64 arithmetic)
    Readings where the pages are silent:
      * the k largest logits are chosen; equal logits go to the lower expert index;
        the k experts are listed by logit descending (ties: lower index first);
      * renorm=True: the weights are the softmax over the k chosen logits;
        renorm=False: the weights are the full softmax over all E experts,
        read at the chosen ones.

    Returns (idx int32 [B, k], w fp64 [B, k], logits fp64 [B, E]).
    """
    xs = _f64(x)
    wr = _f64(w_router)
    logits = xs @ wr
    B, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    idx = np.empty((B, k), dtype=np.int32)
    w = np.empty((B, k), dtype=np.float64)
    for b in range(B):
        order = np.lexsort((np.arange(E), -logits[b]))  # key 1: -logit, key 2: index
        sel = order[:k]
        idx[b] = sel
        lsel = logits[b, sel] if renorm else logits[b]
        p = np.exp(lsel - lsel.max())
        p /= p.sum()
        w[b] = p if renorm else p[sel]
    return idx, w, logits


# ---------------------------------------------------------------------------
# Sparse SwiGLU expert ([FloE] Algorithm 1 "Efficient Sparse Kernel")
# ---------------------------------------------------------------------------

def expert_up(x, w_up_deq):
    """Step 1 of Algorithm 1 (also the intra-expert predictor): v = x . W~^up."""
    return _f64(x) @ _f64(w_up_deq)


def sparse_swiglu_expert(x, w_gate, w_up_deq, w_down, t, mask=None):
    """One expert, Algorithm 1 of [FloE] taken step by step:

      1: v      = x W^up
      2: mask   = |v| > t                       (strict; NaN is dropped)
      3: x'     = SiLU(x W^gate[:, mask]) (.) v[mask]
      4: output = x' W^down[mask, :]

    x [n, d]; w_gate [d, f]; w_up_deq [d, f] (dequantised INT2); w_down [f, d]:
    row i of W^down is the d-vector that intermediate column i multiplies (the
    "transposed, column-major W^down" of the kernel's optimisation list).  With
    t = 0 this is the dense SwiGLU expert (SiLU(xW^gate) (.) xW^up) W^down of
    sec. 三 except for columns with v exactly 0, which contribute 0 either way.

    ``mask`` (bool [n, f]) replaces step 2 when given; the parity tests use it to
    substitute the kernel's choice for columns inside the rounding band.
    Returns (y fp64 [n, d], v fp64 [n, f], mask bool [n, f]).
    """
    xs = _f64(x)
    n = xs.shape[0]
    d = xs.shape[1]
    v = xs @ _f64(w_up_deq)                       # step 1
    if mask is None:
        mask = np.abs(v) > t                      # step 2
    mask = np.asarray(mask, dtype=bool)
    y = np.zeros((n, d), dtype=np.float64)
    for b in range(n):
        kept = np.flatnonzero(mask[b])
        if kept.size == 0:
            continue
        g = xs[b] @ _f64(w_gate[:, kept])         # gate only over kept columns
        h = silu(g) * v[b, kept]                  # step 3
        y[b] = h @ _f64(w_down[kept, :])          # step 4: kept rows of W^down
    return y, v, mask


def quantile_threshold(v, pct):
    """Per-expert threshold t_ij of Algorithm 1 (one scalar per layer i, expert j).

    The pages do not say how t_ij is calibrated.  Reading: the nearest-rank
    pct-quantile of |v| pooled over all (calibration token, column) pairs of the
    expert: t = sorted(|v|)[ceil(pct * n / 100) - 1]; pct = 0 gives t = 0 exactly,
    so that 0 % sparsity is the dense expert by definition.  pct is an integer
    percentage in [0, 100].
    """
    pct = int(pct)
    if not 0 <= pct <= 100:
        raise ValueError("pct must be in [0, 100]")
    if pct == 0:
        return 0.0
    a = np.sort(np.abs(_f64(v)).ravel())
    r = (pct * a.size + 99) // 100
    return float(a[r - 1])


def rmsnorm(y, eps=1e-6):
    """RMSNorm between stacked layers (not on the pages; unit weight, eps 1e-6):
    y / sqrt(mean(y^2) + eps) along the hidden dimension, fp64."""
    ys = _f64(y)
    return ys / np.sqrt(np.mean(ys * ys, axis=-1, keepdims=True) + eps)


# ---------------------------------------------------------------------------
# One MoE decode layer
# ---------------------------------------------------------------------------

def _up_deq(ex):
    if "w_up_deq" in ex:
        return ex["w_up_deq"]
    return dequantize_int2(ex["q"], ex["scale"], ex["zero"])


def moe_layer(x, w_router, experts, k, renorm=True, shared=(), rmsnorm_out=False,
              route=None, masks=None):
    """One decode MoE layer: y_b = sum_j w_bj E_{idx_bj}(x_b) + sum_s E_s(x_b).

    The weighted sum of the selected experts' outputs is the plain reading of the
    router description ([MoE-Lightning] sec. 三); shared experts (not on the
    pages) are always on with weight 1 and their own thresholds.  With
    ``rmsnorm_out`` the result is passed through ``rmsnorm``.

    experts / shared: sequences of dicts with keys w_gate [d, f], w_down [f, d],
    thr (float), and either w_up_deq [d, f] or (q, scale, zero).
    route: optional (idx, w) that replaces the router's choice (band cases).
    masks: optional dict {("r", e) or ("s", s): bool [n_e, f]} replacing step 2
    for the tokens of that expert, in ascending token order.

    Returns (y fp64 [B, d], info dict with idx, w, logits, and per-expert
    tokens / v / mask).
    """
    xs = np.asarray(x)
    B, d = xs.shape
    if route is None:
        idx, w, logits = route_topk(xs, w_router, k, renorm)
    else:
        idx, w = (np.asarray(route[0]), _f64(route[1]))
        logits = None
    masks = masks or {}
    y = np.zeros((B, d), dtype=np.float64)
    per_expert = {}
    for e in range(len(experts)):
        rows, cols = np.nonzero(idx == e)
        if rows.size == 0:
            continue
        order = np.argsort(rows, kind="stable")
        toks, slots = rows[order], cols[order]
        ex = experts[e]
        ye, v, m = sparse_swiglu_expert(xs[toks], ex["w_gate"], _up_deq(ex), ex["w_down"],
                                        ex["thr"], mask=masks.get(("r", e)))
        y[toks] += w[toks, slots][:, None] * ye
        per_expert[("r", e)] = dict(tokens=toks, v=v, mask=m)
    for s, ex in enumerate(shared):
        ye, v, m = sparse_swiglu_expert(xs, ex["w_gate"], _up_deq(ex), ex["w_down"],
                                        ex["thr"], mask=masks.get(("s", s)))
        y += ye
        per_expert[("s", s)] = dict(tokens=np.arange(B), v=v, mask=m)
    if rmsnorm_out:
        y = rmsnorm(y)
    return y, dict(idx=idx, w=w, logits=logits, experts=per_expert)
