"""Comparison rules between the CUDA path and the fp64 oracle.

Integer decisions taken from floating point (the router's top-k, the mask |v| > t)
must agree exactly unless the exact value lies within the fp32 rounding band of
the decision boundary; inside the band either answer is accepted, counted, and
the oracle is re-run with the kernel's choice so that the outputs can be compared.

Band half-width: TAU * S, where S is the magnitude sum of the terms that the
kernel adds in fp32.  For v = x . s (q - z) the kernel forms, per 64-row group g,
A_g = sum q x (tensor cores, fp32 accumulate) and X_g = sum x, then
s * (A_g - z X_g), so S = sum_k |x_k| |s| (q_k + |z|).  The kernel's
accumulation chains are at most ~32 mma k-steps, 64-term group sums of x and
d/512 + 3 superblock / lane additions, i.e. n < 128 rounding steps of 2^-24:
|v_gpu - v| <= 128 * 2^-24 * S = 2^-17 S.  TAU = 2^-16 keeps a factor-2 margin.
"""

from __future__ import annotations

import numpy as np

TAU = 2.0 ** -16
Y_MAX_ABS = 2e-2
Y_REL_L2 = 5e-3


def up_magnitude(x, q, scale, zero):
    """S_j = sum_k |x_k| |s_gj| (q_kj + |z_gj|) for x [n, d] -> [n, f] (fp64)."""
    sg = np.repeat(np.abs(scale.astype(np.float64)), 64, axis=0)
    zg = np.repeat(np.abs(zero.astype(np.float64)), 64, axis=0)
    return np.abs(x.astype(np.float64)) @ (sg * (q.astype(np.float64) + zg))


def unpack_mask(words, f):
    """int32 [..., ceil(f/32)] bit words -> bool [..., f]."""
    w = np.asarray(words).astype(np.uint32)
    bits = (w[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1
    return bits.reshape(*w.shape[:-1], -1)[..., :f].astype(bool)


def check_mask(mask_gpu, v_ref, S, t):
    """-> (#mismatches outside the band, #decisions inside the band)."""
    ref = np.abs(v_ref) > t
    band = np.abs(np.abs(v_ref) - t) <= TAU * S
    return int(((mask_gpu != ref) & ~band).sum()), int(band.sum())


def mask_excused(mask_gpu, v_ref, S, t):
    """#decisions the band excuses: inside it, and the kernel's differs from the oracle's."""
    ref = np.abs(v_ref) > t
    band = np.abs(np.abs(v_ref) - t) <= TAU * S
    return int(((mask_gpu != ref) & band).sum())


def check_v(v_gpu, v_ref, S):
    """Largest |v_gpu - v| / S (must stay below TAU for the band rule to hold)."""
    return float(np.max(np.abs(v_gpu.astype(np.float64) - v_ref) / np.maximum(S, 1e-300)))


def route_band(logits, S, idx_gpu, k):
    """Top-k parity: outside the band the kernel's ordered choice equals the oracle's.
    -> (ok, n_band_tokens).  Near-ties (gap <= TAU * (S_a + S_b)) between any two
    experts whose order decides the output are treated as band cases, in which the
    kernel's choice must still be a valid top-k of the exact logits up to the band."""
    B, E = logits.shape
    n_band = 0
    for b in range(B):
        order = np.lexsort((np.arange(E), -logits[b]))
        ref = order[:k]
        got = np.asarray(idx_gpu[b])
        if list(ref) == list(got):
            continue
        # band: every swapped pair must be a near tie
        thr = logits[b, order[k - 1]]
        tol = TAU * 2 * S[b].max()
        if len(set(got)) != k:
            return False, n_band
        sel_ok = all(logits[b, e] >= thr - tol for e in got)
        ord_ok = all(logits[b, got[i]] >= logits[b, got[i + 1]] - tol for i in range(k - 1))
        if not (sel_ok and ord_ok):
            return False, n_band
        n_band += 1
    return True, n_band


def check_y(y_gpu, y_ref):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    diff = np.abs(y_gpu - y_ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    denom = float(np.linalg.norm(y_ref))
    rel = float(np.linalg.norm(y_gpu - y_ref) / denom) if denom > 0 else float(np.linalg.norm(y_gpu))
    return max_abs, rel
