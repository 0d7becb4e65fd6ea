"""Oracle of the expert activation tracking and the sparsity-aware expert cache.

TEST INFRASTRUCTURE ONLY: imported by the tests, never by the product path.  Plain
Python over integer counts; the floating-point steps are the same IEEE double
operations, in the same order, that the definitions below state, so that every
distance, likelihood and priority is reproducible bit for bit.

Source: "MOE-INFINITY: Efficient MoE Inference on Personal Machines with Sparsity-Aware
Expert Cache":
  sec. 4.3 "解码过程中激活预测的形式化" -- the expert activation matrix (EAM): L x E,
      cell [i][j] = tokens routed to expert j of MoE layer i; the iteration EAM (iEAM)
      and the request EAM (rEAM, the running sum of the iterations' iEAMs);
  sec. 4.5 "请求级稀疏激活追踪" -- the EAM collection (EAMC); matching by the cosine
      distance of the flattened matrices, the nearest being the match; PredictEAM:
      the matched EAMs summed cell by cell, each row normalised, each cell scaled by
      1 - (i - l)/L (l the current layer, i the cell's layer);
  sec. 4.7, Algorithm 1 "专家缓存检索" -- hit, cold fill, and on a full cache eviction of
      the cached expert with the lowest (p_eam[layer][expert] + eps) / n_token *
      (1 - layer / L), n_token = the sum of p_eam's row for that layer;
  appendix B.1 "预测器运行时效率" -- a fixed-capacity EAMC that, when full, replaces the
      stored EAM most similar to (nearest to) the new one.

Readings where the pages are silent:
  * the cosine distance of an all-zero matrix to anything is 1 (no direction);
  * "possibly several matched EAMs": the n_match nearest, ties to the lower index;
  * a row of the summed matches that sums to 0 stays 0 (nothing to normalise);
  * the proximity factor 1 - (i - l)/L applies to every row, as the pages state it for
    every cell (rows before l get factors above 1);
  * n_token = 0 (the evicted expert's layer has no prediction): divide by 1;
  * eps is a caller parameter; ties in the eviction priority go to the expert
    inserted earliest (the first minimum in insertion order, as the algorithm's
    strict comparison over the cache in insertion order gives).
"""

from __future__ import annotations

import math
from typing import List, Optional, Sequence, Tuple

import numpy as np


def cosine_distance(a: np.ndarray, b: np.ndarray) -> float:
    """1 - a.b / (|a| |b|) of two flattened EAMs (sec. 4.5); the integer sums are exact."""
    x = [int(v) for v in np.asarray(a).ravel()]
    y = [int(v) for v in np.asarray(b).ravel()]
    ab = sum(p * q for p, q in zip(x, y))
    aa = sum(p * p for p in x)
    bb = sum(q * q for q in y)
    if aa == 0 or bb == 0:
        return 1.0
    return 1.0 - float(ab) / (math.sqrt(float(aa)) * math.sqrt(float(bb)))


def nearest(entries: Sequence[np.ndarray], cur: np.ndarray, n: int) -> Tuple[List[int], List[float]]:
    """The n entries nearest to cur, by (distance, index) ascending (sec. 4.5)."""
    d = [cosine_distance(cur, e) for e in entries]
    order = sorted(range(len(entries)), key=lambda i: (d[i], i))[:n]
    return order, [d[i] for i in order]


def add_counts(eam: np.ndarray, layer: int, counts) -> None:
    """rEAM accumulation (sec. 4.3): row `layer` gains this iteration's token counts."""
    eam[layer] += np.asarray(counts, dtype=eam.dtype)


class Eamc:
    """The EAM collection with the replacement of appendix B.1."""

    def __init__(self, L: int, E: int, capacity: int):
        self.L, self.E, self.capacity = L, E, capacity
        self.entries: List[np.ndarray] = []

    def insert(self, ream: np.ndarray) -> int:
        ream = np.array(ream, dtype=np.int64)
        if len(self.entries) < self.capacity:
            self.entries.append(ream)
            return len(self.entries) - 1
        (slot,), _ = nearest(self.entries, ream, 1)
        self.entries[slot] = ream
        return slot


def predict(eamc: Eamc, cur: np.ndarray, layer: int, n_match: int) -> np.ndarray:
    """PredictEAM (sec. 4.5): sum the n_match nearest EAMs, normalise every row, scale
    row i by 1 - (i - layer)/L."""
    L, E = eamc.L, eamc.E
    idx, _ = nearest(eamc.entries, cur, n_match)
    p = np.zeros((L, E), dtype=np.float64)
    for i in range(L):
        cells = [sum(int(eamc.entries[t][i][j]) for t in idx) for j in range(E)]
        rs = sum(cells)
        scale = 1.0 - float(i - layer) / float(L)
        for j in range(E):
            p[i][j] = float(cells[j]) / float(rs) * scale if rs > 0 else 0.0
    return p


class ExpertCache:
    """Algorithm 1 (sec. 4.7): (layer, expert) ids in insertion order."""

    def __init__(self, capacity: int, L: int, E: int):
        self.capacity, self.L, self.E = capacity, L, E
        self.items: List[Tuple[int, int]] = []

    def lookup(self, eamc: Eamc, cur: np.ndarray, layer: int, expert: int, n_match: int,
               eps: float) -> Tuple[bool, Optional[Tuple[int, int]]]:
        key = (layer, expert)
        if key in self.items:                      # steps 1-3: hit
            return True, None
        if len(self.items) < self.capacity:        # steps 4-7: room left
            self.items.append(key)
            return False, None
        p = predict(eamc, cur, layer, n_match)     # step 8
        victim, p_min = None, math.inf             # steps 9-16
        for (li, ej) in self.items:
            n_token = 0.0
            for j in range(self.E):
                n_token += p[li][j]
            if n_token == 0.0:
                n_token = 1.0
            pr = (p[li][ej] + eps) / n_token * (1.0 - float(li) / float(self.L))
            if pr < p_min:
                p_min, victim = pr, (li, ej)
        self.items.remove(victim)                  # steps 17-19
        self.items.append(key)
        return False, victim
