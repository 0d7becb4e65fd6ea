"""Seeded synthetic inputs for the tests, the benchmark and the CPU oracle checks.

Only draws from torch generators and dtype casts live here: none of the method's
arithmetic.  Every tensor is identified by (seed, stream id); the same call on the
same device gives the same bits.  Workloads (sizes from the model shapes the
benchmarks are quoted on; weights are random, no checkpoint is involved):

  tokens x ~ N(0, 1) in fp16 (their RMS is 1 up to O(1/sqrt(d)) sampling noise)
  W^gate, W^up, W^down, W_router ~ N(0, 0.02) in fp16
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

WEIGHT_STD = 0.02

# stream ids
_TOKENS, _CALIB, _ROUTER, _UP, _GATE, _DOWN = 1, 2, 3, 4, 5, 6


def _generator(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(stream)) % (2 ** 63 - 1))
    return g


def normal_f16(shape, std: float, seed: int, stream: int, device="cpu") -> torch.Tensor:
    g = _generator(seed, stream, device)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.float16)


def tokens(B: int, d: int, seed: int, device="cpu", stream: int = _TOKENS) -> torch.Tensor:
    """Decode tokens x fp16 [B, d] ~ N(0, 1)."""
    return normal_f16((B, d), 1.0, seed, stream, device)


def calibration_tokens(n: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    """Calibration tokens fp16 [n, d] ~ N(0, 1), a stream separate from the decode tokens."""
    return normal_f16((n, d), 1.0, seed, _CALIB, device)


def router(d: int, E: int, seed: int, device="cpu", layer: int = 0) -> torch.Tensor:
    """W_router fp16 [d, E] ~ N(0, 0.02)."""
    return normal_f16((d, E), WEIGHT_STD, seed, _ROUTER + 100 * layer, device)


@dataclass
class DenseExperts:
    """fp16 weights of E experts: w_up [E, d, f]; gate_t, down [E, f, d]."""
    w_up: torch.Tensor
    gate_t: torch.Tensor
    down: torch.Tensor


def experts(E: int, d: int, f: int, seed: int, device="cpu", layer: int = 0,
            kind: int = 0) -> DenseExperts:
    """E experts ~ N(0, 0.02); kind 0 = routed, 1 = shared (independent streams)."""
    base = 1000 * (1 + layer) + 500 * kind
    w_up = torch.empty((E, d, f), dtype=torch.float16, device=device)
    gate_t = torch.empty((E, f, d), dtype=torch.float16, device=device)
    down = torch.empty((E, f, d), dtype=torch.float16, device=device)
    for e in range(E):
        w_up[e] = normal_f16((d, f), WEIGHT_STD, seed, base + 10 * e + _UP, device)
        gate_t[e] = normal_f16((f, d), WEIGHT_STD, seed, base + 10 * e + _GATE, device)
        down[e] = normal_f16((f, d), WEIGHT_STD, seed, base + 10 * e + _DOWN, device)
    return DenseExperts(w_up, gate_t, down)
