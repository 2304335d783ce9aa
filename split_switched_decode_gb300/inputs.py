"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

Holds none of the method's arithmetic: only seeded random draws in the shapes and
distributions of the decode workloads (activations ~ N(0,1), weights ~ N(0, 0.02^2),
residual ~ N(0,1), all bfloat16). Every tensor has its own generator seeded from
(seed, workload, tensor name[, expert]) through a stable hash, so one expert of a
weight bank can be regenerated or checked alone.
"""
from __future__ import annotations

import zlib

import torch

WEIGHT_STD = 0.02


def seed_of(seed: int, *parts) -> int:
    key = "/".join([str(seed)] + [str(p) for p in parts]).encode()
    return zlib.crc32(key) & 0x7FFFFFFF


def _gen(device, seed: int, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed_of(seed, *parts))
    return g


def randn_bf16(shape, std: float, device, seed: int, *parts) -> torch.Tensor:
    g = _gen(device, seed, *parts)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def activations(B: int, K: int, device, seed: int = 0, name: str = "x") -> torch.Tensor:
    return randn_bf16((B, K), 1.0, device, seed, name, B, K)


def weight(N: int, K: int, device, seed: int = 0, name: str = "w") -> torch.Tensor:
    return randn_bf16((N, K), WEIGHT_STD, device, seed, name, N, K)


def residual(B: int, N: int, device, seed: int = 0, name: str = "r") -> torch.Tensor:
    return randn_bf16((B, N), 1.0, device, seed, name, B, N)


def expert_bank(E: int, H: int, I: int, device, seed: int = 0, name: str = "experts"):
    """Wgu [E, 2I, H] and Wd [E, H, I], expert e drawn from its own generator."""
    Wgu = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=device)
    Wd = torch.empty((E, H, I), dtype=torch.bfloat16, device=device)
    for e in range(E):
        Wgu[e] = randn_bf16((2 * I, H), WEIGHT_STD, device, seed, name, "gu", e, H, I)
        Wd[e] = randn_bf16((H, I), WEIGHT_STD, device, seed, name, "d", e, H, I)
    return Wgu, Wd


def shared_expert(H: int, I: int, device, seed: int = 0, name: str = "shared"):
    return (randn_bf16((2 * I, H), WEIGHT_STD, device, seed, name, "gu", H, I),
            randn_bf16((H, I), WEIGHT_STD, device, seed, name, "d", H, I))


def bits(t: torch.Tensor):
    """Raw bf16 bit patterns as a numpy uint16 array on the host (for the oracle)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")
