"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds no arithmetic of the GEMMs: it only draws random tensors.
The oracle and the CUDA path read the very same CPU tensors (copied to the GPU
for the latter), so neither side re-implements the generator.

Recipe: a CPU ``torch.Generator`` seeded with ``seed * 16 + role``; ``randn``
in FP32; multiplied by the scale; for BF16 operands rounded by ``.to(bfloat16)``.
Roles keep X, W and dY independent for one seed.

Workloads (shapes from the pages' tables):
  * dense projection  X[T,K], W[N,K] (scaled 1/sqrt(K)), dY[T,N]   bf16 N(0,1)
  * wide projection   4096 -> 12288, W scaled 1/64                  bf16 N(0,1)
  * thin-N wgrad      dY[T,N], X[T,K]                                bf16 N(0,1)
  * router            X[T,H] N(0,1), W[256,H] N(0, 0.02^2), dY[T,256] N(0,1), fp32
"""
from __future__ import annotations

import torch

ROLE_X, ROLE_W, ROLE_DY = 1, 2, 3

_CHUNK = 1 << 24  # draw in chunks so a 300M-element operand needs no 1 GB temporary


def _generator(seed: int, role: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 16 + int(role))
    return g


def normal(shape, seed: int, role: int, scale: float = 1.0, dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, scale^2) samples, drawn in FP32 then cast to ``dtype`` (CPU tensor)."""
    g = _generator(seed, role)
    numel = 1
    for s in shape:
        numel *= int(s)
    out = torch.empty(numel, dtype=dtype)
    for lo in range(0, numel, _CHUNK):
        hi = min(numel, lo + _CHUNK)
        v = torch.randn(hi - lo, generator=g, dtype=torch.float32)
        if scale != 1.0:
            v.mul_(scale)
        out[lo:hi] = v.to(dtype)
    return out.view(*shape)


def small_ints(shape, seed: int, role: int, lo: int = -3, hi: int = 3, dtype=torch.bfloat16) -> torch.Tensor:
    """Integers uniform in [lo, hi] (exact in bf16 and fp32), for brute-force cases."""
    g = _generator(seed, role)
    v = torch.randint(lo, hi + 1, tuple(int(s) for s in shape), generator=g, dtype=torch.int32)
    return v.to(dtype)


def dense_projection(T: int, N: int, K: int, seed: int, w_scale: float | None = None) -> dict:
    """X[T,K], W[N,K], dY[T,N] in bf16; W scaled 1/sqrt(K) unless ``w_scale`` is given."""
    if w_scale is None:
        w_scale = 1.0 / float(K) ** 0.5
    return {
        "X": normal((T, K), seed, ROLE_X),
        "W": normal((N, K), seed, ROLE_W, w_scale),
        "dY": normal((T, N), seed, ROLE_DY),
    }


def thin_wgrad(T: int, N: int, K: int, seed: int) -> dict:
    """dY[T,N] and X[T,K], bf16 N(0,1), for the bandwidth-bound weight gradient."""
    return {"dY": normal((T, N), seed, ROLE_DY), "X": normal((T, K), seed, ROLE_X)}


def router(T: int, K: int, seed: int, experts: int = 256, w_std: float = 0.02) -> dict:
    """FP32 router operands: X[T,K] N(0,1), W[experts,K] N(0, w_std^2), dY[T,experts] N(0,1)."""
    return {
        "X": normal((T, K), seed, ROLE_X, 1.0, torch.float32),
        "W": normal((experts, K), seed, ROLE_W, w_std, torch.float32),
        "dY": normal((T, experts), seed, ROLE_DY, 1.0, torch.float32),
    }


def integer_case(T: int, N: int, K: int, seed: int, lo: int = -3, hi: int = 3, dtype=torch.bfloat16) -> dict:
    """Small-integer X, W, dY: every product and partial sum is exact in FP32."""
    return {
        "X": small_ints((T, K), seed, ROLE_X, lo, hi, dtype),
        "W": small_ints((N, K), seed, ROLE_W, lo, hi, dtype),
        "dY": small_ints((T, N), seed, ROLE_DY, lo, hi, dtype),
    }
