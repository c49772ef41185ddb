"""Seeded synthetic inputs for the W8A8 FP8 block-scaled linear layer.

This module only draws random numbers; it holds none of the method's
arithmetic (no scaling, no quantisation, no GEMM).  Both the CUDA path and the
CPU oracle are fed from it.

Recipe (all on the CPU with ``torch.Generator('cpu').manual_seed``; values are
drawn in fp32 and rounded to bf16 with round-to-nearest-even):

* activations ``x`` use ``seed``; weights ``W`` use ``seed + 1``;
* ``normal``: x ~ N(0, 1);  ``laplace``: x ~ Laplace(0, 1) by the inverse CDF
  of seeded uniforms;  ``outliers``: N(0, 1), then round(frac * K) channels
  chosen by ``randperm(K)`` are multiplied by ``outlier_gain``;
* weights: W ~ N(0, 0.02).

The shapes stand in for the DeepSeek-V4.1-Flash dense linears of sglang PR
#42604 "[SM90] Use native block32 DeepGEMM for DeepSeek-V4.1" (Motivation and
the fixed 16k-in / 1k-out serving workload); no model weights are used.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def activation(M: int, K: int, seed: int = 0, dist: str = "normal",
               outlier_frac: float = 0.0, outlier_gain: float = 50.0) -> torch.Tensor:
    """bf16 [M, K] on the CPU."""
    g = torch.Generator("cpu").manual_seed(seed)
    if dist == "normal":
        x = torch.randn(M, K, generator=g, dtype=torch.float32)
    elif dist == "laplace":
        u = torch.rand(M, K, generator=g, dtype=torch.float32) - 0.5
        x = -torch.sign(u) * torch.log1p(-2.0 * u.abs())
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * K))
        ch = torch.randperm(K, generator=g)[:n_out]
        x[:, ch] *= outlier_gain
    return x.to(torch.bfloat16)


def weight(N: int, K: int, seed: int = 0, std: float = 0.02) -> torch.Tensor:
    """bf16 [N, K] on the CPU, drawn with ``seed + 1``."""
    g = torch.Generator("cpu").manual_seed(seed + 1)
    return (torch.randn(N, K, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


@dataclass(frozen=True)
class Case:
    """One GEMM problem of a workload."""
    name: str
    M: int
    N: int
    K: int
    blk_n: int
    blk_k: int
    ue8m0: bool
    dist: str = "normal"
    outlier_frac: float = 0.0
    seed: int = 0

    @property
    def group(self) -> int:
        return self.blk_k

    def x(self) -> torch.Tensor:
        return activation(self.M, self.K, self.seed, self.dist, self.outlier_frac)

    def w(self) -> torch.Tensor:
        return weight(self.N, self.K, self.seed)

    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def gemm_bytes(self, scale_bytes: int = 4) -> float:
        """Algorithmic GEMM bytes: Aq + As + Wq + Ws + D (scale_bytes per
        scale: 4 for fp32, 1 for UE8M0 bytes)."""
        M, N, K = self.M, self.N, self.K
        return (M * K + scale_bytes * M * K / self.blk_k + N * K
                + scale_bytes * math.ceil(N / self.blk_n) * K / self.blk_k + 2 * M * N)

    def quant_bytes(self, scale_bytes: int = 4) -> float:
        """Algorithmic quant bytes: bf16 read + codes + scales written."""
        M, K = self.M, self.K
        return 2 * M * K + M * K + scale_bytes * M * K / self.group


def _cases() -> dict:
    c = {}
    c["tiny"] = [Case("tiny", 16, 256, 512, 128, 128, False)]
    c["decode_block32"] = [Case(f"decode_block32_M{m}", m, 7168, 2048, 32, 32, True)
                           for m in (1, 4, 16, 64)]
    c["prefill_block128"] = [Case("prefill_block128", 4096, 7168, 7168, 128, 128, True,
                                  "normal", 0.001)]
    c["prefill_block32"] = [Case("prefill_block32", 4096, 4096, 7168, 32, 32, True,
                                 "laplace")]
    sweep = []
    for (N, K) in ((24576, 1536), (1536, 7168)):
        for blk in (128, 32):
            for m in (1, 2, 4, 8, 32, 128, 512, 2048, 8192):
                sweep.append(Case(f"sweep_N{N}_K{K}_b{blk}_M{m}", m, N, K, blk, blk, True))
    c["sweep"] = sweep
    return c


WORKLOADS = _cases()
