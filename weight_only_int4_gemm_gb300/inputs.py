"""Seeded synthetic inputs for the W4A16 linear layer.

This module only draws random numbers; it holds none of the layer's
arithmetic (no unpacking, dequantisation or products), so the CPU oracle and
the CUDA library can both be fed from it without sharing any of the method.

Recipe (shapes and value distributions of the workloads):
  * codes    -- canonical ``qweight`` uint32 [K/8][N]: uniform random 32-bit
                words, i.e. eight independent uniform codes 0..15 per word;
  * scales   -- bf16 [K/128][N]: |N(0, 1)| * 0.02, rounded to bf16;
  * zeros    -- canonical ``qzeros`` uint32 [K/128][N/8]: uniform random
                words, i.e. uniform zero-points 0..15 (asymmetric variant);
  * x        -- bf16 [B][K]: N(0, 1) rounded to bf16; with ``outlier_frac``,
                round(outlier_frac * K) input channels picked without
                replacement are multiplied by 20 before the rounding;
  * routing  -- mixture-of-experts layers: every token picks k distinct
                experts of E uniformly at random (the uniform-routing
                assumption of the pages' effective-M estimate); the routed
                rows are grouped by expert, giving per-expert row offsets;
                expert e's weights are drawn like one layer's, seed + e;
  * dense    -- bf16 weights W [K][N] for the quantisers and the FP8
                comparison path: N(0, 1) * 0.02 rounded to bf16;
  * bias     -- bf16 [N]: N(0, 1) * 0.5 rounded to bf16;
  * fp16     -- the fp16-activation variant draws x and the scales the same
                way and rounds them to fp16 instead (``dtype=torch.float16``).

Draws use ``torch.Generator(device).manual_seed(seed)``; CPU and CUDA
generators give different streams, so each comparison uses one generated copy
(moved between devices as needed), never two independent draws.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

GROUP = 128


@dataclass
class LinearProblem:
    x: torch.Tensor          # bf16 [B][K]
    qweight: torch.Tensor    # int32 [K/8][N]   (bit pattern of uint32 words)
    scales: torch.Tensor     # bf16 [K/128][N]
    qzeros: torch.Tensor | None  # int32 [K/128][N/8] or None (symmetric)

    @property
    def shape(self):
        B, K = self.x.shape
        return B, K, self.qweight.shape[1]

    def to(self, device) -> "LinearProblem":
        return LinearProblem(
            self.x.to(device), self.qweight.to(device), self.scales.to(device),
            None if self.qzeros is None else self.qzeros.to(device))


def random_words(shape, gen: torch.Generator, device) -> torch.Tensor:
    """Uniform random 32-bit words (int32 storage)."""
    return torch.randint(-2**31, 2**31, shape, dtype=torch.int32, generator=gen, device=device)


def make_weights(K: int, N: int, seed: int, *, zero_points: bool = False, device="cpu",
                 dtype=torch.bfloat16):
    """(qweight, scales, qzeros-or-None) for one K x N layer."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    qweight = random_words((K // 8, N), gen, device)
    scales = (torch.randn((K // GROUP, N), generator=gen, device=device).abs_() * 0.02).to(dtype)
    qzeros = random_words((K // GROUP, N // 8), gen, device) if zero_points else None
    return qweight, scales, qzeros


def make_activations(B: int, K: int, seed: int, *, outlier_frac: float = 0.0, device="cpu",
                     dtype=torch.bfloat16):
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = torch.randn((B, K), generator=gen, device=device)
    n_out = int(round(outlier_frac * K))
    if n_out > 0:
        channels = torch.randperm(K, generator=gen, device=device)[:n_out]
        x[:, channels] *= 20.0
    return x.to(dtype)


def make_problem(B: int, K: int, N: int, seed: int, *, zero_points: bool = False,
                 outlier_frac: float = 0.0, device="cpu", dtype=torch.bfloat16) -> LinearProblem:
    """One seeded layer: weights from ``seed``, activations from ``seed + 1``
    (x and scales in ``dtype``: bf16, or fp16 for the fp16 variant)."""
    qweight, scales, qzeros = make_weights(K, N, seed, zero_points=zero_points, device=device,
                                           dtype=dtype)
    x = make_activations(B, K, seed + 1_000_003, outlier_frac=outlier_frac, device=device,
                         dtype=dtype)
    return LinearProblem(x, qweight, scales, qzeros)


def make_routing(tokens: int, E: int, k: int, seed: int) -> torch.Tensor:
    """Row offsets int32 [E+1] of ``tokens * k`` routed rows grouped by expert:
    each token picks k distinct experts uniformly at random."""
    gen = torch.Generator()
    gen.manual_seed(seed)
    picks = torch.rand((tokens, E), generator=gen).argsort(dim=1)[:, :k]
    counts = torch.bincount(picks.reshape(-1), minlength=E)
    offsets = torch.zeros(E + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(counts, 0)
    return offsets.to(torch.int32)


def offsets_from_counts(counts) -> torch.Tensor:
    """Row offsets int32 [E+1] for explicit per-expert row counts."""
    c = torch.as_tensor(counts, dtype=torch.int64)
    offsets = torch.zeros(c.numel() + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(c, 0)
    return offsets.to(torch.int32)


@dataclass
class GroupedProblem:
    x: torch.Tensor          # bf16 [T][K], rows grouped by expert
    offsets: torch.Tensor    # int32 [E+1]
    qweight: torch.Tensor    # int32 [E][K/8][N]
    scales: torch.Tensor     # bf16 [E][K/128][N]
    qzeros: torch.Tensor | None  # int32 [E][K/128][N/8] or None

    def to(self, device) -> "GroupedProblem":
        return GroupedProblem(
            self.x.to(device), self.offsets.to(device), self.qweight.to(device),
            self.scales.to(device), None if self.qzeros is None else self.qzeros.to(device))


def make_grouped_problem(offsets: torch.Tensor, K: int, N: int, seed: int, *,
                         zero_points: bool = False, device="cpu") -> GroupedProblem:
    """E experts' weights (expert e from seed + e) and T = offsets[-1] rows of x."""
    E = offsets.numel() - 1
    T = int(offsets[-1])
    ws = [make_weights(K, N, seed + e, zero_points=zero_points, device=device) for e in range(E)]
    qweight = torch.stack([w[0] for w in ws])
    scales = torch.stack([w[1] for w in ws])
    qzeros = torch.stack([w[2] for w in ws]) if zero_points else None
    x = make_activations(T, K, seed + 1_000_003, device=device)
    return GroupedProblem(x, offsets.to(device), qweight, scales, qzeros)


def make_dense_weight(K: int, N: int, seed: int, *, device="cpu") -> torch.Tensor:
    """bf16 W [K][N], N(0, 1) * 0.02."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return (torch.randn((K, N), generator=gen, device=device) * 0.02).to(torch.bfloat16)


def make_bias(N: int, seed: int, *, device="cpu") -> torch.Tensor:
    """bf16 bias [N], N(0, 1) * 0.5."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return (torch.randn(N, generator=gen, device=device) * 0.5).to(torch.bfloat16)
