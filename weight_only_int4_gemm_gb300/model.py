"""Roofline and decode-step arithmetic for the W4A16 linear layer.

Two pieces:

* the per-linear algorithmic traffic and work used for every roofline figure
  the benchmark prints: bytes = K*N/2 (codes) + (K/128)*N*2 (bf16 scales)
  [+ (K/128)*N/2 (4-bit zero-points)] + B*K*2 (bf16 x) + B*N*2 (bf16 y);
  flops = 2*B*K*N (the dequantisation is not counted as flops);

* the two-term decode-step model of "When quantization pays -- and when it does
  not" (sections "Model one decode step ..." and "The three regimes"): a memory
  pipe and a math pipe that overlap,
      t(B) = max(W * b_w / beta,  2*W*B / P + W*c / D),
  with W streamed weights, b_w bytes per stored weight, beta the HBM bandwidth,
  P the tensor-core peak, c the non-tensor instruction slots spent per weight on
  the dequantisation and D the non-tensor issue rate.  The equation itself was
  lost from the page's text; this form is the one its definitions and every
  number it prints agree with (checked in the tests).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

GROUP = 128
BYTES_PER_WEIGHT_SYM = 0.515625      # 4 bits + one bf16 scale per 128 weights
BYTES_PER_WEIGHT_ZP = 0.51953125     # ... + one 4-bit zero-point per 128 weights


def linear_bytes(B: int, K: int, N: int, zero_points: bool = False) -> int:
    groups = K // GROUP
    b = K * N // 2 + groups * N * 2 + B * K * 2 + B * N * 2
    if zero_points:
        b += groups * N // 2
    return b


def linear_flops(B: int, K: int, N: int) -> int:
    return 2 * B * K * N


def roofline_time(B: int, K: int, N: int, hbm_bytes_per_s: float, flops_per_s: float,
                  zero_points: bool = False) -> float:
    """max(bytes / beta, flops / P): the time no kernel can beat."""
    return max(linear_bytes(B, K, N, zero_points) / hbm_bytes_per_s,
               linear_flops(B, K, N) / flops_per_s)


def ridge_batch(hbm_bytes_per_s: float, flops_per_s: float,
                bytes_per_weight: float = BYTES_PER_WEIGHT_SYM) -> float:
    """Batch at which 2*B flops per weight take as long as streaming it."""
    return bytes_per_weight * flops_per_s / (2.0 * hbm_bytes_per_s)


@dataclass(frozen=True)
class Scheme:
    """One weight format in the two-term model."""
    bytes_per_weight: float
    tensor_peak: float           # P, flop/s of the mma the kernel issues
    c: float = 0.0               # dequant instruction slots per weight
    issue_rate: float = math.inf  # D, non-tensor instruction lanes per second


def step_time(W: float, B: float, beta: float, s: Scheme) -> float:
    memory = W * s.bytes_per_weight / beta
    math_pipe = 2.0 * W * B / s.tensor_peak + W * s.c / s.issue_rate
    return max(memory, math_pipe)


def memory_floor(W: float, beta: float, s: Scheme) -> float:
    return W * s.bytes_per_weight / beta


def mma_slope(W: float, s: Scheme) -> float:
    """Seconds added per unit of batch by the tensor-core term."""
    return 2.0 * W / s.tensor_peak


def dequant_tax(W: float, s: Scheme) -> float:
    return W * s.c / s.issue_rate


def batch_where_math_reaches(level_s: float, W: float, s: Scheme) -> float:
    """Batch at which the math term 2WB/P + Wc/D equals ``level_s``."""
    return (level_s - dequant_tax(W, s)) * s.tensor_peak / (2.0 * W)
