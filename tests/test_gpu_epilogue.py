"""GPU parity of the fused epilogues (w4a16_gemm_fused) against the oracle,
on every kernel path (small-batch, TMEM tensor-core, wide tensor-core), with
and without a K split and zero-points.

Bar: the GEMM bound carried through the epilogue (oracle.gemm_epilogue):
bias adds one bf16 step of |bias|; SiLU(gate) * up uses the slope bound of
silu (<= 1.1) on the gate's error and |silu(g)| on the up's error, plus one
bf16 step of the result.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_int4_gemm_gb300 as w
from tests.bf16_exact import bits_to_f64
from tests.gpu_util import bits, sample_columns
from weight_only_int4_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

MODES = [w.EPI_BIAS, w.EPI_SILU_MUL, w.EPI_BIAS | w.EPI_SILU_MUL]


def run_fused(p, mode, bias):
    g = p.to("cuda")
    packed = w.w4a16_pack(g.qweight, g.qzeros)
    y = w.w4a16_gemm_fused(g.x, packed, g.scales, g.qzeros is not None, mode,
                           None if bias is None else bias.cuda())
    torch.cuda.synchronize()
    assert w.w4a16_device_status() == 0
    return y.cpu()


def check(p, mode, bias, y, cols=None):
    """cols: output columns to check (gate columns 2j for the SiLU form)."""
    yo, _, bound = oracle.gemm_epilogue(
        bits(p.x), bits(p.qweight), bits(p.scales), None if p.qzeros is None else bits(p.qzeros),
        bias=None if bias is None else bits(bias), mode=mode, cols=cols)
    yg = bits_to_f64(bits(y))
    if cols is not None:
        sel = np.asarray(cols) // 2 if mode & w.EPI_SILU_MUL else np.asarray(cols)
        yg = yg[:, sel]
    yo = bits_to_f64(yo)
    assert np.all(np.isfinite(yg)), "non-finite GPU output"
    bad = np.abs(yg - yo) > bound
    if bad.any():
        b, n = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} of {bad.size} outside the bound; first at "
                             f"({b}, {n}): gpu={yg[b, n]!r} oracle={yo[b, n]!r} bound={bound[b, n]!r}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("B,K,N,zp", [
    (1, 4096, 1032, False),    # small-batch kernel, K split, ragged tile
    (5, 1024, 520, True),      # small-batch kernel, zero-points
    (16, 2048, 264, False),    # small-batch kernel, 16-row tiles
    (40, 2048, 1032, True),    # TMEM tensor-core kernel
    (128, 4096, 520, False),   # TMEM tensor-core kernel, K split
    (200, 1024, 264, True),    # wide tensor-core kernel
])
def test_fused_epilogue(mode, B, K, N, zp):
    p = inputs.make_problem(B, K, N, 100 + B + mode, zero_points=zp)
    bias = inputs.make_bias(N, 7 + mode) if mode & w.EPI_BIAS else None
    check(p, mode, bias, run_fused(p, mode, bias))


@pytest.mark.parametrize("B", [1, 64, 512])
def test_gated_mlp_full_size(B):
    """Llama-3-8B gate+up (4096 -> 2 x 14336, interleaved) fused with SiLU:
    sampled gate columns, all rows."""
    K, N = 4096, 28672
    p = inputs.make_problem(B, K, N, 300 + B)
    y = run_fused(p, w.EPI_SILU_MUL, None)
    assert y.shape == (B, N // 2)
    gates = 2 * (sample_columns(N // 2, 128, B) )
    check(p, w.EPI_SILU_MUL, None, y, cols=gates)


def test_no_flags_is_the_plain_gemm():
    p = inputs.make_problem(9, 1024, 264, 5).to("cuda")
    packed = w.w4a16_pack(p.qweight, None)
    y0 = w.w4a16_gemm(p.x, packed, p.scales, False)
    y1 = w.w4a16_gemm_fused(p.x, packed, p.scales, False, w.EPI_NONE)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
