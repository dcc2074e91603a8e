"""Pins for the oracle's fused epilogues (``oracle.gemm_epilogue``): bias add
and the gated-MLP SiLU(gate) * up on interleaved columns.

Closed forms: with unit scales, constant codes per column and x all ones,
every sum is K * (code - 8), so the epilogue's result is known exactly; silu
is checked against an independent route, silu(g) = g (1 + tanh(g/2)) / 2.
A swapped gate/up pair, a bias on the wrong column or a missing rounding
changes a value.
"""
import numpy as np
import pytest

import oracle
from tests.bf16_exact import bits_to_f64

ONE = 0x3F80


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def layer(K, codes):
    """qweight with a constant code per column, unit scales."""
    N = len(codes)
    qw = np.zeros((K // 8, N), dtype=np.uint32)
    for n, c in enumerate(codes):
        qw[:, n] = sum(int(c) << (4 * j) for j in range(8))
    sc = np.full((K // 128, N), ONE, dtype=np.uint16)
    return qw, sc


def bf16(v):
    f = np.asarray(v, dtype=np.float32)
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)
    return (b >> 16).astype(np.uint16)


def test_bias_closed_form():
    K = 128
    qw, sc = layer(K, [9, 9, 7, 8, 12, 8, 8, 8])        # sums 128, 128, -128, 0, 512, 0, 0, 0
    bias = bf16([0.5, 1.0, -3.0, 2.5, 0.0, -0.25, 0.0, 7.0])
    x = np.full((2, K), ONE, dtype=np.uint16)
    y, v, bound = oracle.gemm_epilogue(x, qw, sc, bias=bias, mode=oracle.EPI_BIAS)
    want_v = np.array([128.5, 129.0, -131.0, 2.5, 512.0, -0.25, 0.0, 7.0])
    assert np.array_equal(v[0], want_v) and np.array_equal(v[1], want_v)
    # 128.5 lies halfway between the bf16 neighbours 128 and 129: ties to even
    want_y = np.array([128.0, 129.0, -131.0, 2.5, 512.0, -0.25, 0.0, 7.0])
    assert np.array_equal(bits_to_f64(y[0]), want_y)
    # the bias widens the bound by one bf16 step of its own size
    assert bound[0, 0] == pytest.approx(8e-3 * 128 + 1e-6 + 2.0 ** -7 * 0.5)


def test_silu_gate_closed_form():
    """Gate sums 0 (code 8) give 0; gate sums 896 (code 15) give silu = 896
    exactly in binary64 (e^-896 underflows), so h = 896 * 128 * (c_up - 8),
    exact in bf16; gate -896 (code 1) gives silu = -0.0 * ..., i.e. zero."""
    K = 128
    gates = [8, 15, 15, 15, 1, 15]
    ups = [13, 9, 11, 1, 15, 8]
    codes = [c for pair in zip(gates, ups) for c in pair]   # interleaved 2j, 2j + 1
    qw, sc = layer(K, codes)
    x = np.full((1, K), ONE, dtype=np.uint16)
    y, h, _ = oracle.gemm_epilogue(x, qw, sc, mode=oracle.EPI_SILU_MUL)
    want = np.array([0.0, 896 * 128 * 1, 896 * 128 * 3, 896 * 128 * -7, 0.0, 0.0])
    assert np.array_equal(h[0], want)
    assert np.array_equal(bits_to_f64(y[0]), want)
    # column subset: gate columns 2 and 6 -> outputs 1 and 3
    y2, _, _ = oracle.gemm_epilogue(x, qw, sc, mode=oracle.EPI_SILU_MUL,
                                    cols=np.array([2, 6], dtype=np.int32))
    assert np.array_equal(y2[0], y[0, [1, 3]])


def test_bias_then_silu_order():
    """The bias is added to gate and up before the activation: gate code 8
    (sum 0) with bias 1.0 gives silu(1) * (up + bias_up)."""
    K = 128
    qw, sc = layer(K, [8, 10])                       # g = 0, u = 256
    bias = bf16([1.0, -0.5])
    x = np.full((1, K), ONE, dtype=np.uint16)
    _, h, _ = oracle.gemm_epilogue(x, qw, sc, bias=bias, mode=oracle.EPI_BIAS | oracle.EPI_SILU_MUL)
    assert h[0, 0] == pytest.approx((1.0 / (1.0 + np.exp(-1.0))) * 255.5, rel=1e-15)


def test_silu_matches_the_tanh_route():
    """g (1 + tanh(g/2)) / 2 for g > -4 (where 1 + tanh keeps its digits), and
    g e^g / (1 + e^g) below."""
    g = np.random.default_rng(0).standard_normal(20000) * 12.0
    hi = g > -4
    ref = np.where(hi, g * (1.0 + np.tanh(g / 2.0)) / 2.0, g * np.exp(g) / (1.0 + np.exp(g)))
    assert np.allclose(oracle.silu(g), ref, rtol=1e-12, atol=0)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    # sup of the slope used in the bound
    t = np.linspace(-20, 20, 400001)
    slope = np.gradient(oracle.silu(t), t)
    assert slope.max() < oracle.SILU_SLOPE_MAX and slope.min() > -oracle.SILU_SLOPE_MAX
