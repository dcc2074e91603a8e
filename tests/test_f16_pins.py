"""Pins of the fp16-activation oracle ("Give Me BF16 or Give Me Death",
"W4A16-INT Quantization", paragraph "Inference with W4A16": fp16 weights,
scales and tensor-core products) against what IEEE binary16 and the
arithmetic fix.

Nothing here retypes the oracle's formulas: decoding is checked against
numpy's float16, rounding against an enumeration of every binary16 value and
against numpy's float64 -> float16 conversion, dot products against exact
rationals and integer matmuls.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.f16_exact import f16_bits_to_f64, nearest_f16_bits, nearest_f16_bits_fraction

ALL = np.arange(0x10000, dtype=np.uint32)


def _codes(qweight, K, N):
    return ((qweight[:, None, :] >> (4 * np.arange(8, dtype=np.uint32))[None, :, None]) & 0xF) \
        .reshape(K, N).astype(np.int64)


# ---------------------------------------------------------------- codec

def test_decode_every_pattern_matches_numpy():
    lib = oracle._load()
    got = np.array([lib.oracle_f16_to_double(int(h)) for h in ALL])
    want = f16_bits_to_f64(ALL)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])
    # signed zeros keep their sign
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_roundtrip_every_finite_pattern():
    for h in ALL:
        v = oracle.f16_to_double(int(h))
        if not np.isnan(v):
            assert oracle.f16_from_double(v) == h, hex(h)


def test_every_midpoint_and_quarter_point():
    """Between each pair of neighbouring non-negative finite values a < b:
    the midpoint goes to the one with the even pattern, the quarter points
    to the nearer one (and the same mirrored for negatives)."""
    bits = np.arange(0, 0x7C00, dtype=np.uint32)
    vals = f16_bits_to_f64(bits)
    a, b = vals[:-1], vals[1:]
    mid = (a + b) / 2
    even_is_b = (bits[1:] % 2 == 0)
    want_mid = np.where(even_is_b, bits[1:], bits[:-1]).astype(np.uint16)
    got_mid = oracle.f16_round(mid)
    np.testing.assert_array_equal(got_mid, want_mid)
    np.testing.assert_array_equal(oracle.f16_round(-mid), want_mid | 0x8000)
    np.testing.assert_array_equal(oracle.f16_round(a + (b - a) / 4), bits[:-1].astype(np.uint16))
    np.testing.assert_array_equal(oracle.f16_round(b - (b - a) / 4), bits[1:].astype(np.uint16))


def test_rounding_matches_enumeration_and_numpy_on_random_doubles():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.standard_normal(200_000) * 10.0 ** rng.integers(-9, 6, 200_000),
        rng.standard_normal(2000) * 2.0 ** -25,              # subnormal range
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e6, 2.0 ** -24,
                  2.0 ** -25, 1.5 * 2.0 ** -24, 2.0 ** -14 * (1 - 2.0 ** -12)]),
    ])
    got = oracle.f16_round(vals)
    np.testing.assert_array_equal(got, nearest_f16_bits(vals))
    np.testing.assert_array_equal(got, vals.astype(np.float16).view(np.uint16))


def test_ties_and_overflow_by_hand():
    assert oracle.f16_from_double(1.0 + 2.0 ** -11) == 0x3C00        # tie -> even (1.0)
    assert oracle.f16_from_double(1.0 + 3 * 2.0 ** -11) == 0x3C02    # tie -> even (1 + 2^-9)
    assert oracle.f16_from_double(65519.0) == 0x7BFF
    assert oracle.f16_from_double(65520.0) == 0x7C00                 # tie past max -> inf
    assert oracle.f16_from_double(2.0 ** -25) == 0x0000              # tie -> even (zero)
    assert oracle.f16_from_double(3 * 2.0 ** -25) == 0x0002          # tie -> even (2 * 2^-24)


# ---------------------------------------------------------------- dequant

def test_magic_decode_constants():
    """fp16 1024.0 is 0x6400 and its 10 fraction bits hold a nibble exactly:
    0x6400 | q decodes to 1024 + q, and 1032 (0x6408) takes the bias 8 off."""
    assert oracle.f16_from_double(1024.0) == 0x6400
    assert oracle.f16_from_double(1032.0) == 0x6408
    for q in range(16):
        assert oracle.f16_to_double(0x6400 | q) - oracle.f16_to_double(0x6408) == q - 8


def test_dequant_every_code_times_every_finite_scale():
    """All 16 codes x every finite fp16 scale, with z = 8 and with every z:
    RNE_f16((q - z) * s) against numpy's float64 -> float16 conversion of the
    exact product."""
    scale_bits = ALL[np.isfinite(f16_bits_to_f64(ALL))].astype(np.uint16)
    s = f16_bits_to_f64(scale_bits)
    N = scale_bits.size - scale_bits.size % 8
    scale_bits, s = scale_bits[:N], s[:N]
    qweight = np.full((16, N), 0x88888888, dtype=np.uint32)
    qweight[0, :] = 0x76543210
    qweight[1, :] = 0xFEDCBA98
    for z in (8, 0, 3, 15):
        qzeros = None if z == 8 else np.full((1, N // 8), z * 0x11111111, dtype=np.uint32)
        w = oracle.dequant_f16(qweight, scale_bits[None, :], qzeros)
        for q in range(16):
            want = (np.float64(q - z) * s).astype(np.float16).view(np.uint16)
            np.testing.assert_array_equal(w[q], want, err_msg=f"q={q} z={z}")


def test_dequant_one_agrees_with_the_array_form():
    for q, z, sb in [(0, 8, 0x3C00), (15, 8, 0x7BFF), (15, 0, 0x7BFF), (9, 8, 0x0001),
                     (3, 8, 0x8001), (8, 8, 0x7C00 - 1)]:
        want = np.float16(np.float64(q - z) * f16_bits_to_f64(sb)).view(np.uint16)
        assert oracle.dequant_one_f16(q, z, sb) == want


# ---------------------------------------------------------------- GEMM

@pytest.mark.parametrize("zp", [False, True])
def test_gemm_integer_case_is_exact(zp):
    """s = 1 and integer x: the reference equals an int64 matmul of (q - z)."""
    rng = np.random.default_rng(5)
    B, K, N = 4, 384, 24
    qweight = rng.integers(0, 2 ** 32, (K // 8, N), dtype=np.uint64).astype(np.uint32)
    qzeros = rng.integers(0, 2 ** 32, (K // 128, N // 8), dtype=np.uint64).astype(np.uint32) \
        if zp else None
    scales = np.full((K // 128, N), 0x3C00, dtype=np.uint16)
    xi = rng.integers(-4, 5, (B, K))
    x = xi.astype(np.float16).view(np.uint16)
    codes = _codes(qweight, K, N)
    if zp:
        zc = ((qzeros[:, :, None] >> (4 * np.arange(8, dtype=np.uint32))[None, None, :]) & 0xF) \
            .reshape(K // 128, N).astype(np.int64)
        zk = np.repeat(zc, 128, axis=0)
    else:
        zk = 8
    exact = xi @ (codes - zk)
    y, acc, bound = oracle.gemm_f16(x, qweight, scales, qzeros)
    np.testing.assert_array_equal(acc, exact.astype(np.float64))
    np.testing.assert_array_equal(y, nearest_f16_bits(exact.astype(np.float64)))
    mag = np.abs(xi) @ np.abs(codes - zk)
    np.testing.assert_allclose(bound, 2e-3 * mag + 2.0 ** -24 * (1 + np.abs(xi).sum(1))[:, None],
                               rtol=1e-15, atol=0)


@pytest.mark.parametrize("zp,B,K,N", [(False, 3, 256, 16), (True, 2, 128, 8)])
def test_gemm_brute_force_exact_rationals(zp, B, K, N):
    rng = np.random.default_rng(100 + B + K)
    qweight = rng.integers(0, 2 ** 32, (K // 8, N), dtype=np.uint64).astype(np.uint32)
    qzeros = rng.integers(0, 2 ** 32, (K // 128, N // 8), dtype=np.uint64).astype(np.uint32) \
        if zp else None
    scales = (rng.uniform(0.002, 0.05, (K // 128, N))).astype(np.float16).view(np.uint16)
    x = rng.standard_normal((B, K)).astype(np.float16).view(np.uint16)
    codes = _codes(qweight, K, N)
    if zp:
        zc = ((qzeros[:, :, None] >> (4 * np.arange(8, dtype=np.uint32))[None, None, :]) & 0xF) \
            .reshape(K // 128, N)
        zk = np.repeat(zc, 128, axis=0).astype(np.int64)
    else:
        zk = np.full((K, N), 8, dtype=np.int64)
    s_k = np.repeat(f16_bits_to_f64(scales), 128, axis=0)
    w_bits = nearest_f16_bits((codes - zk) * s_k)
    np.testing.assert_array_equal(oracle.dequant_f16(qweight, scales, qzeros), w_bits)
    w, xv = f16_bits_to_f64(w_bits), f16_bits_to_f64(x)
    y, acc, bound = oracle.gemm_f16(x, qweight, scales, qzeros)
    for b in range(B):
        for n in range(N):
            exact = sum((Fraction(float(xv[b, k])) * Fraction(float(w[k, n])) for k in range(K)),
                        Fraction(0))
            mag = float(np.sum(np.abs(xv[b] * w[:, n])))
            assert abs(Fraction(float(acc[b, n])) - exact) <= Fraction(1e-12) * Fraction(mag)
            assert y[b, n] == nearest_f16_bits_fraction(exact)
            want_bound = 2e-3 * mag + 2.0 ** -24 * (1 + float(np.abs(xv[b]).sum()))
            assert abs(bound[b, n] - want_bound) <= 1e-12 * (mag + 1)


def test_bf16_and_f16_oracles_agree_where_both_are_exact():
    """Small integers and power-of-two scales are exact in both formats: the
    two oracles' unrounded sums are equal, and the fp16 output is that sum
    rounded by the enumeration."""
    rng = np.random.default_rng(9)
    B, K, N = 3, 256, 16
    qweight = rng.integers(0, 2 ** 32, (K // 8, N), dtype=np.uint64).astype(np.uint32)
    s = np.exp2(rng.integers(-3, 2, (K // 128, N))).astype(np.float64)
    xi = rng.integers(-8, 9, (B, K)).astype(np.float64)
    s_bf16 = (s.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x_bf16 = (xi.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    _, acc_b, _ = oracle.gemm(x_bf16, qweight, s_bf16)
    y_h, acc_h, _ = oracle.gemm_f16(xi.astype(np.float16).view(np.uint16), qweight,
                                    s.astype(np.float16).view(np.uint16))
    np.testing.assert_array_equal(acc_b, acc_h)
    np.testing.assert_array_equal(y_h, nearest_f16_bits(acc_h))
