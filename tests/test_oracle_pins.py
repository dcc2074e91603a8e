"""Pins of the CPU oracle against what the pages and the arithmetic fix.

None of these retypes the oracle's formulas: rounding is checked against an
enumeration of all bf16 values (``bf16_exact``), dot products against exact
rationals or integer matmuls, and layouts against hand-built single-nibble
cases whose answer is known by construction.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.bf16_exact import bits_to_f64, nearest_bf16_bits, nearest_bf16_bits_fraction
from weight_only_int4_gemm_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _np(t):
    return t.contiguous().view(dtype=__import__("torch").int16).numpy().view(np.uint16) \
        if str(t.dtype) == "torch.bfloat16" else t.contiguous().numpy()


# ---------------------------------------------------------------- bf16 codec

def test_bf16_roundtrip_every_pattern():
    lib = oracle._load()
    for h in range(0x10000):
        v = lib.oracle_bf16_to_double(h)
        if np.isnan(v):
            continue
        assert lib.oracle_bf16_from_double(v) == h, hex(h)


def test_magic_constants_from_the_page():
    """EX holds bf16 128.0, SUB holds bf16 136.0, and 0x4300|q decodes to 128+q."""
    g = _golden("magic_constants.json")
    ex, sub, mask = int(g["EX"], 16), int(g["SUB"], 16), int(g["MASK"], 16)
    assert oracle.bf16_from_double(g["EX_half_value"]) == ex & 0xFFFF == ex >> 16
    assert oracle.bf16_from_double(g["SUB_half_value"]) == sub & 0xFFFF == sub >> 16
    assert mask & 0xFFFF == 0xF and mask >> 16 == 0xF
    for q in range(16):
        v = oracle.bf16_to_double((ex & 0xFFFF) | q)
        assert v == 128.0 + q
        assert v - oracle.bf16_to_double(sub & 0xFFFF) == q - g["bias"]
    assert g["non_tensor_instructions_per_4_weights"] / g["weights_per_32bit_word_in_one_call"] == g["c"]


def test_rounding_matches_enumeration_on_random_doubles():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(200_000) * 10.0 ** rng.integers(-45, 39, 200_000),
        rng.standard_normal(2000) * 2.0 ** -134,            # deep subnormal range
        np.array([0.0, -0.0, 3.4e38, 3.39e38, -3.4e38, 1e39, 2.0 ** -133, 2.0 ** -134,
                  1.5 * 2.0 ** -133, 2.0 ** -126 * (1 - 2.0 ** -9)]),
    ])
    got = np.array([oracle.bf16_from_double(float(v)) for v in vals], dtype=np.uint16)
    want = nearest_bf16_bits(vals)
    np.testing.assert_array_equal(got, want)


def test_rounding_ties_go_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: tie -> even (1.0)
    assert oracle.bf16_from_double(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even)
    assert oracle.bf16_from_double(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # halfway past the largest finite value rounds to infinity
    assert oracle.bf16_from_double((2 - 2.0 ** -8) * 2.0 ** 127) == 0x7F80
    assert oracle.bf16_from_double(-(2 - 2.0 ** -8) * 2.0 ** 127) == 0xFF80


# ------------------------------------------------------- dequant, exhaustive

def _all_codes_by_all_scales():
    """K = 128, N = 65536: rows 0..15 hold codes 0..15 in every column, column n
    carries scale bit pattern n (non-finite patterns replaced by 0 and masked)."""
    N = 0x10000
    qweight = np.full((16, N), 0x88888888, dtype=np.uint32)
    qweight[0, :] = 0x76543210           # rows 0..7 -> codes 0..7
    qweight[1, :] = 0xFEDCBA98           # rows 8..15 -> codes 8..15
    scale_bits = np.arange(N, dtype=np.uint32).astype(np.uint16)
    finite = np.isfinite(bits_to_f64(scale_bits))
    scales = np.where(finite, scale_bits, 0).astype(np.uint16)[None, :]
    return qweight, scales, finite


def test_dequant_exhaustive_symmetric():
    """All 16 codes x all finite bf16 scales: w == nearest_bf16((q - 8) * s)."""
    qweight, scales, finite = _all_codes_by_all_scales()
    w = oracle.dequant(qweight, scales)
    s = bits_to_f64(scales[0])
    for q in range(16):
        want = nearest_bf16_bits((q - 8) * s)
        np.testing.assert_array_equal(w[q][finite], want[finite], err_msg=f"code {q}")
    # rows 16.. hold code 8 -> (8 - 8) * s = signed zero
    np.testing.assert_array_equal(w[16:][:, finite], np.where(np.signbit(s[finite]), 0x8000, 0)[None, :]
                                  .repeat(112, 0).astype(np.uint16))


def test_dequant_unit_scale_gives_integer_codes():
    qweight, _, _ = _all_codes_by_all_scales()
    ones = np.full((1, 0x10000), 0x3F80, dtype=np.uint16)
    w = oracle.dequant(qweight[:, :64], ones[:, :64])
    for q in range(16):
        assert np.all(bits_to_f64(w[q]) == q - 8)


def test_dequant_exhaustive_zero_points():
    """All (q, z) pairs x all finite scales: w == nearest_bf16((q - z) * s)."""
    qweight, scales, finite = _all_codes_by_all_scales()
    s = bits_to_f64(scales[0])
    for z in range(16):
        qzeros = np.full((1, 0x10000 // 8), z * 0x11111111, dtype=np.uint32)
        w = oracle.dequant(qweight, scales, qzeros)
        for q in range(16):
            want = nearest_bf16_bits((q - z) * s)
            np.testing.assert_array_equal(w[q][finite], want[finite], err_msg=f"q={q} z={z}")


def test_zero_point_eight_is_the_symmetric_format():
    p = inputs.make_problem(3, 384, 40, seed=11)
    qw, sc = _np(p.qweight), _np(p.scales)
    eights = np.full((3, 5), 0x88888888, dtype=np.uint32)
    np.testing.assert_array_equal(oracle.dequant(qw, sc), oracle.dequant(qw, sc, eights))
    y0, a0, _ = oracle.gemm(_np(p.x), qw, sc)
    y1, a1, _ = oracle.gemm(_np(p.x), qw, sc, eights)
    np.testing.assert_array_equal(y0, y1)
    np.testing.assert_array_equal(a0, a1)


# ------------------------------------------------------- layout, by construction

@pytest.mark.parametrize("kk,j,n", [(0, 0, 0), (0, 7, 5), (3, 4, 17), (31, 1, 23), (17, 6, 0)])
def test_single_nibble_lands_on_row_8kk_plus_j(kk, j, n):
    K, N = 256, 24
    qweight = np.full((K // 8, N), 0x88888888, dtype=np.uint32)
    qweight[kk, n] = (qweight[kk, n] & ~np.uint32(0xF << (4 * j))) | np.uint32(0xB << (4 * j))
    assert oracle.code(qweight, 8 * kk + j, n) == 0xB
    # scales differ per group and column so a wrong group index is visible
    scales = np.empty((K // 128, N), dtype=np.uint16)
    for g in range(K // 128):
        for c in range(N):
            scales[g, c] = oracle.bf16_from_double(2.0 ** (g - 3) * (1 + c / 32))
    w = bits_to_f64(oracle.dequant(qweight, scales))
    nz = np.argwhere(w != 0)
    assert nz.tolist() == [[8 * kk + j, n]]
    k = 8 * kk + j
    assert w[k, n] == (0xB - 8) * bits_to_f64(scales[k // 128, n])


@pytest.mark.parametrize("g,nn,j", [(0, 0, 0), (1, 2, 7), (2, 1, 3)])
def test_single_zero_point_nibble_lands_on_column_8nn_plus_j(g, nn, j):
    K, N = 384, 24
    qweight = np.full((K // 8, N), 0x55555555, dtype=np.uint32)      # every code is 5
    qzeros = np.full((K // 128, N // 8), 0x55555555, dtype=np.uint32)  # every zero is 5
    qzeros[g, nn] = (qzeros[g, nn] & ~np.uint32(0xF << (4 * j))) | np.uint32(0x2 << (4 * j))
    n = 8 * nn + j
    assert oracle.zero(qzeros, N, g, n) == 2
    assert oracle.zero(None, N, g, n) == 8
    scales = np.full((K // 128, N), 0x3F80, dtype=np.uint16)
    w = bits_to_f64(oracle.dequant(qweight, scales, qzeros))
    nz = np.argwhere(w != 0)
    rows = set(nz[:, 0].tolist())
    assert rows == set(range(128 * g, 128 * (g + 1)))
    assert set(nz[:, 1].tolist()) == {n}
    assert np.all(w[128 * g:128 * (g + 1), n] == 3.0)


# ------------------------------------------------------------- GEMM pins

@pytest.mark.parametrize("zp", [False, True])
def test_gemm_integer_special_case_is_exact(zp):
    """s = 1 and integer x: every product and partial sum is an exact integer,
    so the reference equals an int64 matmul of (q - z) and x."""
    rng = np.random.default_rng(3)
    B, K, N = 5, 384, 24
    qweight = rng.integers(0, 2 ** 32, (K // 8, N), dtype=np.uint64).astype(np.uint32)
    qzeros = rng.integers(0, 2 ** 32, (K // 128, N // 8), dtype=np.uint64).astype(np.uint32) if zp else None
    scales = np.full((K // 128, N), 0x3F80, dtype=np.uint16)
    xi = rng.integers(-4, 5, (B, K))
    x = nearest_bf16_bits(xi.astype(np.float64))
    codes = ((qweight[:, None, :] >> (4 * np.arange(8, dtype=np.uint32))[None, :, None]) & 0xF) \
        .reshape(K, N).astype(np.int64)
    if zp:
        zc = ((qzeros[:, :, None] >> (4 * np.arange(8, dtype=np.uint32))[None, None, :]) & 0xF) \
            .reshape(K // 128, N).astype(np.int64)
        zk = np.repeat(zc, 128, axis=0)
    else:
        zk = 8
    exact = xi @ (codes - zk)
    y, acc, bound = oracle.gemm(x, qweight, scales, qzeros)
    np.testing.assert_array_equal(acc, exact.astype(np.float64))
    np.testing.assert_array_equal(y, nearest_bf16_bits(exact.astype(np.float64)))
    np.testing.assert_array_equal(bound, 8e-3 * (np.abs(xi) @ np.abs(codes - zk)) + 1e-6)


@pytest.mark.parametrize("zp,B,K,N", [(False, 3, 256, 16), (True, 2, 128, 8), (False, 4, 128, 16)])
def test_gemm_brute_force_exact_rationals(zp, B, K, N):
    p = inputs.make_problem(B, K, N, seed=100 + B + K, zero_points=zp)
    x, qw, sc = _np(p.x), _np(p.qweight).view(np.uint32), _np(p.scales)
    qz = None if p.qzeros is None else _np(p.qzeros).view(np.uint32)
    codes = ((qw[:, None, :] >> (4 * np.arange(8, dtype=np.uint32))[None, :, None]) & 0xF).reshape(K, N)
    if zp:
        zc = ((qz[:, :, None] >> (4 * np.arange(8, dtype=np.uint32))[None, None, :]) & 0xF).reshape(K // 128, N)
        zk = np.repeat(zc, 128, axis=0).astype(np.int64)
    else:
        zk = np.full((K, N), 8, dtype=np.int64)
    s_k = np.repeat(bits_to_f64(sc), 128, axis=0)
    w_bits = nearest_bf16_bits((codes.astype(np.int64) - zk) * s_k)
    np.testing.assert_array_equal(oracle.dequant(qw, sc, qz), w_bits)
    w = bits_to_f64(w_bits)
    xv = bits_to_f64(x)
    y, acc, bound = oracle.gemm(x, qw, sc, qz)
    for b in range(B):
        for n in range(N):
            exact = sum((Fraction(float(xv[b, k])) * Fraction(float(w[k, n])) for k in range(K)),
                        Fraction(0))
            mag = float(np.sum(np.abs(xv[b] * w[:, n])))
            assert abs(Fraction(float(acc[b, n])) - exact) <= Fraction(1e-12) * Fraction(mag)
            assert y[b, n] == nearest_bf16_bits_fraction(exact)
            assert abs(bound[b, n] - (8e-3 * mag + 1e-6)) <= 1e-12 * (mag + 1)


def test_bound_hand_computed():
    """x0 = 3, x1 = 1.5, s = 0.5, q0 = 10 -> w0 = 1, q1 = 4 -> w1 = -2, rest 0:
    acc = 3 - 3 = 0 and sum|x*w| = 6, so the bound is 0.048 + 1e-6."""
    K, N = 128, 8
    qweight = np.full((K // 8, N), 0x88888888, dtype=np.uint32)
    qweight[0, 0] = (0x88888888 & ~0xFF) | 0x4A           # k0 -> 0xA, k1 -> 0x4
    scales = np.full((1, N), oracle.bf16_from_double(0.5), dtype=np.uint16)
    x = np.zeros((1, K), dtype=np.uint16)
    x[0, 0] = oracle.bf16_from_double(3.0)
    x[0, 1] = oracle.bf16_from_double(1.5)
    y, acc, bound = oracle.gemm(x, qweight, scales)
    assert acc[0, 0] == 0.0 and y[0, 0] == 0
    assert bound[0, 0] == pytest.approx(0.048001, rel=0, abs=1e-15)
    assert np.all(acc[0, 1:] == 0.0) and np.all(bound[0, 1:] == 1e-6)


def test_gemm_invariants():
    p = inputs.make_problem(3, 512, 32, seed=5, zero_points=True)
    x, qw, sc, qz = _np(p.x), _np(p.qweight), _np(p.scales), _np(p.qzeros)
    y, acc, _ = oracle.gemm(x, qw, sc, qz)
    # doubling every scale doubles every weight and every sum exactly
    sc2 = ((sc.astype(np.uint32) << 16).view(np.float32) * 2).view(np.uint32) >> 16
    y2, acc2, _ = oracle.gemm(x, qw, sc2.astype(np.uint16), qz)
    np.testing.assert_array_equal(acc2, 2 * acc)
    np.testing.assert_array_equal(bits_to_f64(y2), 2 * bits_to_f64(y))
    # negating x negates the result exactly
    yn, accn, _ = oracle.gemm(x ^ np.uint16(0x8000), qw, sc, qz)
    np.testing.assert_array_equal(accn, -acc)
    np.testing.assert_array_equal(bits_to_f64(yn), -bits_to_f64(y))
    # a column subset agrees with the full product
    cols = np.array([31, 0, 7, 8, 19], dtype=np.int32)
    ys, accs, _ = oracle.gemm(x, qw, sc, qz, cols=cols)
    np.testing.assert_array_equal(ys, y[:, cols])
    np.testing.assert_array_equal(accs, acc[:, cols])
    # splitting K into halves and adding matches to double rounding
    h = 256
    _, a_lo, b_lo = oracle.gemm(np.ascontiguousarray(x[:, :h]), np.ascontiguousarray(qw[:h // 8]),
                                np.ascontiguousarray(sc[:h // 128]), np.ascontiguousarray(qz[:h // 128]))
    _, a_hi, b_hi = oracle.gemm(np.ascontiguousarray(x[:, h:]), np.ascontiguousarray(qw[h // 8:]),
                                np.ascontiguousarray(sc[h // 128:]), np.ascontiguousarray(qz[h // 128:]))
    mag = (b_lo + b_hi - 2e-6) / 8e-3
    assert np.all(np.abs(a_lo + a_hi - acc) <= 1e-13 * mag + 1e-300)


# ------------------------------------------------------------ format size

def test_effective_bits_per_weight():
    g = _golden("format_accounting.json")
    for K, N in [(4096, 4096), (14336, 4096), (4096, 128256)]:
        assert oracle.format_bits_per_weight(K, N, False) == g["bits_per_weight_symmetric"]
        assert oracle.format_bits_per_weight(K, N, False) - 4 == g["scale_overhead_bits"]
        # a 4-bit zero-point per group of 128 adds 4/128 bit
        assert oracle.format_bits_per_weight(K, N, True) == g["bits_per_weight_symmetric"] + 4 / 128
