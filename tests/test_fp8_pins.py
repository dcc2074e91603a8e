"""Pins for the oracle's W8A8-FP8 path ("Give Me BF16 or Give Me Death",
section "W8A8-FP Quantization: 8-Bit Floating-Point Weights and Activations").

The E4M3 codec is pinned to the format's published constants (OCP 8-bit
floating point, E4M3: bias 7, no infinities, largest finite 448 = S.1111.110,
NaN = S.1111.111, smallest normal 2^-6, smallest subnormal 2^-9) and the
encoder to a brute-force nearest search over every finite code.  The
quantisers are pinned by invariants (the largest element maps to +-448, power
of two scaling, sign symmetry, transposition), the GEMM by an exact int64
product of the codes and a hand-computed case.
"""
import numpy as np
import pytest

import oracle
from tests.bf16_exact import bits_to_f64, nearest_bf16_bits


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def table():
    return np.array([oracle.e4m3_to_double(c) for c in range(256)])


def test_published_constants():
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0xFE) == -448.0
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_double(0x07) == 0.875 * 2.0 ** -6
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_double(0x38) == 1.0
    assert oracle.e4m3_to_double(0x40) == 2.0
    assert oracle.e4m3_to_double(0x00) == 0.0
    assert np.signbit(oracle.e4m3_to_double(0x80))
    assert np.isnan(oracle.e4m3_to_double(0x7F)) and np.isnan(oracle.e4m3_to_double(0xFF))


def test_codes_are_ordered_and_mirrored():
    t = table()
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(t[0x80:0xFF], -pos)


def brute_force_nearest(v, t):
    """Nearest finite E4M3 code by comparison, ties to the even code, and
    saturation at +-448."""
    codes = np.array([c for c in range(256) if np.isfinite(t[c]) and c != 0x80])
    vals = t[codes]
    out = []
    for x in v:
        if abs(x) >= 448.0:
            out.append(0x7E if x > 0 else 0xFE)
            continue
        d = np.abs(vals - x)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            best = [b for b in best if codes[b] % 2 == 0]
        c = int(codes[best[0]])
        if c == 0 and np.signbit(x):
            c = 0x80
        out.append(c)
    return np.array(out)


def test_encoder_is_the_nearest_code():
    t = table()
    rng = np.random.default_rng(0)
    mags = np.exp2(rng.uniform(-12, 9.5, 6000))
    vals = mags * rng.choice([-1.0, 1.0], size=mags.shape)
    # every exact midpoint between neighbouring codes (ties) and the codes themselves
    pos = t[:0x7F]
    mids = (pos[1:] + pos[:-1]) / 2
    vals = np.concatenate([vals, pos, -pos[1:], mids, -mids, [460.0, 464.0, 470.0, 1e6]])
    got = np.array([oracle.e4m3_from_double(x) for x in vals])
    assert np.array_equal(got, brute_force_nearest(vals, t))


def bf16(v):
    f = np.asarray(v, dtype=np.float32)
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)
    return (b >> 16).astype(np.uint16)


def rand_bf16(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    f = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def test_largest_element_maps_to_qmax_and_zero_rows():
    x = rand_bf16((6, 256), 1)
    x[3] = 0
    codes, s = oracle.fp8_quantize_rows(x)
    t = table()
    xv = bits_to_f64(x)
    for b in range(6):
        if b == 3:
            assert s[b] == 0 and np.all(codes[b] == 0)
            continue
        i = int(np.argmax(np.abs(xv[b])))
        assert abs(t[codes[b, i]]) == 448.0
        # dequantised values are within half a code step (relative 2^-4) plus
        # the subnormal quantum of the input
        deq = t[codes[b]] * float(s[b])
        assert np.all(np.abs(deq - xv[b]) <= np.abs(xv[b]) * 2.0 ** -4 + float(s[b]) * 2.0 ** -10)


def test_power_of_two_and_sign_invariance():
    x = rand_bf16((4, 384), 2)
    c1, s1 = oracle.fp8_quantize_rows(x)
    x4 = bf16(bits_to_f64(x) * 4.0)
    c4, s4 = oracle.fp8_quantize_rows(x4)
    assert np.array_equal(c1, c4) and np.array_equal(s1 * 4, s4)
    cn, sn = oracle.fp8_quantize_rows(x ^ np.uint16(0x8000))
    assert np.array_equal(sn, s1)
    nz = c1 != 0
    assert np.array_equal(cn[nz], c1[nz] ^ 0x80)


def test_columns_are_rows_of_the_transpose():
    w = rand_bf16((256, 24), 3, 0.02)
    cc, sc = oracle.fp8_quantize_cols(w)
    cr, sr = oracle.fp8_quantize_rows(np.ascontiguousarray(w.T))
    assert np.array_equal(cc, cr) and np.array_equal(sc, sr)


def test_gemm_sum_is_exact_int_product():
    """Every E4M3 value times 2^9 is an integer: acc * 2^18 must equal the int64
    product of the scaled codes exactly, for any codes."""
    t = table()
    rng = np.random.default_rng(4)
    finite = np.array([c for c in range(256) if np.isfinite(t[c])], dtype=np.uint8)
    B, K, N = 5, 1024, 12
    xq = rng.choice(finite, size=(B, K))
    wq = rng.choice(finite, size=(N, K))
    sx = np.ones(B, dtype=np.float32)
    sw = np.ones(N, dtype=np.float32)
    _, acc, _ = oracle.fp8_gemm(xq, sx, wq, sw)
    xi = (t[xq] * 512).astype(np.int64)
    wi = (t[wq] * 512).astype(np.int64)
    assert np.array_equal((acc * 2.0 ** 18).astype(np.int64), xi @ wi.T)


def test_gemm_output_is_nearest_bf16_of_scaled_sum():
    t = table()
    rng = np.random.default_rng(5)
    B, K, N = 3, 256, 7
    xq = rng.integers(0, 0x7F, size=(B, K)).astype(np.uint8)
    wq = rng.integers(0x80, 0xFF, size=(N, K)).astype(np.uint8)
    sx = np.array([2.0 ** -3, 1.0, 2.0 ** 5], dtype=np.float32)
    sw = np.exp2(rng.integers(-4, 4, N)).astype(np.float32)
    y, acc, _ = oracle.fp8_gemm(xq, sx, wq, sw)
    exact = (t[xq] @ t[wq].T) * sx[:, None].astype(np.float64) * sw[None, :].astype(np.float64)
    assert np.array_equal(y.astype(np.uint32), nearest_bf16_bits(exact))
    cols = np.array([6, 0, 3], dtype=np.int32)
    yc, _, _ = oracle.fp8_gemm(xq, sx, wq, sw, cols=cols)
    assert np.array_equal(yc, y[:, cols])


def test_bound_hand_case():
    """x = [1, -2] (codes 0x38, 0xC0), w = [3, 0.5] (0x44, 0x30), s_x = 0.5,
    s_w = 4: acc = 3 - 1 = 2, y = 4, bound = 8e-3 * (3 + 1) * 2 + 1e-6."""
    y, acc, bound = oracle.fp8_gemm(np.array([[0x38, 0xC0]]), np.array([0.5]),
                                    np.array([[0x44, 0x30]]), np.array([4.0]))
    assert acc[0, 0] == 2.0
    assert bits_to_f64(y)[0, 0] == 4.0
    assert bound[0, 0] == pytest.approx(8e-3 * 4 * 2 + 1e-6, rel=1e-12)
