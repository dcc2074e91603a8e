"""Pins for the oracle's offline quantizer (round to nearest with MSE-optimal
clipping, "Give Me BF16 or Give Me Death", section "W4A16-INT Quantization",
paragraph "Weight quantization algorithm: GPTQ with MSE-optimal clipping").

Each pin is fixed by construction or by hand, not by re-running the
quantizer's own formula: a group that lies exactly on an abs-max grid, a group
of zeros, exact invariances (power-of-two scaling, sign), and a worked example
whose optimum clipping ratio is derived in the docstring.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def bf16_bits(v):
    """Exact float32 -> bf16 bits (test values are chosen exactly representable)."""
    f = np.asarray(v, dtype=np.float32)
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "test value not exactly representable in bf16"
    return (b >> 16).astype(np.uint16)


def codes_of(qw):
    """Canonical qweight [K/8][N] -> codes [K][N]."""
    K8, N = qw.shape
    out = np.zeros((K8 * 8, N), dtype=np.int64)
    for j in range(8):
        out[j::8] = (qw >> (4 * j)) & 0xF
    return out


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def test_group_on_the_absmax_grid_is_recovered_exactly():
    """Values c * s0 with c in [-7, 7] (both +-7 present) and s0 = 2^-6: the
    abs-max scale is s0 exactly, every value is reconstructed with no error, so
    the first grid point (alpha = 1) is kept: codes c + 8, scale s0."""
    rng = np.random.default_rng(1)
    c = rng.integers(-7, 8, size=(128, 3))
    c[0] = 7
    c[1] = -7
    s0 = 2.0 ** -6
    qw, sc = oracle.quantize_rtn_mse(bf16_bits(c * s0))
    assert np.array_equal(codes_of(qw), c + 8)
    assert np.all(sc == bf16_bits(s0))


def test_zero_group_has_zero_scale_and_zero_codes():
    w = np.zeros((256, 8), dtype=np.float32)
    w[128:, :] = 1.0  # second group non-zero
    qw, sc = oracle.quantize_rtn_mse(bf16_bits(w))
    assert np.all(sc[0] == 0) and np.all(codes_of(qw)[:128] == 8)
    assert np.all(sc[1] != 0)


def test_outlier_worked_example_clips_at_seven_eighths():
    """127 weights of 5u and one of 8u, u = 2^-10.

    alpha = 1: s = RNE_bf16(8u/7) = 1.140625u; 5u -> round(4.38) = 4 -> 4.5625u,
    error 127 * 0.4375^2 u^2 = 24.3 u^2 (the outlier maps to 8u exactly).
    alpha = 7/8 (grid point 4): s = 0.875 * 8u / 7 = u exactly; the 127 weights
    are exact (code 5) and the outlier saturates at 7 -> 7u, error 1 u^2.
    Any smaller scale saturates the outlier below 7u (error > 1 u^2); any larger
    scale on the grid (1.0357u and up) puts error > 1 u^2 on the 127 weights.
    So: scale u, codes 13 for the 127 weights and 15 for the outlier."""
    u = 2.0 ** -10
    w = np.full((128, 1), 5 * u)
    w[37, 0] = 8 * u
    qw, sc = oracle.quantize_rtn_mse(bf16_bits(w))
    codes = codes_of(qw)[:, 0]
    assert sc[0, 0] == bf16_bits(u)
    assert codes[37] == 15
    assert np.all(np.delete(codes, 37) == 13)


def test_power_of_two_scaling_scales_only_the_scale():
    """x -> 4x is exact in bf16 and every step of the quantizer commutes with
    it (products, quotients and roundings scale exactly): same codes, scale
    exponent + 2."""
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((256, 24)) * 0.03).astype(np.float32)
    w[5, 3] = 0.4  # an outlier
    b = (w.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16
    w4 = (b.astype(np.uint32) << 16).view(np.float32) * 4.0
    qa, sa = oracle.quantize_rtn_mse(b)
    qb, sb = oracle.quantize_rtn_mse(bf16_bits(w4))
    assert np.array_equal(qa, qb)
    fa = (sa.astype(np.uint32) << 16).view(np.float32)
    fb = (sb.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(fa * 4.0, fb)


def test_sign_flip_mirrors_the_codes():
    """x -> -x: round-half-even and the clamp to [-7, 7] are odd functions, so
    q -> -q (code c -> 16 - c) and the scale is unchanged."""
    rng = np.random.default_rng(3)
    b = (((rng.standard_normal((256, 16)) * 0.02).astype(np.float32)).view(np.uint32) >> 16) \
        .astype(np.uint16)
    qa, sa = oracle.quantize_rtn_mse(b)
    qb, sb = oracle.quantize_rtn_mse(b ^ np.uint16(0x8000))
    assert np.array_equal(sa, sb)
    assert np.array_equal(codes_of(qb), 16 - codes_of(qa))


def test_codes_stay_in_the_symmetric_range():
    """Signed INT4 with -8 unused: stored codes 1 .. 15 (8 for exact zeros)."""
    rng = np.random.default_rng(4)
    b = (((rng.standard_normal((512, 40)) * 0.05).astype(np.float32)).view(np.uint32) >> 16) \
        .astype(np.uint16)
    qw, _ = oracle.quantize_rtn_mse(b)
    c = codes_of(qw)
    assert c.min() >= 1 and c.max() <= 15
