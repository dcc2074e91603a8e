"""Pins for the oracle's mixture-of-experts GEMM (``oracle.gemm_grouped``;
"When quantization pays -- and when it does not", section "The three
regimes", mixture-of-experts paragraphs: each routed expert multiplies only
the rows sent to it).

The expected values are closed forms: expert e's codes are a known constant
per column, every scale is 1 and x is all ones, so row r of y is exactly
K * (code - zero) of the expert that owns r.  A wrong expert index, an
off-by-one in the row ranges or a dropped empty expert changes a value.
"""
import numpy as np
import pytest

import oracle

ONE_BF16 = 0x3F80


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def expert_tables(E, K, N, code_of, zero_of=None):
    """Canonical qweight / scales / qzeros per expert with constant codes per column."""
    qw = np.zeros((E, K // 8, N), dtype=np.uint32)
    for e in range(E):
        for n in range(N):
            c = code_of(e, n)
            qw[e, :, n] = sum(c << (4 * j) for j in range(8))
    sc = np.full((E, K // 128, N), ONE_BF16, dtype=np.uint16)
    qz = None
    if zero_of is not None:
        qz = np.zeros((E, K // 128, N // 8), dtype=np.uint32)
        for e in range(E):
            for n in range(N):
                qz[e, :, n // 8] |= np.uint32(zero_of(e, n) << (4 * (n % 8)))
    return qw, sc, qz


def bf16_value(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("zp", [False, True])
def test_rows_get_their_experts_closed_form(zp):
    E, K, N = 5, 128, 16
    counts = [2, 0, 3, 1, 0]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(offsets[-1])

    def code_of(e, n):
        return (3 * e + n) % 16

    def zero_of(e, n):
        return (e + 2 * n) % 16

    qw, sc, qz = expert_tables(E, K, N, code_of, zero_of if zp else None)
    x = np.full((T, K), ONE_BF16, dtype=np.uint16)
    y, acc, _ = oracle.gemm_grouped(x, offsets, qw, sc, qz)
    owner = np.repeat(np.arange(E), counts)
    for r in range(T):
        e = owner[r]
        for n in range(N):
            want = K * (code_of(e, n) - (zero_of(e, n) if zp else 8))
            assert acc[r, n] == want
            assert bf16_value(y[r, n]) == want  # |want| <= 1920 = 15 * 128 is exact in bf16


def test_single_expert_is_the_plain_gemm_and_columns_subset():
    """E = 1 covers every row with one weight set: the plain GEMM (itself pinned
    by the oracle's own tests); a column subset returns those columns."""
    rng = np.random.default_rng(7)
    K, N, T = 256, 24, 5
    qw = rng.integers(0, 2**32, size=(1, K // 8, N), dtype=np.uint32)
    sc = ((np.abs(rng.standard_normal((1, K // 128, N))) * 0.02).astype(np.float32)
          .view(np.uint32) >> 16).astype(np.uint16)
    x = ((rng.standard_normal((T, K))).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    y, acc, bound = oracle.gemm_grouped(x, np.array([0, T], dtype=np.int32), qw, sc)
    y1, acc1, bound1 = oracle.gemm(x, qw[0], sc[0])
    assert np.array_equal(y, y1) and np.array_equal(acc, acc1) and np.array_equal(bound, bound1)
    cols = np.array([0, 5, 23], dtype=np.int32)
    yc, _, _ = oracle.gemm_grouped(x, np.array([0, T], dtype=np.int32), qw, sc, cols=cols)
    assert np.array_equal(yc, y[:, cols])


def test_malformed_offsets_are_rejected():
    qw, sc, _ = expert_tables(2, 128, 8, lambda e, n: 8)
    x = np.zeros((3, 128), dtype=np.uint16)
    with pytest.raises(AssertionError):
        oracle.gemm_grouped(x, np.array([0, 2, 1], dtype=np.int32), qw, sc)
    with pytest.raises(AssertionError):
        oracle.gemm_grouped(x, np.array([0, 1, 2], dtype=np.int32), qw, sc)
