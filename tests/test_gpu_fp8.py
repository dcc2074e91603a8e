"""GPU parity of the W8A8-FP8 comparison path against the oracle, through the
C ABI: the two quantisers bit-exact (codes and binary32 scales), the GEMM
within |y_gpu - y_oracle| <= 8e-3 * sum_k |x^ w^| + 1e-6 (x^, w^ the
dequantised operands), and bit-exact where fp32 accumulation is exact.
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


def gpu_act(x):
    xq, sx = w.w8a8_fp8_quantize_act(x.cuda())
    torch.cuda.synchronize()
    return xq.cpu().numpy(), sx.cpu().numpy()


def gpu_weight(wt):
    wq, sw = w.w8a8_fp8_quantize_weight(wt.cuda())
    torch.cuda.synchronize()
    return wq.cpu().numpy(), sw.cpu().numpy()


@pytest.mark.parametrize("B,K,outl", [(1, 128, 0.0), (7, 4096, 0.0), (33, 14336, 0.01)])
def test_activation_quantizer_bit_exact(B, K, outl):
    x = inputs.make_activations(B, K, 3 + B, outlier_frac=outl)
    if B > 1:
        x[1] = 0                       # an all-zero token
        x[2, : K // 2] *= 1e-6         # codes down in the subnormal range and zeros
    xq, sx = gpu_act(x)
    oq, osx = oracle.fp8_quantize_rows(bits(x))
    assert np.array_equal(sx.view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(xq, oq)


@pytest.mark.parametrize("K,N", [(128, 8), (4096, 264), (1024, 1000)])
def test_weight_quantizer_bit_exact(K, N):
    wt = inputs.make_dense_weight(K, N, 5)
    wt[:, 3] = 0                       # an all-zero channel
    wq, sw = gpu_weight(wt)
    oq, osw = oracle.fp8_quantize_cols(bits(wt))
    assert np.array_equal(sw.view(np.uint32), osw.view(np.uint32))
    assert np.array_equal(wq, oq)


def check_gemm(xq, sx, wq, sw, cols=None, exact=False):
    packed = w.w8a8_fp8_pack_weight(torch.from_numpy(np.ascontiguousarray(wq)).cuda())
    y = w.w8a8_fp8_gemm(torch.from_numpy(xq).cuda(), torch.from_numpy(sx).cuda(),
                        packed, torch.from_numpy(sw).cuda())
    torch.cuda.synchronize()
    assert w.w4a16_device_status() == 0
    yo, _, bound = oracle.fp8_gemm(xq, sx, wq, sw, cols=cols)
    yg = bits(y)
    if cols is not None:
        yg = yg[:, cols]
    if exact:
        assert np.array_equal(yg, yo)
        return
    g, o = bits_to_f64(yg), bits_to_f64(yo)
    assert np.all(np.isfinite(g))
    bad = np.abs(g - o) > bound
    assert not bad.any(), f"{int(bad.sum())} outputs outside the bound"


@pytest.mark.parametrize("B,K,N", [(1, 4096, 4096), (16, 4096, 6144), (17, 1024, 520),
                                   (5, 128, 8), (300, 2048, 1032), (64, 14336, 4096)])
def test_gemm_against_oracle(B, K, N):
    x = inputs.make_activations(B, K, 11 + B, outlier_frac=0.01)
    wt = inputs.make_dense_weight(K, N, 13 + N)
    xq, sx = oracle.fp8_quantize_rows(bits(x))
    wq, sw = oracle.fp8_quantize_cols(bits(wt))
    cols = None if B * K * N <= 2 ** 33 else sample_columns(N, 256, 1)
    check_gemm(xq, sx, wq, sw, cols=cols)


@pytest.mark.parametrize("B,K,N", [(3, 4096, 4096), (40, 2048, 1032), (520, 1024, 264)])
def test_gemm_bit_exact_on_integer_codes(B, K, N):
    """Codes of the integers -16..16 (exact in E4M3) and power-of-two scales:
    every fp32 partial sum is an integer below 2^24, so the tensor-core sum is
    exact in any order and y must equal the oracle's bit for bit."""
    rng = np.random.default_rng(B)
    ints = np.array([oracle.e4m3_from_double(v) for v in range(-16, 17)], dtype=np.uint8)
    xq = rng.choice(ints, size=(B, K))
    wq = rng.choice(ints, size=(N, K))
    sx = np.exp2(rng.integers(-6, 3, B)).astype(np.float32)
    sw = np.exp2(rng.integers(-12, -4, N)).astype(np.float32)
    check_gemm(xq, sx, wq, sw, exact=True)
    check_gemm(xq, sx, wq, sw, exact=True)  # the split-K workspace is clean again


@pytest.mark.parametrize("K,N", [(128, 8), (1024, 264), (256, 1000)])
def test_pack_layout(K, N):
    """The packed weight blocks hold exactly the codes, tiled and swizzled:
    checked by rebuilding the blocks on the host from the layout's definition."""
    rng = np.random.default_rng(K + N)
    wq = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    got = w.w8a8_fp8_pack_weight(torch.from_numpy(wq).cuda()).cpu().numpy()
    tiles, nkb = -(-N // 128), K // 128
    want = np.zeros((tiles, nkb, 128, 8, 16), dtype=np.uint8)
    pad = np.zeros((tiles * 128, K), dtype=np.uint8)
    pad[:N] = wq
    src = pad.reshape(tiles, 128, nkb, 8, 16).transpose(0, 2, 1, 3, 4)  # [t][kb][r][c][16]
    for c in range(8):
        for r in range(128):
            want[:, :, r, c ^ (r & 7)] = src[:, :, r, c]
    assert np.array_equal(got, want.reshape(-1))


def test_pipeline_on_the_gpu():
    """Both quantisers and the GEMM on the device, the oracle's chain beside it."""
    B, K, N = 24, 4096, 4096
    x = inputs.make_activations(B, K, 21, outlier_frac=0.01)
    wt = inputs.make_dense_weight(K, N, 22)
    xq, sx = w.w8a8_fp8_quantize_act(x.cuda())
    wq, sw = w.w8a8_fp8_quantize_weight(wt.cuda())
    y = w.w8a8_fp8_gemm(xq, sx, w.w8a8_fp8_pack_weight(wq), sw)
    torch.cuda.synchronize()
    assert w.w4a16_device_status() == 0
    oxq, osx = oracle.fp8_quantize_rows(bits(x))
    owq, osw = oracle.fp8_quantize_cols(bits(wt))
    assert np.array_equal(xq.cpu().numpy(), oxq) and np.array_equal(wq.cpu().numpy(), owq)
    cols = sample_columns(N, 512, 2)
    yo, _, bound = oracle.fp8_gemm(oxq, osx, owq, osw, cols=cols)
    g, o = bits_to_f64(bits(y))[:, cols], bits_to_f64(yo)
    assert np.all(np.abs(g - o) <= bound)
