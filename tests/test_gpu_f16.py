"""GPU parity of the fp16-activation variant (w4a16_gemm_f16,
w4a16_dequant_ref_f16) against the fp16 oracle, through the C ABI, on every
kernel path.

Bars: the dequantised fp16 weights bit-exact; every GEMM output within
|y_gpu - y_oracle| <= 2e-3 * sum|x*w| + 2^-24 * (1 + sum|x|) (the fp16
oracle's bound: two fp16 unit roundoffs, fp32 accumulation, one subnormal
step per unit of sum|x|).
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_int4_gemm_gb300 as w
from tests.f16_exact import f16_bits_to_f64
from tests.gpu_util import bits, sample_columns
from weight_only_int4_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

F16 = torch.float16


def paths():
    out = [w.PATH_AUTO, w.PATH_SKINNY]
    if w.w4a16_select_path(4096, 4096, 4096) == w.PATH_TCGEN05:
        out.append(w.PATH_TCGEN05)
    return out


def run(p, path=w.PATH_AUTO, workspace=None):
    g = p.to("cuda")
    packed = w.w4a16_pack(g.qweight, g.qzeros)
    y = w.w4a16_gemm_f16(g.x, packed, g.scales, g.qzeros is not None, path=path,
                         workspace=workspace)
    torch.cuda.synchronize()
    assert w.w4a16_device_status() == 0
    return y.cpu()


def check(y, p, cols=None, rows=None):
    if rows is not None:
        idx = torch.as_tensor(np.asarray(rows), dtype=torch.long)
        p = inputs.LinearProblem(p.x[idx], p.qweight, p.scales, p.qzeros)
        y = y[idx]
    yo, _, bound = oracle.gemm_f16(bits(p.x), bits(p.qweight), bits(p.scales),
                                   None if p.qzeros is None else bits(p.qzeros), cols=cols)
    yg = f16_bits_to_f64(bits(y))
    if cols is not None:
        yg = yg[:, cols]
    yo = f16_bits_to_f64(yo)
    assert np.all(np.isfinite(yg)), "non-finite GPU output"
    bad = np.abs(yg - yo) > bound
    if bad.any():
        b, n = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} of {bad.size} outside the bound; first at "
                             f"({b}, {n}): gpu={yg[b, n]!r} oracle={yo[b, n]!r} "
                             f"bound={bound[b, n]!r}")


# ------------------------------------------------------------ dequant, bit-exact

def _gpu_dequant_f16(qweight, scales, qzeros=None):
    K = qweight.shape[0] * 8
    qw = torch.from_numpy(qweight.view(np.int32)).cuda()
    sc = torch.from_numpy(scales.view(np.int16)).view(F16).cuda()
    qz = None if qzeros is None else torch.from_numpy(qzeros.view(np.int32)).cuda()
    packed = w.w4a16_pack(qw, qz)
    out = w.w4a16_dequant_ref_f16(packed, sc, qz is not None, K)
    torch.cuda.synchronize()
    return bits(out)


def test_dequant_every_code_times_every_finite_fp16_scale():
    allb = np.arange(0x10000, dtype=np.uint32)
    finite = np.isfinite(f16_bits_to_f64(allb))
    N = 0x10000
    qweight = np.full((16, N), 0x88888888, dtype=np.uint32)
    qweight[0, :] = 0x76543210
    qweight[1, :] = 0xFEDCBA98
    scales = np.where(finite, allb, 0).astype(np.uint16)[None, :]
    for z in (None, 0, 5, 15):
        qzeros = None if z is None else np.full((1, N // 8), z * 0x11111111, dtype=np.uint32)
        got = _gpu_dequant_f16(qweight, scales, qzeros)
        want = oracle.dequant_f16(qweight, scales, qzeros)
        mism = (got != want)[:, finite]
        assert not mism.any(), f"z={z}: {int(mism.sum())} mismatching weights"


@pytest.mark.parametrize("zp", [False, True])
def test_dequant_random_layer_bit_exact(zp):
    p = inputs.make_problem(1, 4096, 4104, seed=3, zero_points=zp, dtype=F16)
    qw, sc = bits(p.qweight), bits(p.scales)
    qz = None if p.qzeros is None else bits(p.qzeros)
    np.testing.assert_array_equal(_gpu_dequant_f16(qw, sc, qz), oracle.dequant_f16(qw, sc, qz))


# ------------------------------------------------------------ GEMM

SMALL = [(1, 128, 8), (3, 384, 24), (8, 512, 64), (9, 256, 136), (16, 1024, 200),
         (17, 384, 64), (64, 512, 128), (100, 384, 264), (257, 256, 136)]


@pytest.mark.parametrize("zp", [False, True])
@pytest.mark.parametrize("B,K,N", SMALL)
def test_gemm_small_shapes_every_path(B, K, N, zp):
    p = inputs.make_problem(B, K, N, seed=B * 5 + K + N, zero_points=zp, dtype=F16)
    for path in paths():
        check(run(p, path), p)


@pytest.mark.parametrize("B,K,N", [(1, 4096, 4096), (16, 4096, 264), (40, 1024, 520),
                                   (300, 512, 392)])
def test_gemm_integer_case_is_bit_exact(B, K, N):
    """Integer x in [-4, 4] and power-of-two scales: every product and partial
    sum is exact in fp32, so every path must equal the oracle bit for bit."""
    g = torch.Generator().manual_seed(B + N)
    x = torch.randint(-4, 5, (B, K), generator=g).to(F16)
    qw, _, _ = inputs.make_weights(K, N, seed=N)
    sc = torch.pow(2.0, torch.randint(-4, 1, (K // 128, N), generator=g).float()).to(F16)
    p = inputs.LinearProblem(x, qw, sc, None)
    yo, _, _ = oracle.gemm_f16(bits(x), bits(qw), bits(sc))
    for path in paths():
        np.testing.assert_array_equal(bits(run(p, path)), yo, err_msg=f"path {path}")


@pytest.mark.parametrize("B", [1, 16, 64, 512])
@pytest.mark.parametrize("K,N", [(4096, 6144), (14336, 4096)])
def test_decoder_shapes_full_columns_on_boundary_rows(B, K, N):
    p = inputs.make_problem(B, K, N, seed=K + B, dtype=F16)
    y = run(p)
    rows = sorted({0, B - 1} | {r for r in range(0, B, 128)} | {min(B - 1, r + 127)
                                                               for r in range(0, B, 128)})
    check(y, p, rows=rows)
    check(y, p, cols=sample_columns(N, 64, seed=B))


@pytest.mark.parametrize("B", [1, 64, 512])
def test_zero_points_70b_shape_sampled(B):
    K, N = 8192, 10240
    p = inputs.make_problem(B, K, N, seed=B + 7, zero_points=True, dtype=F16)
    check(run(p), p, cols=sample_columns(N, 96, seed=B))


def test_outliers_and_repeated_calls_reuse_the_workspace():
    p = inputs.make_problem(64, 4096, 1032, seed=21, outlier_frac=0.01, dtype=F16)
    ws = torch.zeros(max(16, w.w4a16_workspace_bytes(64, 4096, 1032)), dtype=torch.uint8,
                     device="cuda")
    for _ in range(2):
        check(run(p, workspace=ws), p)
    assert int(ws.count_nonzero()) == 0


def test_bf16_and_fp16_entry_points_agree_where_both_are_exact():
    """Integer activations and power-of-two scales are exact in both formats:
    w4a16_gemm and w4a16_gemm_f16 give the same values."""
    B, K, N = 8, 1024, 264
    g = torch.Generator().manual_seed(5)
    xi = torch.randint(-3, 4, (B, K), generator=g).float()
    qw, _, _ = inputs.make_weights(K, N, seed=9)
    s = torch.pow(2.0, torch.randint(-3, 0, (K // 128, N), generator=g).float())
    packed = w.w4a16_pack(qw.cuda())
    yb = w.w4a16_gemm(xi.to(torch.bfloat16).cuda(), packed, s.to(torch.bfloat16).cuda(), False)
    yh = w.w4a16_gemm_f16(xi.to(F16).cuda(), packed, s.to(F16).cuda(), False)
    torch.cuda.synchronize()
    # sums are multiples of 1/8; below 32 they are exact in bf16 (8 significand
    # bits) as well as in fp16
    exact_small = yh.float().abs() < 32
    assert torch.equal(yb.float()[exact_small], yh.float()[exact_small])


def test_fp16_entry_point_validation():
    lib = w.load()
    B, K, N = 2, 128, 8
    x = torch.zeros((B, K), dtype=F16, device="cuda")
    packed = torch.zeros(w.w4a16_packed_bytes(K, N, False), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((1, N), dtype=F16, device="cuda")
    y = torch.zeros((B, N), dtype=F16, device="cuda")
    assert lib.w4a16_gemm_f16(x.data_ptr(), packed.data_ptr(), sc.data_ptr(), 0, y.data_ptr(),
                              B, K, N, 64, None, 0, None) == 4   # UNSUPPORTED group size
    assert lib.w4a16_gemm_f16(x.data_ptr(), packed.data_ptr(), sc.data_ptr(), 0, y.data_ptr(),
                              B, 100, N, 128, None, 0, None) == 2  # SHAPE
    assert lib.w4a16_gemm_f16(None, packed.data_ptr(), sc.data_ptr(), 0, y.data_ptr(),
                              B, K, N, 128, None, 0, None) == 1   # NULL
    assert lib.w4a16_dequant_ref_f16(packed.data_ptr() + 2, sc.data_ptr(), 0, y.data_ptr(),
                                     K, N, 128, None) == 3        # ALIGN
