"""GPU parity: the CUDA library against the CPU oracle on identical seeded
inputs, through the C ABI (via its Python binding).

Bars: dequantised weights bit-exact; every GEMM output within
|y_gpu - y_oracle| <= 8e-3 * sum_k |x_k * w_kn| + 1e-6.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_int4_gemm_gb300 as w
from tests.bf16_exact import bits_to_f64
from tests.gpu_util import assert_within_bound, bits, oracle_gemm, sample_columns
from weight_only_int4_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

LAYER_SHAPES = {"qkv": (4096, 6144), "o_proj": (4096, 4096), "gate_up": (4096, 28672),
                "down": (14336, 4096)}


def available_paths():
    paths = [w.PATH_SKINNY]
    # the tensor-core path exists when the library reports it can select it
    if w.w4a16_select_path(4096, 4096, 4096) == w.PATH_TCGEN05:
        paths.append(w.PATH_TCGEN05)
    return paths


def run_gemm(p, path=w.PATH_AUTO):
    g = p.to("cuda")
    packed = w.w4a16_pack(g.qweight, g.qzeros)
    y = w.w4a16_gemm(g.x, packed, g.scales, g.qzeros is not None, path=path)
    torch.cuda.synchronize()
    assert w.w4a16_device_status() == 0
    return y.cpu()


# ------------------------------------------------------------ dequant, bit-exact

def _all_codes_by_all_scales():
    N = 0x10000
    qweight = np.full((16, N), 0x88888888, dtype=np.uint32)
    qweight[0, :] = 0x76543210
    qweight[1, :] = 0xFEDCBA98
    scale_bits = np.arange(N, dtype=np.uint32).astype(np.uint16)
    finite = np.isfinite(bits_to_f64(scale_bits))
    scales = np.where(finite, scale_bits, 0).astype(np.uint16)[None, :]
    return qweight, scales, finite


def _gpu_dequant(qweight, scales, qzeros=None):
    K = qweight.shape[0] * 8
    qw = torch.from_numpy(qweight.view(np.int32)).cuda()
    sc = torch.from_numpy(scales.view(np.int16)).view(torch.bfloat16).cuda()
    qz = None if qzeros is None else torch.from_numpy(qzeros.view(np.int32)).cuda()
    packed = w.w4a16_pack(qw, qz)
    out = w.w4a16_dequant_ref(packed, sc, qz is not None, K)
    torch.cuda.synchronize()
    return bits(out)


def test_dequant_exhaustive_symmetric_bit_exact():
    qweight, scales, finite = _all_codes_by_all_scales()
    got = _gpu_dequant(qweight, scales)
    want = oracle.dequant(qweight, scales)
    mism = (got != want)[:, finite]
    assert not mism.any(), f"{int(mism.sum())} mismatching weights"


def test_dequant_exhaustive_zero_points_bit_exact():
    qweight, scales, finite = _all_codes_by_all_scales()
    for z in range(16):
        qzeros = np.full((1, 0x10000 // 8), z * 0x11111111, dtype=np.uint32)
        got = _gpu_dequant(qweight, scales, qzeros)
        want = oracle.dequant(qweight, scales, qzeros)
        mism = (got != want)[:, finite]
        assert not mism.any(), f"z={z}: {int(mism.sum())} mismatching weights"


@pytest.mark.parametrize("zp", [False, True])
@pytest.mark.parametrize("K,N", [(128, 8), (384, 264), (4096, 4104)])
def test_dequant_random_layers_bit_exact(K, N, zp):
    p = inputs.make_problem(1, K, N, seed=K + N, zero_points=zp)
    qw, sc = bits(p.qweight), bits(p.scales)
    qz = None if p.qzeros is None else bits(p.qzeros)
    np.testing.assert_array_equal(_gpu_dequant(qw, sc, qz), oracle.dequant(qw, sc, qz))


# ------------------------------------------------------------ GEMM, small shapes

SMALL = [(1, 128, 8), (2, 256, 16), (3, 384, 24), (5, 128, 72), (8, 512, 64), (9, 256, 136),
         (16, 1024, 200), (17, 384, 64), (33, 256, 40), (64, 512, 128), (100, 384, 264),
         (257, 256, 136),
         # outputs narrower than one 32-column store box on the tensor-core path
         (40, 256, 8), (24, 128, 16), (100, 384, 24)]


@pytest.mark.parametrize("zp", [False, True])
@pytest.mark.parametrize("B,K,N", SMALL)
def test_gemm_small_shapes_all_paths(B, K, N, zp):
    p = inputs.make_problem(B, K, N, seed=B * 7 + K + N, zero_points=zp)
    for path in [w.PATH_AUTO] + available_paths():
        assert_within_bound(run_gemm(p, path), p)


@pytest.mark.parametrize("zp", [False, True])
@pytest.mark.parametrize("B,K,N", [(1, 4096, 4096), (16, 4096, 264), (40, 1024, 520), (300, 512, 392)])
def test_gemm_integer_case_is_bit_exact(B, K, N, zp):
    """Unit scales and integer x in [-4, 4]: every partial sum is an integer
    below 2^24, so any fp32 accumulation order is exact and the GPU result
    must equal the oracle's bit for bit."""
    p = inputs.make_problem(B, K, N, seed=99, zero_points=zp)
    gen = torch.Generator().manual_seed(5)
    xi = torch.randint(-4, 5, (B, K), generator=gen).to(torch.bfloat16)
    p = inputs.LinearProblem(xi, p.qweight, torch.ones_like(p.scales), p.qzeros)
    y_o, acc, _ = oracle_gemm(p)
    assert np.all(np.abs(acc) < 2 ** 24)
    for path in available_paths():
        np.testing.assert_array_equal(bits(run_gemm(p, path)), y_o, err_msg=f"path {path}")


# ------------------------------------------------------------ workload-sized parity

def test_single_linear_4096_b1_seed0_full():
    """Single linear 4096 -> 4096 at B = 1, seed 0: every output."""
    p = inputs.make_problem(1, 4096, 4096, seed=0)
    assert_within_bound(run_gemm(p), p)


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16])
def test_decoder_layer_linear_set_full(B):
    """One Llama-3-8B decoder layer's four linears at decode: every output."""
    for i, (name, (K, N)) in enumerate(LAYER_SHAPES.items()):
        p = inputs.make_problem(B, K, N, seed=1000 + 10 * i)
        assert_within_bound(run_gemm(p), p)


@pytest.mark.parametrize("B", [1, 4, 8, 12, 16, 64, 128, 256, 270, 384, 512, 1024])
def test_lm_head_sampled_columns(B):
    """4096 -> 128256 lm_head (largest N) at every batch of the decode-step
    sweep and at 8 and 12 rows (both kernels, full and ragged batch tiles):
    sampled columns, all rows."""
    p = inputs.make_problem(B, 4096, 128256, seed=77)
    y = run_gemm(p)
    assert_within_bound(y, p, cols=sample_columns(128256, 96 if B > 64 else 384))


def boundary_rows(B: int, step: int = 16) -> np.ndarray:
    """The first and last row of every `step`-row block of the batch (every
    batch tile of the tensor-core kernels starts on a multiple of 16 rows),
    and the last row of the ragged final block."""
    rows = {0, B - 1}
    for r in range(0, B, step):
        rows |= {r, min(B - 1, r + step - 1)}
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("B", [17, 64, 128, 256, 270, 384, 512, 1024])
def test_lm_head_every_column_on_tile_boundary_rows(B):
    """4096 -> 128256 lm_head on the tensor-core kernels: every one of the
    128256 columns (every column tile, the persistent scheduler's every item
    and K split), on the first and last rows of every 16-row block."""
    p = inputs.make_problem(B, 4096, 128256, seed=77)
    y = run_gemm(p)
    assert_within_bound(y, p, rows=boundary_rows(B, 16 if B <= 384 else 32))


@pytest.mark.parametrize("name", ["qkv", "gate_up", "down"])
def test_prefill_m2048_every_column_on_tile_boundary_rows(name):
    K, N = LAYER_SHAPES[name]
    p = inputs.make_problem(2048, K, N, seed=4000 + K + N, outlier_frac=0.01)
    y = run_gemm(p)
    assert_within_bound(y, p, rows=boundary_rows(2048, 64))


@pytest.mark.parametrize("B", [64, 512])
@pytest.mark.parametrize("K,N", [(8192, 10240), (8192, 57344), (28672, 8192)])
def test_zero_point_70b_every_column_on_tile_boundary_rows(K, N, B):
    p = inputs.make_problem(B, K, N, seed=5000 + K + N, zero_points=True)
    y = run_gemm(p)
    assert_within_bound(y, p, rows=boundary_rows(B, 16 if B <= 64 else 64))


@pytest.mark.parametrize("name", ["qkv", "gate_up", "down"])
def test_prefill_m2048_with_outliers_sampled(name):
    K, N = LAYER_SHAPES[name]
    p = inputs.make_problem(2048, K, N, seed=4000 + K + N, outlier_frac=0.01)
    y = run_gemm(p)
    assert_within_bound(y, p, cols=sample_columns(N, 64))


@pytest.mark.parametrize("B", [1, 64, 512])
@pytest.mark.parametrize("K,N", [(8192, 10240), (8192, 57344), (28672, 8192)])
def test_zero_point_70b_shapes_sampled(K, N, B):
    p = inputs.make_problem(B, K, N, seed=5000 + K + N, zero_points=True)
    y = run_gemm(p)
    assert_within_bound(y, p, cols=sample_columns(N, 64 if B >= 512 else 192))


# ------------------------------------------------------------ behaviour

def test_repeated_calls_reuse_workspace_across_shapes():
    """One workspace shared by calls of different shapes and paths: every call
    leaves it zeroed, so every result stays within the bound."""
    p = inputs.make_problem(4, 4096, 4096, seed=3)
    g = p.to("cuda")
    packed = w.w4a16_pack(g.qweight)
    ys = [w.w4a16_gemm(g.x, packed, g.scales, False).clone() for _ in range(3)]
    q = inputs.make_problem(64, 4096, 4096, seed=4).to("cuda")         # tensor-core split-K
    w.w4a16_gemm(q.x, w.w4a16_pack(q.qweight), q.scales, False)
    r = inputs.make_problem(2, 14336, 4096, seed=5).to("cuda")         # small-batch split-K
    w.w4a16_gemm(r.x, w.w4a16_pack(r.qweight), r.scales, False)
    ys.append(w.w4a16_gemm(g.x, packed, g.scales, False))
    torch.cuda.synchronize()
    assert w.w4a16_device_status() == 0
    for y in ys:
        assert_within_bound(y.cpu(), p)


def test_without_split_k_results_are_bit_identical():
    """A shape that needs no K split has one summation order: repeated calls
    are bit-identical."""
    B, K, N = 8, 1024, 128256
    assert w.w4a16_workspace_bytes(B, K, N) <= 65536   # counters only, no accumulator
    g = inputs.make_problem(B, K, N, seed=6).to("cuda")
    packed = w.w4a16_pack(g.qweight)
    ys = [w.w4a16_gemm(g.x, packed, g.scales, False).clone() for _ in range(3)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))


def test_output_guard_band_untouched():
    B, K, N = 3, 1024, 200
    p = inputs.make_problem(B, K, N, seed=8).to("cuda")
    packed = w.w4a16_pack(p.qweight)
    buf = torch.full((B * N + 4096,), 12345, dtype=torch.int16, device="cuda")
    y = buf[:B * N].view(torch.bfloat16).view(B, N)
    w.w4a16_gemm(p.x, packed, p.scales, False, out=y)
    torch.cuda.synchronize()
    assert torch.all(buf[B * N:] == 12345)
    assert_within_bound(y.cpu(), p.to("cpu"))


def test_runs_on_a_side_stream():
    p = inputs.make_problem(8, 2048, 1024, seed=9).to("cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        packed = w.w4a16_pack(p.qweight)
        y = w.w4a16_gemm(p.x, packed, p.scales, False)
    s.synchronize()
    assert_within_bound(y.cpu(), p.to("cpu"))


def test_workspace_validation_on_tensor_core_split():
    """A tensor-core shape that splits K needs workspace: missing / too small."""
    B, K, N = 64, 4096, 4096
    need = w.w4a16_workspace_bytes(B, K, N)
    if w.PATH_TCGEN05 not in available_paths() or need == 0:
        pytest.skip("no split-K tensor-core plan for this shape on this device")
    lib = w.load()
    p = inputs.make_problem(B, K, N, seed=12).to("cuda")
    packed = w.w4a16_pack(p.qweight)
    y = torch.empty((B, N), dtype=torch.bfloat16, device="cuda")
    args = (p.x.data_ptr(), packed.data_ptr(), p.scales.data_ptr(), 0, y.data_ptr(), B, K, N, 128)
    assert lib.w4a16_gemm_path(*args, None, 0, w.PATH_TCGEN05, None) == 1          # NULL
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    assert lib.w4a16_gemm_path(*args, ws.data_ptr(), need - 1, w.PATH_TCGEN05, None) == 5  # WORKSPACE
    assert lib.w4a16_gemm_path(*args, ws.data_ptr(), need, w.PATH_TCGEN05, None) == 0
    torch.cuda.synchronize()
    assert_within_bound(y.cpu(), p.to("cpu"), cols=sample_columns(N, 64))


def test_bounded_wait_expires_cleanly_and_context_survives():
    """A wait that nothing satisfies expires after ~50 ms: the status word says
    TIMEOUT, y is untouched, and the next GEMM on the same context is correct.
    The shape splits K, so the call owns a workspace; after the timeout the
    workspace is zero-filled again (the header's rule after a TIMEOUT) and
    reused by the next call, which must then be within the bound."""
    if w.PATH_TCGEN05 not in available_paths():
        pytest.skip("tensor-core kernel unavailable")
    assert w.w4a16_device_status(clear=True) == 0
    B, K, N = 64, 1024, 256
    need = w.w4a16_workspace_bytes(B, K, N)
    assert need > 0, "expected a split-K plan for this shape"
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    p = inputs.make_problem(B, K, N, seed=13).to("cuda")
    packed = w.w4a16_pack(p.qweight)
    y = torch.full((B, N), 7.0, dtype=torch.bfloat16, device="cuda")
    assert w.w4a16_debug_forced_timeout(p.x, packed, p.scales, False, y, wait_ms=50,
                                        workspace=ws) == 0
    torch.cuda.synchronize()
    assert w.w4a16_device_status(clear=True) == 7
    assert torch.all(y == 7.0)
    assert w.w4a16_device_status(clear=False) == 0
    ws.zero_()
    for _ in range(2):
        y2 = w.w4a16_gemm(p.x, packed, p.scales, False, path=w.PATH_TCGEN05, workspace=ws)
        torch.cuda.synchronize()
        assert w.w4a16_device_status() == 0
        assert_within_bound(y2.cpu(), p.to("cpu"))
    # a completed call leaves its workspace all-zero again
    assert int(torch.count_nonzero(ws)) == 0
