"""Guard bands and the debug build.

Every output buffer, every workspace and every input of every entry point
sits inside a larger device allocation whose bytes on both sides hold a
canary pattern.  After the call the canaries must be intact (nothing was
written outside the buffer), the inputs unchanged, the workspace all-zero
again (its documented contract) and the result within the oracle's bound.

The same calls then run through the debug build of the library
(W4A16_DEBUG), whose kernels check the index of every global copy, load and
store against the extent of its buffer and record W4A16_ERR_BOUNDS instead
of trapping: on small and odd shapes on every kernel path the status word
must stay OK.  A last test shrinks the extent the debug kernels are told
the codes have, so that their own checks trip, and checks that they report
it and that the context still computes correctly afterwards.
"""
import contextlib

import numpy as np
import pytest
import torch

import oracle
import weight_only_int4_gemm_gb300 as w
from tests.bf16_exact import bits_to_f64
from tests.gpu_util import assert_within_bound, bits
from weight_only_int4_gemm_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu

PAD = 4096        # canary bytes on each side (keeps the interior 256-byte aligned)
CANARY = 0xA5
STATUS_BOUNDS = 8


class Guarded:
    """A device buffer of `nbytes` with PAD canary bytes before and after it."""

    def __init__(self, nbytes: int, fill: torch.Tensor | int | None = None):
        self.nbytes = nbytes
        self.raw = torch.full((PAD + nbytes + PAD,), CANARY, dtype=torch.uint8, device="cuda")
        if isinstance(fill, torch.Tensor):
            self.raw[PAD:PAD + nbytes] = fill.contiguous().view(-1).view(torch.uint8)
        elif fill is not None:
            self.raw[PAD:PAD + nbytes] = fill

    @classmethod
    def holding(cls, t: torch.Tensor) -> "Guarded":
        g = cls(t.numel() * t.element_size(), t.cuda())
        g.dtype, g.shape = t.dtype, tuple(t.shape)
        g.saved = g.raw[PAD:PAD + g.nbytes].clone()
        return g

    def view(self, dtype=None, shape=None) -> torch.Tensor:
        dtype = dtype or self.dtype
        shape = shape or self.shape
        return self.raw[PAD:PAD + self.nbytes].view(dtype).view(shape)

    def check_canaries(self, what: str):
        head, tail = self.raw[:PAD], self.raw[PAD + self.nbytes:]
        assert bool((head == CANARY).all()), f"{what}: bytes written before the buffer"
        assert bool((tail == CANARY).all()), f"{what}: bytes written after the buffer"

    def check_unchanged(self, what: str):
        self.check_canaries(what)
        assert torch.equal(self.raw[PAD:PAD + self.nbytes], self.saved), f"{what}: input modified"


def workspace(nbytes: int) -> Guarded:
    return Guarded(max(nbytes, 16), 0)


def check_workspace(ws: Guarded):
    ws.check_canaries("workspace")
    assert int(ws.raw[PAD:PAD + ws.nbytes].count_nonzero()) == 0, "workspace not left zero"


def finish(lib_name: str):
    torch.cuda.synchronize()
    st = w.w4a16_device_status()
    assert st == 0, f"device status {st} on the {lib_name} build"


@pytest.fixture(scope="module")
def debug_built():
    from weight_only_int4_gemm_gb300 import build
    build.build_library(debug=True)
    assert _lib.load_debug().w4a16_debug_build() == 1
    assert _lib.load().w4a16_debug_build() == 0


@pytest.fixture(params=["release", "debug"])
def lib(request):
    """Runs the test body once on each build (the binding routed to it)."""
    if request.param == "debug":
        request.getfixturevalue("debug_built")
        with _lib.debug_library():
            w.w4a16_device_status()      # start from a clear word on this build
            yield "debug"
    else:
        yield "release"


def path_available(path: int) -> bool:
    return path != w.PATH_TCGEN05 or w.w4a16_select_path(4096, 4096, 4096) == w.PATH_TCGEN05


# --------------------------------------------------------------- plain GEMM

GEMM_CASES = [
    # B, K, N, zero-points, forced path (AUTO: skinny up to 16 rows, wide above)
    (1, 4096, 1032, False, w.PATH_AUTO),     # small-batch kernel, K split, ragged tile
    (3, 384, 72, True, w.PATH_AUTO),         # small-batch kernel, one partial tile
    (7, 128, 8, False, w.PATH_AUTO),         # a single group and an 8-column layer
    (16, 1024, 200, True, w.PATH_AUTO),      # 16-row tile, ragged columns
    (5, 1024, 264, False, w.PATH_TCGEN05),   # TMEM tensor-core kernel
    (16, 4096, 520, True, w.PATH_TCGEN05),   # TMEM tensor-core kernel, K split
    (17, 384, 64, False, w.PATH_AUTO),       # wide kernel, one row past a tile
    (64, 4096, 520, False, w.PATH_AUTO),     # wide kernel, K split
    (100, 1024, 264, True, w.PATH_AUTO),     # wide kernel, zero-points, ragged rows
    (257, 2048, 1032, False, w.PATH_AUTO),   # wide kernel, 128-row blocks + 1 row
    (40, 256, 8, False, w.PATH_AUTO),        # wide kernel, an 8-column layer
    (300, 512, 136, False, w.PATH_AUTO),     # wide kernel, tensor stores over a ragged edge
]


@pytest.mark.parametrize("B,K,N,zp,path", GEMM_CASES)
def test_gemm_guard_bands(lib, B, K, N, zp, path):
    if not path_available(path):
        pytest.skip("tensor-core kernel unavailable")
    p = inputs.make_problem(B, K, N, seed=B + K + N, zero_points=zp)
    packed = w.w4a16_pack(p.qweight.cuda(), None if p.qzeros is None else p.qzeros.cuda())
    x, pk, sc = Guarded.holding(p.x), Guarded.holding(packed.cpu()), Guarded.holding(p.scales)
    y = Guarded(B * N * 2)
    ws = workspace(w.w4a16_workspace_bytes(B, K, N))
    for _ in range(2):                  # the second call reuses the workspace
        w.w4a16_gemm(x.view(), pk.view(), sc.view(), zp, out=y.view(torch.bfloat16, (B, N)),
                     workspace=ws.view(torch.uint8, (ws.nbytes,)), path=path)
        finish(lib)
        y.check_canaries("y")
        check_workspace(ws)
    for g, name in ((x, "x"), (pk, "packed"), (sc, "scales")):
        g.check_unchanged(name)
    assert_within_bound(y.view(torch.bfloat16, (B, N)).cpu(), p)


@pytest.mark.parametrize("B,K,N", [(1, 1024, 264), (40, 512, 136)])
def test_static_scratch_guard_bands(lib, B, K, N):
    p = inputs.make_problem(B, K, N, seed=3 * B + N)
    g = p.to("cuda")
    packed = w.w4a16_pack(g.qweight)
    y = Guarded(B * N * 2)
    st = _lib.load().w4a16_gemm_static_scratch(
        g.x.data_ptr(), packed.data_ptr(), g.scales.data_ptr(), 0,
        y.view(torch.bfloat16, (B, N)).data_ptr(), B, K, N, 128, None)
    assert st == 0
    finish(lib)
    y.check_canaries("y")
    assert_within_bound(y.view(torch.bfloat16, (B, N)).cpu(), p)


# --------------------------------------------------------------- fused epilogue

@pytest.mark.parametrize("B,K,N,zp", [(3, 1024, 264, False), (40, 2048, 520, True),
                                      (200, 1024, 1032, False)])
@pytest.mark.parametrize("mode", [w.EPI_BIAS, w.EPI_BIAS | w.EPI_SILU_MUL])
def test_fused_guard_bands(lib, B, K, N, zp, mode):
    p = inputs.make_problem(B, K, N, seed=5 * B + N, zero_points=zp)
    bias = inputs.make_bias(N, 7)
    g = p.to("cuda")
    packed = w.w4a16_pack(g.qweight, g.qzeros)
    n_out = N // 2 if mode & w.EPI_SILU_MUL else N
    bz = Guarded.holding(bias)
    y = Guarded(B * n_out * 2)
    ws = workspace(w.w4a16_workspace_bytes(B, K, N))
    w.w4a16_gemm_fused(g.x, packed, g.scales, zp, mode, bz.view(),
                       out=y.view(torch.bfloat16, (B, n_out)),
                       workspace=ws.view(torch.uint8, (ws.nbytes,)))
    finish(lib)
    y.check_canaries("y")
    bz.check_unchanged("bias")
    check_workspace(ws)
    yo, _, bound = oracle.gemm_epilogue(bits(p.x), bits(p.qweight), bits(p.scales),
                                        None if p.qzeros is None else bits(p.qzeros),
                                        bias=bits(bias), mode=mode)
    yg = bits_to_f64(bits(y.view(torch.bfloat16, (B, n_out))))
    assert np.all(np.abs(yg - bits_to_f64(yo)) <= bound)


# --------------------------------------------------------------- grouped (MoE)

@pytest.mark.parametrize("counts,K,N,max_rows", [([0, 5, 17, 1, 0, 33], 1024, 264, 33),
                                                 ([1, 0, 2, 1], 4096, 520, 2),
                                                 ([40, 0, 70], 512, 136, 70)])
def test_grouped_guard_bands(lib, counts, K, N, max_rows):
    off = inputs.offsets_from_counts(counts)
    p = inputs.make_grouped_problem(off, K, N, 17 + K)
    g = p.to("cuda")
    E, T = len(counts), int(off[-1])
    packed = torch.stack([w.w4a16_pack(g.qweight[e]) for e in range(E)])
    pk, offs = Guarded.holding(packed.cpu()), Guarded.holding(off)
    y = Guarded(T * N * 2)
    ws = workspace(w.w4a16_grouped_workspace_bytes(T, E, max_rows, K, N))
    w.w4a16_gemm_grouped(g.x, offs.view(), pk.view(), g.scales, False, max_rows,
                         out=y.view(torch.bfloat16, (T, N)),
                         workspace=ws.view(torch.uint8, (ws.nbytes,)))
    finish(lib)
    y.check_canaries("y")
    pk.check_unchanged("packed")
    offs.check_unchanged("offsets")
    check_workspace(ws)
    yo, _, bound = oracle.gemm_grouped(bits(p.x), off.numpy(),
                                       [bits(p.qweight[e]) for e in range(E)],
                                       [bits(p.scales[e]) for e in range(E)])
    yg = bits_to_f64(bits(y.view(torch.bfloat16, (T, N))))
    assert np.all(np.abs(yg - bits_to_f64(yo)) <= bound)


# --------------------------------------------------------------- dequant, pack, quantize

@pytest.mark.parametrize("K,N,zp", [(128, 8, False), (384, 264, True)])
def test_pack_and_dequant_guard_bands(lib, K, N, zp):
    p = inputs.make_problem(1, K, N, seed=K + N, zero_points=zp)
    qw, qz = Guarded.holding(p.qweight), None if p.qzeros is None else Guarded.holding(p.qzeros)
    pk = Guarded(w.w4a16_packed_bytes(K, N, zp))
    w.w4a16_pack(qw.view(), None if qz is None else qz.view(),
                 out=pk.view(torch.uint8, (pk.nbytes,)))
    out = Guarded(K * N * 2)
    w.w4a16_dequant_ref(pk.view(torch.uint8, (pk.nbytes,)), p.scales.cuda(), zp, K,
                        out=out.view(torch.bfloat16, (K, N)))
    finish(lib)
    qw.check_unchanged("qweight")
    if qz is not None:
        qz.check_unchanged("qzeros")
    pk.check_canaries("packed")
    out.check_canaries("dequantised W")
    want = oracle.dequant(bits(p.qweight), bits(p.scales),
                          None if p.qzeros is None else bits(p.qzeros))
    assert np.array_equal(bits(out.view(torch.bfloat16, (K, N))), want)


@pytest.mark.parametrize("K,N", [(128, 8), (256, 264)])
def test_quantizer_guard_bands(lib, K, N):
    wt = inputs.make_dense_weight(K, N, 9)
    src = Guarded.holding(wt)
    qw, sc = Guarded(K // 8 * N * 4), Guarded(K // 128 * N * 2)
    st = _lib.load().w4a16_quantize_rtn(src.view().data_ptr(), K, N, 128,
                                        qw.view(torch.int32, (K // 8, N)).data_ptr(),
                                        sc.view(torch.bfloat16, (K // 128, N)).data_ptr(), None)
    assert st == 0
    finish(lib)
    src.check_unchanged("w")
    qw.check_canaries("qweight")
    sc.check_canaries("scales")
    qo, so = oracle.quantize_rtn_mse(bits(wt))
    assert np.array_equal(qw.view(torch.int32, (K // 8, N)).cpu().numpy().view(np.uint32), qo)
    assert np.array_equal(bits(sc.view(torch.bfloat16, (K // 128, N))), so)


# --------------------------------------------------------------- W8A8-FP8 path

@pytest.mark.parametrize("B,K,N", [(1, 1024, 264), (17, 2048, 520), (300, 512, 136)])
def test_fp8_guard_bands(lib, B, K, N):
    x = inputs.make_activations(B, K, 21 + B)
    wt = inputs.make_dense_weight(K, N, 23 + N)
    xq_o, sx_o = oracle.fp8_quantize_rows(bits(x))
    wq_o, sw_o = oracle.fp8_quantize_cols(bits(wt))
    xg = Guarded.holding(x)
    xq, sx = Guarded(B * K), Guarded(B * 4)
    w.w8a8_fp8_quantize_act(xg.view(), out=(xq.view(torch.uint8, (B, K)),
                                            sx.view(torch.float32, (B,))))
    packed = w.w8a8_fp8_pack_weight(torch.from_numpy(np.ascontiguousarray(wq_o)).cuda())
    y = Guarded(B * N * 2)
    ws = workspace(w.w8a8_fp8_workspace_bytes(B, K, N))
    w.w8a8_fp8_gemm(xq.view(torch.uint8, (B, K)), sx.view(torch.float32, (B,)), packed,
                    torch.from_numpy(sw_o).cuda(), out=y.view(torch.bfloat16, (B, N)),
                    workspace=ws.view(torch.uint8, (ws.nbytes,)))
    finish(lib)
    xg.check_unchanged("x")
    for g, name in ((xq, "xq"), (sx, "sx"), (y, "y")):
        g.check_canaries(name)
    check_workspace(ws)
    assert np.array_equal(xq.view(torch.uint8, (B, K)).cpu().numpy(), xq_o)
    yo, _, bound = oracle.fp8_gemm(xq_o, sx_o, wq_o, sw_o)
    yg = bits_to_f64(bits(y.view(torch.bfloat16, (B, N))))
    assert np.all(np.abs(yg - bits_to_f64(yo)) <= bound)


# --------------------------------------------------------------- debug checks fire

@contextlib.contextmanager
def shrunk_code_bound(nbytes: int):
    assert _lib.load().w4a16_debug_shrink_code_bound(nbytes) == 0
    try:
        yield
    finally:
        assert _lib.load().w4a16_debug_shrink_code_bound(0) == 0


@pytest.mark.parametrize("B,K,N,path", [(2, 1024, 264, w.PATH_AUTO),
                                        (8, 1024, 264, w.PATH_TCGEN05),
                                        (40, 1024, 264, w.PATH_AUTO)])
def test_debug_bounds_check_reports_and_context_survives(debug_built, B, K, N, path):
    """The kernels are told the codes end 16 bytes early: the copy of the
    last codes is then out of their bounds, so they skip it (the real buffer
    is never left) and report W4A16_ERR_BOUNDS; with the true extent back,
    the next call on the same context is correct and reports OK."""
    if not path_available(path):
        pytest.skip("tensor-core kernel unavailable")
    p = inputs.make_problem(B, K, N, seed=31 + B)
    g = p.to("cuda")
    with _lib.debug_library():
        assert w.w4a16_device_status() == 0
        packed = w.w4a16_pack(g.qweight)
        y = Guarded(B * N * 2)
        ws = workspace(w.w4a16_workspace_bytes(B, K, N))
        with shrunk_code_bound(16):
            w.w4a16_gemm(g.x, packed, g.scales, False, out=y.view(torch.bfloat16, (B, N)),
                         workspace=ws.view(torch.uint8, (ws.nbytes,)), path=path)
            assert w.w4a16_device_status() == STATUS_BOUNDS
        y.check_canaries("y")
        check_workspace(ws)
        w.w4a16_gemm(g.x, packed, g.scales, False, out=y.view(torch.bfloat16, (B, N)),
                     workspace=ws.view(torch.uint8, (ws.nbytes,)), path=path)
        finish("debug")
    assert_within_bound(y.view(torch.bfloat16, (B, N)).cpu(), p)


def test_release_build_refuses_the_debug_hook():
    assert _lib.load().w4a16_debug_build() == 0
    assert _lib.load().w4a16_debug_shrink_code_bound(16) == 4  # W4A16_ERR_UNSUPPORTED
