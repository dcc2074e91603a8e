"""The allocation-free GEMM entry point (w4a16_gemm_static_scratch).

Callers that cannot allocate device memory use this entry point; its split-K
scratch is a device array inside the library.  Here it is called through the
C ABI, twice in a row on the same inputs, and each result is checked against
the regular entry point (w4a16_gemm with a caller-allocated workspace) and
against the CPU oracle's error bound.  This file is collected last on
purpose, and passes both alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import weight_only_int4_gemm_gb300 as w
from tests.bf16_exact import bits_to_f64
from tests.gpu_util import assert_within_bound, bits, oracle_gemm
from weight_only_int4_gemm_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu


def _static_gemm(x, packed, scales, has_zeros, y, stream):
    B, K = x.shape
    N = scales.shape[1]
    return _lib.load().w4a16_gemm_static_scratch(
        x.data_ptr(), packed.data_ptr(), scales.data_ptr(), 1 if has_zeros else 0,
        y.data_ptr(), B, K, N, 128, ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("B,K,N,zp", [(4, 4096, 4096, False), (1, 14336, 4096, True),
                                      (16, 4096, 6144, False), (64, 4096, 1024, False)])
def test_static_scratch_matches_regular_entry_point_twice(B, K, N, zp):
    p = inputs.make_problem(B, K, N, seed=600 + B + K + N, zero_points=zp)
    g = p.to("cuda")
    packed = w.w4a16_pack(g.qweight, g.qzeros)
    ref = w.w4a16_gemm(g.x, packed, g.scales, zp)
    stream = torch.cuda.current_stream()
    outs = []
    for _ in range(2):
        y = torch.full((B, N), 3.0, dtype=torch.bfloat16, device="cuda")
        assert _static_gemm(g.x, packed, g.scales, zp, y, stream) == 0
        outs.append(y)
    torch.cuda.synchronize()
    assert w.w4a16_device_status() == 0
    ref_o = bits(ref)
    for y in outs:
        # within the GEMM error bound of the oracle, and of the regular call
        # (split-K sums may differ from it in the last bits: arrival order)
        worst = assert_within_bound(y.cpu(), p)
        assert worst <= 1.0
        diff = np.abs(bits_to_f64(bits(y)) - bits_to_f64(ref_o))
        _, _, bound = oracle_gemm(p)
        assert np.all(diff <= bound)


def test_static_scratch_rejects_problems_larger_than_its_array():
    """A shape whose split-K scratch exceeds the 4 MiB array is refused with
    W4A16_ERR_WORKSPACE before anything is launched."""
    big = None
    for B, K, N in [(2048, 8192, 1024), (4096, 8192, 512), (1024, 16384, 1024)]:
        if w.w4a16_workspace_bytes(B, K, N) > 4 << 20:
            big = (B, K, N)
            break
    if big is None:
        pytest.skip("no candidate shape needs more scratch than the array on this device")
    B, K, N = big
    x = torch.zeros((B, K), dtype=torch.bfloat16, device="cuda")
    scales = torch.zeros((K // 128, N), dtype=torch.bfloat16, device="cuda")
    packed = torch.zeros(w.w4a16_packed_bytes(K, N, False), dtype=torch.uint8, device="cuda")
    y = torch.zeros((B, N), dtype=torch.bfloat16, device="cuda")
    assert _static_gemm(x, packed, scales, False, y, torch.cuda.current_stream()) == 5
    torch.cuda.synchronize()
    assert torch.all(y == 0)


def test_static_scratch_after_an_expired_wait():
    """A GEMM whose bounded wait expires stops part-way.  The allocation-free
    entry point clears all of the scratch a shape uses before every call, so
    the next call through it is still within the error bound -- twice in a
    row, on a shape that splits K."""
    if w.w4a16_select_path(64, 4096, 4096) != w.PATH_TCGEN05:
        pytest.skip("tensor-core kernel unavailable")
    B, K, N = 64, 1024, 256
    assert w.w4a16_workspace_bytes(B, K, N) > 0
    p = inputs.make_problem(B, K, N, seed=613)
    g = p.to("cuda")
    packed = w.w4a16_pack(g.qweight)
    ws = torch.zeros(w.w4a16_workspace_bytes(B, K, N), dtype=torch.uint8, device="cuda")
    y = torch.zeros((B, N), dtype=torch.bfloat16, device="cuda")
    assert w.w4a16_device_status(clear=True) == 0
    assert w.w4a16_debug_forced_timeout(g.x, packed, g.scales, False, y, wait_ms=20,
                                        workspace=ws) == 0
    torch.cuda.synchronize()
    assert w.w4a16_device_status(clear=True) == 7
    stream = torch.cuda.current_stream()
    for _ in range(2):
        y = torch.full((B, N), 3.0, dtype=torch.bfloat16, device="cuda")
        assert _static_gemm(g.x, packed, g.scales, False, y, stream) == 0
        torch.cuda.synchronize()
        assert w.w4a16_device_status() == 0
        assert_within_bound(y.cpu(), p)
