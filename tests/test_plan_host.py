"""Host-side planning (no GPU): w4a16_describe_plan for a device with a
given SM count, checked for the invariants the kernels rely on -- every batch
row and every weight column covered once, no empty K split, the rings and
tensor-memory columns within what the kernels are launched with, the
workspace within w4a16_workspace_bytes -- over decode, prefill, 70B and odd
shapes, batch 1 .. 4096 and several SM counts."""
import math
import os

import pytest

import weight_only_int4_gemm_gb300 as w

pytestmark = pytest.mark.skipif(os.environ.get("W4A16_FORCE_PATH") is not None,
                                reason="the automatic path is overridden in this process")

SHAPES = [(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096), (4096, 128256),
          (8192, 10240), (8192, 57344), (28672, 8192),
          (128, 8), (256, 264), (1024, 520), (384, 136), (14336, 4104), (128, 40)]
BATCHES = list(range(1, 41)) + [48, 63, 64, 65, 96, 100, 127, 128, 129, 160, 161, 176, 192, 200,
                                208, 255, 256, 257, 270, 300, 384, 500, 512, 513, 1000, 1024,
                                1500, 2048, 4096]
SM_SMEM_PER_CTA = 227 * 1024     # largest dynamic shared memory of one CTA
SM_SMEM = 228 * 1024             # shared memory of one SM
MAX_COUNTERS = 16384 - 2         # split-K arrival counters in the workspace prefix


def check(plan, B, K, N, sms):
    G = K // 128
    rows, bt = plan["batch_rows"], plan["batch_tiles"]
    assert bt * rows >= B and (bt - 1) * rows < B, "batch tiles cover B exactly"
    assert plan["col_tiles"] == math.ceil(N / 128)
    s, gps = plan["k_splits"], plan["groups_per_split"]
    assert s >= 1 and gps >= 1 and s * gps >= G and (s - 1) * gps < G, "no empty K split"
    units = bt * plan["col_tiles"] * s
    assert 1 <= plan["grid"] <= min(units, sms * plan["ctas_per_sm"])
    assert plan["workspace_bytes"] <= w.w4a16_workspace_bytes(B, K, N)
    if s > 1:
        assert plan["workspace_bytes"] >= 4 * B * N, "room for the fp32 accumulator"
    if plan["kernel_name"] == "skinny_kernel":
        assert B <= 16
        assert rows in (8, 16) and rows >= min(B, 16) and plan["ctas_per_sm"] in (2, 3)
        assert plan["smem_bytes"] <= SM_SMEM_PER_CTA
        assert plan["ctas_per_sm"] * plan["smem_bytes"] <= SM_SMEM
        if s > 1:
            assert bt * plan["col_tiles"] <= MAX_COUNTERS
    else:
        assert plan["kernel_name"] == "wide_kernel" and B > 16
        assert rows % 16 == 0 and 32 <= rows <= 256
        assert plan["issuers"] == (2 if rows <= 128 else 1)
        assert plan["block_rows"] == (128 if rows <= 160 else 64)
        assert plan["acc_buffers"] in (1, 2)
        slots = plan["tile_slots"]
        assert slots >= 4 and slots % 2 == 0 and slots % plan["issuers"] == 0
        assert plan["x_slots"] == slots and plan["code_slots"] >= 2
        assert plan["tmem_cols"] <= 512
        acc = (rows + 31) // 32 * 32
        assert plan["tmem_cols"] >= plan["acc_buffers"] * plan["issuers"] * acc
        assert plan["smem_bytes"] <= SM_SMEM_PER_CTA
        if s > 1:
            assert rows <= 160, "no K split beside tiles wider than 160 rows"
            assert bt * plan["col_tiles"] <= MAX_COUNTERS


@pytest.mark.parametrize("sms", [152, 148, 132, 20, 1])
@pytest.mark.parametrize("K,N", SHAPES)
def test_plans_cover_the_problem_and_fit_the_kernels(K, N, sms):
    for B in BATCHES:
        plan = w.w4a16_describe_plan(B, K, N, sms)
        check(plan, B, K, N, sms)


def test_plan_is_a_pure_function_of_the_shape():
    a = [w.w4a16_describe_plan(B, 4096, 28672, 152) for B in (1, 64, 1024)]
    b = [w.w4a16_describe_plan(B, 4096, 28672, 152) for B in (1, 64, 1024)]
    assert a == b


def test_decode_sweep_kernels():
    """The decode sweep's kernels: the small-batch kernel up to 16 rows, the
    wide tensor-core kernel above (whose largest tiles are 256 rows)."""
    for B in (1, 4, 16):
        assert w.w4a16_describe_plan(B, 4096, 4096, 152)["kernel_name"] == "skinny_kernel"
    for B in (17, 64, 128, 256, 270, 384, 512, 1024):
        assert w.w4a16_describe_plan(B, 4096, 4096, 152)["kernel_name"] == "wide_kernel"
    assert w.w4a16_describe_plan(1024, 4096, 28672, 152)["batch_rows"] == 256


@pytest.mark.parametrize("B,K,N,sms", [(0, 4096, 4096, 152), (1, 4000, 4096, 152),
                                       (1, 4096, 4100, 152), (1, 4096, 4096, -1)])
def test_invalid_requests_are_refused(B, K, N, sms):
    with pytest.raises(w.W4A16Error):
        w.w4a16_describe_plan(B, K, N, sms)
