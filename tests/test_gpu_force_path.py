"""The W4A16_FORCE_PATH override (tests and ablations): the automatic path
follows it in a fresh process, workspace sizing included, and the forced
kernel's result is within the oracle bound."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, {root!r})
import torch
import weight_only_int4_gemm_gb300 as w
from weight_only_int4_gemm_gb300 import inputs
from tests.gpu_util import assert_within_bound
B, K, N = {B}, 1024, 520
print("path", w.w4a16_select_path(B, K, N), w.w4a16_kernel_name(B, K, N))
p = inputs.make_problem(B, K, N, seed=5)
g = p.to("cuda")
packed = w.w4a16_pack(g.qweight, g.qzeros)
y = w.w4a16_gemm(g.x, packed, g.scales, False)
torch.cuda.synchronize()
assert w.w4a16_device_status() == 0
assert_within_bound(y.cpu(), p)
print("ok")
"""


def run_child(force, B):
    env = dict(os.environ, W4A16_FORCE_PATH=force)
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, B=B)], env=env,
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = r.stdout.split("\n")
    path_line = [l for l in lines if l.startswith("path")][0].split()
    assert "ok" in lines
    return int(path_line[1]), path_line[2]


def test_force_skinny_at_a_wide_batch():
    assert run_child("skinny", 300) == (0, "skinny_kernel")


def test_force_tensor_cores_at_a_small_batch():
    assert run_child("tcgen05", 4) == (1, "tc_kernel")


def test_unknown_value_keeps_the_automatic_choice():
    assert run_child("bogus", 4) == (0, "skinny_kernel")
    assert run_child("bogus", 300) == (1, "wide_kernel")


def test_device_plan_matches_the_dispatch():
    """w4a16_describe_plan on the current device names the kernel
    w4a16_kernel_name reports and equals the plan for its SM count."""
    import torch
    import weight_only_int4_gemm_gb300 as w
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for B, K, N in ((1, 4096, 4096), (16, 4096, 28672), (17, 384, 64), (270, 14336, 4096),
                    (1024, 4096, 128256)):
        dev = w.w4a16_describe_plan(B, K, N)
        assert dev["kernel_name"] == w.w4a16_kernel_name(B, K, N)
        assert dev == w.w4a16_describe_plan(B, K, N, sms)
