"""The packed blob's layout tag: written by w4a16_pack, checked on the host by
w4a16_packed_check and on the device by every GEMM kernel (a mismatch sets
W4A16_ERR_UNSUPPORTED in the device status word)."""
import pytest
import torch

import weight_only_int4_gemm_gb300 as w
from tests.gpu_util import assert_within_bound
from weight_only_int4_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

OK, ERR_SHAPE, ERR_UNSUP = 0, 2, 4


@pytest.mark.parametrize("zp", [False, True])
def test_pack_writes_a_tag_the_check_accepts(zp):
    p = inputs.make_problem(1, 512, 264, seed=31, zero_points=zp).to("cuda")
    packed = w.w4a16_pack(p.qweight, p.qzeros)
    assert w.w4a16_packed_check(packed, 512, 264, zp) == OK
    # another N (the tag's offset stays inside the blob): its shape word differs
    # or the bytes read there are codes, not a tag
    assert w.w4a16_packed_check(packed, 512, 256, zp) in (ERR_SHAPE, ERR_UNSUP)
    assert w.w4a16_packed_check(packed, 256, 264, zp) in (ERR_SHAPE, ERR_UNSUP)


@pytest.mark.parametrize("B", [1, 40, 300])
def test_gemm_flags_a_blob_of_another_layout_version(B):
    """A blob whose tag names another layout version is refused by the host
    check, and a GEMM on it (every kernel path by batch: small-batch, wide)
    records W4A16_ERR_UNSUPPORTED in the device status word."""
    K, N = 512, 264
    p = inputs.make_problem(B, K, N, seed=32)
    g = p.to("cuda")
    packed = w.w4a16_pack(g.qweight)
    assert w.w4a16_device_status(clear=True) == OK
    good = w.w4a16_gemm(g.x, packed, g.scales, False)
    torch.cuda.synchronize()
    assert w.w4a16_device_status() == OK
    assert_within_bound(good.cpu(), p)
    bad = packed.clone()
    bad[-12] ^= 0x5A  # the layout-version word of the tag
    assert w.w4a16_packed_check(bad, K, N, False) == ERR_UNSUP
    w.w4a16_gemm(g.x, bad, g.scales, False)
    torch.cuda.synchronize()
    assert w.w4a16_device_status(clear=True) == ERR_UNSUP
    # the word is cleared and the next call on a good blob is clean
    w.w4a16_gemm(g.x, packed, g.scales, False)
    torch.cuda.synchronize()
    assert w.w4a16_device_status() == OK
