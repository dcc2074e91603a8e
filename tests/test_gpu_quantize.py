"""GPU parity of the offline quantizer (w4a16_quantize_rtn) with the oracle:
codes and scales bit-identical, on random weights with outliers, a ragged
column tile, all-zero groups and the hand-worked outlier example; then the
quantized layer through pack + GEMM against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_int4_gemm_gb300 as w
from tests.gpu_util import assert_within_bound, bits
from weight_only_int4_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu


def _weights(K, N, seed, outliers=True):
    g = torch.Generator().manual_seed(seed)
    wt = torch.randn((K, N), generator=g) * 0.02
    if outliers:
        idx = torch.randint(0, K * N, (max(1, K * N // 500),), generator=g)
        wt.view(-1)[idx] *= 12.0
    return wt.to(torch.bfloat16)


def _gpu_quantize(wt):
    qw, sc = w.w4a16_quantize_rtn(wt.cuda())
    torch.cuda.synchronize()
    return qw.cpu().numpy().view(np.uint32), bits(sc.cpu())


@pytest.mark.parametrize("K,N", [(128, 8), (256, 264), (1024, 520), (4096, 4096)])
def test_quantizer_matches_oracle_bit_exact(K, N):
    wt = _weights(K, N, seed=K + N)
    if N >= 16:
        wt[:128, 3] = 0  # an all-zero group
    qw, sc = _gpu_quantize(wt)
    qo, so = oracle.quantize_rtn_mse(bits(wt))
    assert np.array_equal(sc, so), f"{int((sc != so).sum())} scales differ"
    assert np.array_equal(qw, qo), f"{int((qw != qo).sum())} code words differ"


def test_quantizer_worked_outlier_example():
    u = 2.0 ** -10
    wt = torch.full((128, 8), 5 * u, dtype=torch.float32)
    wt[37, :] = 8 * u
    qw, sc = _gpu_quantize(wt.to(torch.bfloat16))
    assert np.all(sc == 0x3A80)  # bf16 bits of 2^-10
    codes = np.stack([(qw >> (4 * j)) & 0xF for j in range(8)], axis=1).reshape(128, 8)
    assert np.all(codes[37] == 15) and np.all(np.delete(codes, 37, axis=0) == 13)


def test_quantized_layer_through_pack_and_gemm():
    K, N, B = 1024, 392, 5
    wt = _weights(K, N, seed=7)
    qw, sc = w.w4a16_quantize_rtn(wt.cuda())
    x = inputs.make_activations(B, K, seed=8)
    p = inputs.LinearProblem(x, qw.cpu(), sc.cpu(), None)
    packed = w.w4a16_pack(qw)
    y = w.w4a16_gemm(x.cuda(), packed, sc, False)
    torch.cuda.synchronize()
    assert w.w4a16_device_status() == 0
    assert_within_bound(y.cpu(), p)
