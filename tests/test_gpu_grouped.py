"""GPU parity of the mixture-of-experts GEMM (w4a16_gemm_grouped) against the
oracle's per-expert GEMM, through the C ABI.

Bar: every output within |y_gpu - y_oracle| <= 8e-3 * sum_k |x_k * w_kn| + 1e-6
(the plain GEMM's bound, per row of its own expert).
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


def pack_experts(g: inputs.GroupedProblem) -> torch.Tensor:
    E = g.qweight.shape[0]
    return torch.stack([w.w4a16_pack(g.qweight[e], None if g.qzeros is None else g.qzeros[e])
                        for e in range(E)])


def oracle_grouped(p: inputs.GroupedProblem, offsets, cols=None):
    E = p.qweight.shape[0]
    return oracle.gemm_grouped(
        bits(p.x), offsets.cpu().numpy(), [bits(p.qweight[e]) for e in range(E)],
        [bits(p.scales[e]) for e in range(E)],
        None if p.qzeros is None else [bits(p.qzeros[e]) for e in range(E)], cols=cols)


def check(y_gpu, p, offsets=None, cols=None, rows=None):
    offsets = p.offsets if offsets is None else offsets
    y_o, _, bound = oracle_grouped(p, offsets, cols)
    yg = bits_to_f64(bits(y_gpu))
    if cols is not None:
        yg = yg[:, cols]
    yo = bits_to_f64(y_o)
    if rows is not None:
        yg, yo, bound = yg[rows], yo[rows], bound[rows]
    assert np.all(np.isfinite(yg)), "non-finite GPU output"
    bad = np.abs(yg - yo) > bound
    if bad.any():
        r, n = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} of {bad.size} outside the bound; first at "
                             f"row {r}, col {n}: gpu={yg[r, n]!r} oracle={yo[r, n]!r}")


def run(p: inputs.GroupedProblem, max_rows, out=None):
    g = p.to("cuda")
    packed = pack_experts(g)
    y = w.w4a16_gemm_grouped(g.x, g.offsets, packed, g.scales, g.qzeros is not None, max_rows,
                             out=out)
    torch.cuda.synchronize()
    assert w.w4a16_device_status() == 0
    return y.cpu()


COUNTS = [0, 5, 17, 1, 0, 33, 8, 0]


@pytest.mark.parametrize("zp", [False, True])
@pytest.mark.parametrize("max_rows", [8, 16, 64])
def test_ragged_experts_small(zp, max_rows):
    """Eight experts with 0 .. 33 rows (several empty), a ragged last column tile,
    and a max_rows hint below the largest expert."""
    p = inputs.make_grouped_problem(inputs.offsets_from_counts(COUNTS), 1024, 520, 11,
                                    zero_points=zp)
    check(run(p, max_rows), p)


@pytest.mark.parametrize("zp", [False, True])
def test_tall_experts_32_row_tiles(zp):
    """Few experts with many rows (mean 32): the 32-row batch tile, an expert
    above it split over several tiles, and an empty expert."""
    p = inputs.make_grouped_problem(inputs.offsets_from_counts([40, 0, 70, 18]), 1024, 264, 71,
                                    zero_points=zp)
    check(run(p, 70), p)


@pytest.mark.parametrize("zp", [False, True])
def test_split_k_and_repeat(zp):
    """Few rows over a deep K: the planner splits K (fp32 partials + arrival
    counters); a second call must find the workspace clean again."""
    p = inputs.make_grouped_problem(inputs.offsets_from_counts([1, 0, 2, 1, 0, 3, 0, 1]),
                                    4096, 512, 21, zero_points=zp)
    check(run(p, 8), p)
    check(run(p, 8), p)


def test_max_experts_sparse_routing():
    """256 experts (the limit), 40 tokens routed top-8: many experts empty."""
    off = inputs.make_routing(40, 256, 8, 5)
    p = inputs.make_grouped_problem(off, 256, 264, 31)
    check(run(p, 16), p)


@pytest.mark.parametrize("tokens", [8, 64])
def test_moe_expert_layer_full_size(tokens):
    """A 128-expert, top-8 expert layer (hidden 2048, expert width 768: gate+up
    K=2048 x N=1536, down K=768 x N=2048) at decode batches, sampled columns."""
    for K, N, seed in ((2048, 1536, 41), (768, 2048, 43)):
        off = inputs.make_routing(tokens, 128, 8, seed)
        p = inputs.make_grouped_problem(off, K, N, seed)
        max_rows = int((off[1:] - off[:-1]).max())
        check(run(p, max_rows), p, cols=sample_columns(N, 192, seed))


def test_offsets_written_by_the_previous_kernel():
    """The routing table is produced on the stream right before the call (the
    kernel reads it only after the previous kernel's writes are visible)."""
    counts = torch.tensor(COUNTS, dtype=torch.int32)
    p = inputs.make_grouped_problem(inputs.offsets_from_counts(COUNTS), 1024, 256, 51)
    g = p.to("cuda")
    packed = pack_experts(g)
    torch.cuda.synchronize()
    for _ in range(3):
        off = torch.zeros(len(COUNTS) + 1, dtype=torch.int32, device="cuda")
        off[1:] = torch.cumsum(counts.cuda(), 0).to(torch.int32)
        y = w.w4a16_gemm_grouped(g.x, off, packed, g.scales, False, 33)
        torch.cuda.synchronize()
        assert w.w4a16_device_status() == 0
        check(y.cpu(), p)


def test_malformed_offsets_stay_inside_the_batch():
    """A decreasing entry is lifted to the running maximum and values beyond T
    are clamped: rows 0..39 use expert 0, expert 1 is empty, rows 40..63 use
    expert 2, and nothing outside y is written."""
    T = 64
    good = torch.tensor([0, 40, 40, T], dtype=torch.int32)
    p = inputs.make_grouped_problem(good, 512, 128, 61)
    g = p.to("cuda")
    packed = pack_experts(g)
    for bad in ([0, 40, 20, T], [0, 40, 20, T + 50]):
        guard = torch.full((T + 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
        y = w.w4a16_gemm_grouped(g.x, torch.tensor(bad, dtype=torch.int32, device="cuda"),
                                 packed, g.scales, False, 64, out=guard[1:T + 1])
        torch.cuda.synchronize()
        assert w.w4a16_device_status() == 0
        assert torch.all(guard[0] == 7.0) and torch.all(guard[T + 1] == 7.0)
        check(y.cpu(), p, offsets=good)
