"""Helpers shared by the GPU parity tests: move seeded inputs between torch and
the oracle's numpy views, and check GPU results against the oracle's bound."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tests.bf16_exact import bits_to_f64
from weight_only_int4_gemm_gb300 import inputs


def bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a tensor's bit pattern (uint16 for bf16 and fp16,
    uint32 for int32)."""
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.int32:
        return t.numpy().view(np.uint32)
    raise TypeError(t.dtype)


def oracle_gemm(p: inputs.LinearProblem, cols=None):
    return oracle.gemm(bits(p.x), bits(p.qweight), bits(p.scales),
                       None if p.qzeros is None else bits(p.qzeros), cols=cols)


def sample_columns(N: int, n: int, seed: int = 0) -> np.ndarray:
    """Columns that include both edges (first and ragged last tiles) plus random ones."""
    rng = np.random.default_rng(seed)
    edge = min(N, max(8, n // 4))
    cols = set(range(edge)) | set(range(N - edge, N))
    rest = max(0, n - len(cols))
    if rest:
        cols |= set(rng.choice(N, size=min(rest, N), replace=False).tolist())
    return np.array(sorted(cols), dtype=np.int32)


def assert_within_bound(y_gpu: torch.Tensor, p: inputs.LinearProblem, cols=None, rows=None):
    """|y_gpu - y_oracle| <= 8e-3 * sum|x*w| + 1e-6, element by element.

    Returns the worst ratio |diff| / bound (for reporting)."""
    if rows is not None:
        idx = torch.as_tensor(np.asarray(rows), dtype=torch.long)
        p = inputs.LinearProblem(p.x[idx], p.qweight, p.scales, p.qzeros)
        y_gpu = y_gpu[idx]
    y_o, _, bound = oracle_gemm(p, cols)
    yg = bits_to_f64(bits(y_gpu))
    if cols is not None:
        yg = yg[:, cols]
    yo = bits_to_f64(y_o)
    assert yg.shape == yo.shape
    assert np.all(np.isfinite(yg)), "non-finite GPU output"
    diff = np.abs(yg - yo)
    bad = diff > bound
    if bad.any():
        b, n = np.argwhere(bad)[0]
        raise AssertionError(
            f"{int(bad.sum())} of {bad.size} outputs outside the bound; first at "
            f"(b={b}, col={n if cols is None else cols[n]}): gpu={yg[b, n]!r} "
            f"oracle={yo[b, n]!r} bound={bound[b, n]!r}")
    return float(np.max(diff / bound))
