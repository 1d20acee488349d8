"""The accuracy gates, in one place, and the bit-pattern comparison rule.

Accuracy (GPU vs the fp64 oracle), per output element:
  fp32        |y - ref| <= 1e-5        * nrm
  bf16/fp16   |y - ref| <= 2 * ulp1    * nrm,  ulp1 = ulp of 1.0 in the output
              dtype (bf16 2^-7, fp16 2^-10)
with nrm the sum of the magnitudes of the terms (GEMM: sum_k |a b| (+|bias|,
or |alpha| sum|ab| + |beta c|); attention: sum_j p_j |v_j|).  Below the
normal range of the output dtype one ulp is the fixed subnormal spacing
(fp16 2^-24), so the gate also admits 2 of those absolute ulps.  These are the
gates the published claim states; the tests enforce exactly these numbers.

Invariance (GPU vs GPU): the uint16/uint32 bit patterns must be equal; float
comparisons are never used for it ("mlx-batch-invariant" README, "What
batch-invariant means here").
"""
from __future__ import annotations

import numpy as np
import torch

ULP1 = {torch.float32: 2.0 ** -23, torch.bfloat16: 2.0 ** -7, torch.float16: 2.0 ** -10}
ULP_SUBNORMAL = {torch.float32: 2.0 ** -149, torch.bfloat16: 2.0 ** -133, torch.float16: 2.0 ** -24}


def rel_bound(dtype) -> float:
    return 1e-5 if dtype == torch.float32 else 2.0 * ULP1[dtype]


def check_close(got: torch.Tensor, ref: np.ndarray, nrm: np.ndarray, dtype, what: str,
                floor: float = 0.0):
    """Assert the per-element gate; returns max(err / nrm) for reporting."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nrm = np.asarray(nrm, dtype=np.float64)
    assert g.shape == ref.shape, "%s: shape %s vs %s" % (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), "%s: non-finite output" % what
    err = np.abs(g - ref)
    bound = rel_bound(dtype) * nrm + 2.0 * ULP_SUBNORMAL[dtype] + floor
    bad = err > bound
    ratio = float((err / np.maximum(nrm, 1e-300)).max()) if err.size else 0.0
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError("%s: %d/%d elements over the gate; first at %s: got %.8g ref %.8g "
                             "nrm %.4g (max err/nrm %.3g, gate %.3g)"
                             % (what, int(bad.sum()), bad.size, i, g[i], ref[i], nrm[i], ratio,
                                rel_bound(dtype)))
    return ratio


def bits(t: torch.Tensor) -> torch.Tensor:
    """The raw bit pattern of a float tensor (int16 / int32 view)."""
    t = t.contiguous()
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def count_bit_diffs(a: torch.Tensor, b: torch.Tensor) -> int:
    assert a.shape == b.shape and a.dtype == b.dtype
    return int((bits(a) != bits(b)).sum().item())


def assert_same_bits(a: torch.Tensor, b: torch.Tensor, what: str):
    n = count_bit_diffs(a, b)
    assert n == 0, "%s: %d of %d bit patterns differ" % (what, n, a.numel())
