"""``batch_invariant_mode()``: reroute torch's GEMM and attention ops to the kernels.

"mlx-batch-invariant" README, "Use": inside the block, matmul, addmm, the @
operator, the Linear layer and scaled-dot-product attention run through the
invariant kernels; anything that cannot be made invariant raises
NotImplementedError, unless ``strict=False``, which falls back to the stock
op (useful to find out what a model needs, not something to ship).
"""
from __future__ import annotations

import contextlib
import threading

import torch
import torch.nn.functional as F

from . import api

_DTYPES = (torch.float32, torch.float16, torch.bfloat16)
_lock = threading.Lock()


def _gemm_ok(a: torch.Tensor, b: torch.Tensor) -> bool:
    return (a.is_cuda and b.is_cuda and a.dtype in _DTYPES and b.dtype == a.dtype
            and a.dim() >= 1 and b.dim() == 2 and a.stride(-1) == 1 and b.stride(-1) == 1)


@contextlib.contextmanager
def batch_invariant_mode(strict: bool = True):
    """Patch torch.matmul, Tensor.__matmul__, torch.addmm, F.linear and
    F.scaled_dot_product_attention for the duration of the block.  matmul of
    stacked operands ([..., M, K] @ [..., K, N]) runs the batched GEMM."""
    orig = {
        "matmul": torch.matmul,
        "tmatmul": torch.Tensor.__matmul__,
        "addmm": torch.addmm,
        "linear": F.linear,
        "sdpa": F.scaled_dot_product_attention,
    }

    def fallback(what, fn, *args, **kw):
        if strict:
            raise NotImplementedError("batch_invariant_mode: no batch-invariant kernel for %s "
                                      "(pass strict=False to fall back)" % what)
        return fn(*args, **kw)

    def _linear(input, weight, bias=None):
        if _gemm_ok(input, weight) and (bias is None or bias.is_contiguous()):
            try:
                return api.linear(input, weight, bias)
            except (ValueError, api.L.BiError):
                pass
        return fallback("linear%s" % (tuple(input.shape),), orig["linear"], input, weight, bias)

    def _matmul(a, b, *, out=None):
        if (out is None and b.dim() >= 3 and a.dim() >= 2 and a.is_cuda and b.is_cuda
                and a.dtype in _DTYPES and b.dtype == a.dtype):
            # stacked operands: one batched launch, each entry as the plain GEMM
            try:
                return api.bmm(a, b)
            except (ValueError, api.L.BiError):
                pass
        elif out is None and _gemm_ok(a, b):
            try:
                return api.matmul(a, b)
            except (ValueError, api.L.BiError):
                pass
        elif out is None and b.dim() == 2 and b.stride(0) == 1 and _gemm_ok(a, b.t()):
            # a @ w.t() with w[N, K] contiguous: the nn.Linear layout.
            try:
                return api.linear(a, b.t())
            except (ValueError, api.L.BiError):
                pass
        return fallback("matmul%s@%s" % (tuple(a.shape), tuple(b.shape)), orig["matmul"], a, b,
                        **({} if out is None else {"out": out}))

    def _tmatmul(self, other):
        return _matmul(self, other)

    def _addmm(input, mat1, mat2, *, beta=1, alpha=1, out=None):
        if out is None and _gemm_ok(mat1, mat2) and mat1.dim() == 2:
            try:
                return api.addmm(input, mat1, mat2, alpha=float(alpha), beta=float(beta))
            except (ValueError, api.L.BiError):
                pass
        return fallback("addmm", orig["addmm"], input, mat1, mat2, beta=beta, alpha=alpha,
                        **({} if out is None else {"out": out}))

    def _sdpa(query, key, value, attn_mask=None, dropout_p=0.0, is_causal=False, scale=None,
              enable_gqa=False):
        bool_mask = attn_mask is not None and attn_mask.dtype == torch.bool and not is_causal
        ok = ((attn_mask is None or bool_mask) and dropout_p == 0.0 and query.dim() == 4
              and query.is_cuda and query.dtype in (torch.float16, torch.bfloat16)
              and (enable_gqa or key.shape[1] == query.shape[1]))
        if ok:
            try:
                if bool_mask:
                    # torch's boolean mask: True = the key takes part, as the array form.
                    return api.sdpa(query, key, value, mask=attn_mask, scale=scale)
                # torch's is_causal aligns the mask to the top-left corner: query i sees keys <= i.
                return api.sdpa(query, key, value, causal=bool(is_causal),
                                q_offset=0 if is_causal else None, scale=scale)
            except (ValueError, api.L.BiError):
                pass
        kw = dict(attn_mask=attn_mask, dropout_p=dropout_p, is_causal=is_causal, scale=scale)
        if enable_gqa:
            kw["enable_gqa"] = True
        return fallback("scaled_dot_product_attention", orig["sdpa"], query, key, value, **kw)

    with _lock:
        torch.matmul = _matmul
        torch.Tensor.__matmul__ = _tmatmul
        torch.addmm = _addmm
        F.linear = _linear
        F.scaled_dot_product_attention = _sdpa
    try:
        yield
    finally:
        with _lock:
            torch.matmul = orig["matmul"]
            torch.Tensor.__matmul__ = orig["tmatmul"]
            torch.addmm = orig["addmm"]
            F.linear = orig["linear"]
            F.scaled_dot_product_attention = orig["sdpa"]
