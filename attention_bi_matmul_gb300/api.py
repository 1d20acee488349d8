"""Torch-facing wrappers of the C ABI (include/bi.h).

Each function checks shapes and dtypes, allocates the output with torch when
none is given, and calls the library on the current CUDA stream of the
inputs' device.  No arithmetic happens here: every step runs in the CUDA
kernels of ``libbi.so``.  Errors from the library raise ``BiError``.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib as L

_DT = {torch.float32: L.BI_F32, torch.float16: L.BI_F16, torch.bfloat16: L.BI_BF16}


def _dt(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError("unsupported dtype %s (float32, float16, bfloat16)" % t.dtype) from None


def _cuda(*ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("bi: tensors must live on a CUDA device (got %s)" % t.device)
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("bi: tensors on different devices (%s, %s)" % (dev, t.device))
    return dev


class _On:
    """Make `dev` current for the call (cheap when it already is)."""

    __slots__ = ("dev", "prev")

    def __init__(self, dev):
        self.dev = dev.index if dev.index is not None else torch.cuda.current_device()
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.dev:
            self.prev = cur
            torch.cuda.set_device(self.dev)
        return ctypes.c_void_p(torch.cuda.current_stream(self.dev).cuda_stream)

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
        return False


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _rows(x: torch.Tensor, what: str) -> torch.Tensor:
    """View x[..., K] as [M, K] without copying (last dim contiguous, uniform row stride)."""
    if x.dim() == 0 or x.stride(-1) != 1:
        raise ValueError("%s: the last dimension must be contiguous" % what)
    if x.dim() == 1:
        return x.unsqueeze(0)
    if x.dim() > 2:
        try:
            return x.view(-1, x.shape[-1])
        except RuntimeError:
            raise ValueError("%s: leading dimensions cannot be flattened without a copy" % what) from None
    return x


def _ld(t2: torch.Tensor, cols: int) -> int:
    """Row stride of a [rows, cols] view; a single row gets the smallest aligned stride."""
    if t2.shape[0] > 1:
        return t2.stride(0)
    return max(t2.stride(0), (cols + 7) // 8 * 8)


def _new_rows(M: int, N: int, like: torch.Tensor) -> torch.Tensor:
    """Output [M, N]; 16-bit rows padded to a multiple of 8 elements (16 bytes) when needed."""
    if like.dtype == torch.float32 or N % 8 == 0:
        return torch.empty((M, N), dtype=like.dtype, device=like.device)
    Np = (N + 7) // 8 * 8
    return torch.empty((M, Np), dtype=like.dtype, device=like.device)[:, :N]


# ------------------------------------------------------------------ GEMMs

def linear(x: torch.Tensor, w: torch.Tensor, bias: torch.Tensor | None = None,
           out: torch.Tensor | None = None) -> torch.Tensor:
    """y = x . w^T + bias with w in the nn.Linear layout [N, K]; leading dims of x are batch."""
    dev = _cuda(x, w, bias, out)
    lead = x.shape[:-1]
    x2 = _rows(x, "x")
    M, K = x2.shape
    if w.dim() != 2 or w.shape[1] != K or w.stride(-1) != 1:
        raise ValueError("w must be [N, K=%d] with K contiguous, got %s" % (K, tuple(w.shape)))
    N = w.shape[0]
    if w.dtype != x.dtype or (bias is not None and (bias.dtype != x.dtype or bias.shape != (N,)
                                                     or not bias.is_contiguous())):
        raise ValueError("linear: dtype/shape mismatch")
    y = _new_rows(M, N, x) if out is None else _rows(out, "out")
    if y.shape != (M, N):
        raise ValueError("out must hold [M, N]")
    with _On(dev) as s:
        L.check(L.load().bi_linear(_p(x2), _ld(x2, K), _p(w), _ld(w, K), _p(bias), _p(y),
                                   _ld(y, N), M, N, K, _dt(x), s), "bi_linear")
    return y.view(*lead, N) if out is None and y.is_contiguous() else (y if out is None else out)


def _entry_stride(t: torch.Tensor, nlead: int) -> int | None:
    """One element stride that walks the first `nlead` dims of t in order, or None."""
    if nlead == 0:
        return 0
    sizes, strides = t.shape[:nlead], t.stride()[:nlead]
    live = [(n, st) for n, st in zip(sizes, strides) if n != 1]
    if not live:
        return 0
    if all(st == 0 for _, st in live):
        return 0
    for (n0, st0), (n1, st1) in zip(live, live[1:]):
        if st0 != st1 * n1:
            return None
    return live[-1][1]


def bmm(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """Stacked matmul a[..., M, K] . b[..., K, N] with broadcast leading dims.

    b may be any view whose last two dims are either [K, N] with N contiguous or
    the transpose of an [N, K] block with K contiguous (``w.transpose(-1, -2)``).
    Each entry's bits equal those of the unbatched call on that entry.
    """
    dev = _cuda(a, b, out)
    if a.dim() < 2 or b.dim() < 2 or a.shape[-1] != b.shape[-2] or a.dtype != b.dtype:
        raise ValueError("bmm: a[..., M, K] and b[..., K, N] of one dtype")
    M, K = a.shape[-2:]
    N = b.shape[-1]
    lead = tuple(torch.broadcast_shapes(a.shape[:-2], b.shape[:-2]))
    nl = len(lead)
    ae = a.expand(*lead, M, K)
    be = b.expand(*lead, K, N)
    r8 = lambda n: (n + 7) // 8 * 8
    if out is None:
        # 16-bit rows padded to a multiple of 8 elements (16 bytes) when needed
        Np = N if (a.dtype == torch.float32 or N % 8 == 0) else r8(N)
        y = torch.empty((*lead, M, Np), dtype=a.dtype, device=a.device)[..., :N]
    else:
        y = out
    if tuple(y.shape) != (*lead, M, N) or y.stride(-1) != 1:
        raise ValueError("bmm: out must be [..., M, N] with N contiguous")
    # b's layout: [K, N] with N contiguous (1), or the transpose of [N, K] with K
    # contiguous (0).  The row stride of a single row is never used; it gets the
    # smallest aligned value.
    if N > 1 and be.stride(-1) == 1:
        layout, ldb = 1, (be.stride(-2) if K > 1 else r8(N))
    elif K > 1 and be.stride(-2) == 1:
        layout, ldb = 0, (be.stride(-1) if N > 1 else r8(K))
    elif N == 1 and K == 1:
        layout, ldb = 1, 8
    elif N == 1:
        layout, ldb = 1, be.stride(-2)
    elif K == 1:
        layout, ldb = 0, be.stride(-1)
    else:
        raise ValueError("bmm: b needs N or K contiguous")
    if ae.stride(-1) != 1 and K > 1:
        raise ValueError("bmm: a's last dimension must be contiguous")
    sa, sb, sy = _entry_stride(ae, nl), _entry_stride(be, nl), _entry_stride(y, nl)
    if sa is None or sb is None or sy is None:
        # No single stride walks the leading dims (e.g. b[3,K,N] broadcast to
        # [2,3,K,N]): one launch per index of the first leading dim.  Entries are
        # independent, so this changes no bit.
        if nl < 2:
            raise ValueError("bmm: leading dimensions cannot be walked with one stride")
        for i in range(lead[0]):
            bmm(ae[i], be[i], out=y[i])
        return y
    batch = 1
    for n in lead:
        batch *= n
    lda = ae.stride(-2) if M > 1 else r8(K)
    ldy = y.stride(-2) if M > 1 else r8(N)
    if batch == 0 or M == 0:
        return y
    with _On(dev) as s:
        L.check(L.load().bi_matmul_batched(_p(ae), lda, sa, _p(be), ldb, sb, layout, _p(y), ldy,
                                           sy, batch, M, N, K, _dt(a), s), "bi_matmul_batched")
    return y


def matmul(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """y = a . b with b[K, N] (N contiguous); leading dims of a are batch.  A b with
    leading dims of its own is a stacked matmul (``bmm``)."""
    if b.dim() > 2:
        return bmm(a, b, out)
    dev = _cuda(a, b, out)
    lead = a.shape[:-1]
    a2 = _rows(a, "a")
    M, K = a2.shape
    if b.dim() != 2 or b.shape[0] != K or b.stride(-1) != 1 or b.dtype != a.dtype:
        raise ValueError("b must be [K=%d, N] with N contiguous and a's dtype" % K)
    N = b.shape[1]
    y = _new_rows(M, N, a) if out is None else _rows(out, "out")
    with _On(dev) as s:
        L.check(L.load().bi_matmul(_p(a2), _ld(a2, K), _p(b), _ld(b, N), _p(y), _ld(y, N),
                                   M, N, K, _dt(a), s), "bi_matmul")
    return y.view(*lead, N) if out is None and y.is_contiguous() else (y if out is None else out)


def qlinear(x: torch.Tensor, wq: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
            bits: int, group_size: int, bias: torch.Tensor | None = None,
            out: torch.Tensor | None = None) -> torch.Tensor:
    """y = x . w^T (+ bias) with group-wise affine quantized w[N, K]:
    w[n,k] = scales[n, k//group_size] * q[n,k] + biases[n, k//group_size], q packed in
    wq (int32 or uint32 [N, K*bits/32]) lowest field first.  Leading dims of x are batch."""
    dev = _cuda(x, wq, scales, biases, bias, out)
    lead = x.shape[:-1]
    x2 = _rows(x, "x")
    M, K = x2.shape
    if wq.dim() != 2 or wq.stride(-1) != 1 or wq.element_size() != 4:
        raise ValueError("qlinear: wq must be a 32-bit [N, K*bits/32] tensor, last dim contiguous")
    N = wq.shape[0]
    if scales.shape != biases.shape or scales.dim() != 2 or scales.shape[0] != N:
        raise ValueError("qlinear: scales/biases must be [N, K/group_size]")
    if scales.stride(-1) != 1 or biases.stride(-1) != 1 or scales.stride(0) != biases.stride(0):
        raise ValueError("qlinear: scales and biases need the same contiguous row layout")
    G = scales.shape[1]
    if scales.stride(0) % 8 or scales.data_ptr() % 16 or biases.data_ptr() % 16:
        # The library copies scale rows in 16-byte boxes: give it rows padded to a
        # multiple of 8 elements (a layout copy; pad once ahead of time to avoid it).
        Gp = (G + 7) // 8 * 8
        sp = torch.zeros((N, 2, Gp), dtype=scales.dtype, device=scales.device)
        sp[:, 0, :G] = scales
        sp[:, 1, :G] = biases
        scales, biases = sp[:, 0, :G], sp[:, 1, :G]
    if scales.dtype != x.dtype or biases.dtype != x.dtype or (
            bias is not None and (bias.dtype != x.dtype or bias.shape != (N,)
                                  or not bias.is_contiguous())):
        raise ValueError("qlinear: dtype/shape mismatch")
    y = torch.empty((M, N), dtype=x.dtype, device=x.device) if out is None else _rows(out, "out")
    if y.shape != (M, N):
        raise ValueError("out must hold [M, N]")
    with _On(dev) as s:
        L.check(L.load().bi_qlinear(_p(x2), _ld(x2, K), _p(wq), max(wq.stride(0), wq.shape[1]),
                                    _p(scales), _p(biases), scales.stride(0) if N > 1 else
                                    (G + 7) // 8 * 8, _p(bias), _p(y), y.stride(0) if M > 1 else N,
                                    M, N, K, int(bits), int(group_size), _dt(x), s), "bi_qlinear")
    return y.view(*lead, N) if out is None else out


def addmm(c: torch.Tensor, a: torch.Tensor, b: torch.Tensor, alpha: float = 1.0,
          beta: float = 1.0, out: torch.Tensor | None = None) -> torch.Tensor:
    """y = beta * c + alpha * (a . b); c is [M, N] or a row [N] (broadcast)."""
    dev = _cuda(c, a, b, out)
    if a.dim() != 2:
        raise ValueError("addmm: a must be 2-D")
    M, K = a.shape
    if b.dim() != 2 or b.shape[0] != K or b.stride(-1) != 1:
        raise ValueError("b must be [K, N] with N contiguous")
    N = b.shape[1]
    if c.dtype != a.dtype or b.dtype != a.dtype:
        raise ValueError("addmm: dtype mismatch")
    if c.dim() == 1 or (c.dim() == 2 and c.shape[0] == 1 and M != 1):
        c1 = c.reshape(-1)
        if c1.shape != (N,) or c1.stride(0) != 1:
            raise ValueError("addmm: row c must be [N] contiguous")
        cptr, ldc = c1, 0
    else:
        if c.shape != (M, N) or c.stride(-1) != 1:
            raise ValueError("addmm: c must be [M, N] with N contiguous")
        cptr, ldc = c, _ld(c, N)
    y = _new_rows(M, N, a) if out is None else out
    with _On(dev) as s:
        L.check(L.load().bi_addmm(_p(cptr), ldc, _p(a), _ld(a, K), _p(b), _ld(b, N), _p(y),
                                  _ld(y, N), M, N, K, float(alpha), float(beta), _dt(a), s),
                "bi_addmm")
    return y


def gemm_config(N: int, K: int, dtype=torch.bfloat16, layout: str = "linear"):
    """(block_n, stages) of the GEMM for this (N, K, dtype, layout); M plays no part."""
    bn, st = ctypes.c_int(), ctypes.c_int()
    L.check(L.load().bi_gemm_config(int(N), int(K), _DT[dtype], 0 if layout == "linear" else 1,
                                    ctypes.byref(bn), ctypes.byref(st)), "bi_gemm_config")
    return bn.value, st.value


# ------------------------------------------------------------------ attention

def sdpa(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = True,
         q_offset: int | None = None, scale: float | None = None,
         out: torch.Tensor | None = None, mask: torch.Tensor | None = None,
         sinks: torch.Tensor | None = None) -> torch.Tensor:
    """Attention, q[B,H,Lq,D], k/v[B,Hkv,Lkv,D] (any strides, last dim contiguous).

    Query i sits at absolute position q_offset + i (default Lkv - Lq); with
    ``causal`` it sees keys j <= q_offset + i.  ``mask``: a boolean array mask
    broadcastable to [B,H,Lq,Lkv] (True = visible; overrides ``causal``).
    ``sinks``: fp32 [H] sink logits.  Returns o[B,H,Lq,D].
    """
    if mask is not None or sinks is not None:
        return _sdpa_ex(q, k, v, causal, q_offset, scale, out, mask, sinks)
    dev = _cuda(q, k, v, out)
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("sdpa: q, k, v must be 4-D")
    B, H, Lq, D = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    if k.shape != (B, Hkv, Lkv, D) or v.shape != k.shape:
        raise ValueError("sdpa: k/v must be [B, Hkv, Lkv, D]")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("sdpa: dtype mismatch")
    o = torch.empty((B, H, Lq, D), dtype=q.dtype, device=q.device) if out is None else out
    qo = -1 if q_offset is None else int(q_offset)
    with _On(dev) as s:
        L.check(L.load().bi_sdpa(_p(q), L.i64arr(q.stride()), _p(k), L.i64arr(k.stride()),
                                 _p(v), L.i64arr(v.stride()), _p(o), L.i64arr(o.stride()),
                                 B, H, Hkv, Lq, Lkv, D, 0.0 if scale is None else float(scale),
                                 L.BI_MASK_CAUSAL if causal else L.BI_MASK_NONE, qo, _dt(q), s),
                "bi_sdpa")
    return o


def _sdpa_ex(q, k, v, causal, q_offset, scale, out, mask, sinks):
    dev = _cuda(q, k, v, out, mask, sinks)
    B, H, Lq, D = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    if k.shape != (B, Hkv, Lkv, D) or v.shape != k.shape:
        raise ValueError("sdpa: k/v must be [B, Hkv, Lkv, D]")
    mode = L.BI_MASK_CAUSAL if causal else L.BI_MASK_NONE
    mptr, ms = None, None
    if mask is not None:
        if mask.dtype != torch.bool:
            raise ValueError("sdpa: the array mask must be boolean (True = visible)")
        m4 = mask.reshape((1,) * (4 - mask.dim()) + tuple(mask.shape)) if mask.dim() < 4 else mask
        m4 = m4.expand(B, H, Lq, Lkv)
        if m4.stride(-1) != 1:
            raise ValueError("sdpa: the mask's last dimension must be contiguous")
        mode, mptr, ms = L.BI_MASK_ARRAY, ctypes.c_void_p(m4.data_ptr()), L.i64arr(m4.stride())
    sk = None
    if sinks is not None:
        if sinks.dtype != torch.float32 or sinks.shape != (H,) or not sinks.is_contiguous():
            raise ValueError("sdpa: sinks must be contiguous float32 [H]")
        sk = ctypes.c_void_p(sinks.data_ptr())
    o = torch.empty((B, H, Lq, D), dtype=q.dtype, device=q.device) if out is None else out
    qo = -1 if q_offset is None else int(q_offset)
    with _On(dev) as s:
        L.check(L.load().bi_sdpa_ex(_p(q), L.i64arr(q.stride()), _p(k), L.i64arr(k.stride()),
                                    _p(v), L.i64arr(v.stride()), _p(o), L.i64arr(o.stride()),
                                    B, H, Hkv, Lq, Lkv, D, 0.0 if scale is None else float(scale),
                                    mode, qo, sk, mptr, ms, _dt(q), s), "bi_sdpa_ex")
    return o


# ------------------------------------------------------------------ decoder glue

def rmsnorm(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6,
            out: torch.Tensor | None = None) -> torch.Tensor:
    dev = _cuda(x, w, out)
    x2 = _rows(x, "x")
    M, N = x2.shape
    y = torch.empty_like(x2) if out is None else _rows(out, "out")
    with _On(dev) as s:
        L.check(L.load().bi_rmsnorm(_p(x2), _ld(x2, N), _p(w), _p(y), _ld(y, N), M, N,
                                    float(eps), _dt(x), s), "bi_rmsnorm")
    return y.view(x.shape) if out is None else out


def rope(x: torch.Tensor, pos0: int, base: float = 10000.0,
         out: torch.Tensor | None = None) -> torch.Tensor:
    """Rotate-half RoPE on x[B, L, nh, D]; position of (b, l) is pos0 + l.  ``out`` may be a
    strided view (e.g. a KV-cache slice) of the same shape."""
    dev = _cuda(x, out)
    if x.dim() != 4:
        raise ValueError("rope: x must be [B, L, nh, D]")
    y = torch.empty_like(x) if out is None else out
    if y.shape != x.shape:
        raise ValueError("rope: out shape mismatch")
    B, Lx, nh, D = x.shape
    with _On(dev) as s:
        L.check(L.load().bi_rope(_p(x), L.i64arr(x.stride()), _p(y), L.i64arr(y.stride()), B, Lx,
                                 nh, D, int(pos0), float(base), _dt(x), s), "bi_rope")
    return y


def swiglu(gu: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """silu(gate) * up for gu[..., 2I] = [gate | up]."""
    dev = _cuda(gu, out)
    g2 = _rows(gu, "gu")
    M, I2 = g2.shape
    I = I2 // 2
    y = torch.empty((M, I), dtype=gu.dtype, device=gu.device) if out is None else _rows(out, "out")
    with _On(dev) as s:
        L.check(L.load().bi_swiglu(_p(g2), _ld(g2, I2), _p(y), _ld(y, I), M, I, _dt(gu), s),
                "bi_swiglu")
    return y.view(*gu.shape[:-1], I) if out is None else out


def add(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    dev = _cuda(a, b, out)
    if a.shape != b.shape or not a.is_contiguous() or not b.is_contiguous():
        raise ValueError("add: a and b must be contiguous and of one shape")
    y = torch.empty_like(a) if out is None else out
    with _On(dev) as s:
        L.check(L.load().bi_add(_p(a), _p(b), _p(y), a.numel(), _dt(a), s), "bi_add")
    return y


def embedding(ids: torch.Tensor, table: torch.Tensor, out: torch.Tensor | None = None):
    dev = _cuda(ids, table, out)
    if ids.dtype != torch.int64 or not ids.is_contiguous():
        raise ValueError("embedding: ids must be contiguous int64")
    V, dim = table.shape
    n = ids.numel()
    y = torch.empty((n, dim), dtype=table.dtype, device=table.device) if out is None else out
    with _On(dev) as s:
        L.check(L.load().bi_embedding(_p(ids), n, _p(table), table.stride(0), V, _p(y),
                                      y.stride(0), dim, _dt(table), s), "bi_embedding")
    return y.view(*ids.shape, dim) if out is None else out


def copy4d(src: torch.Tensor, dst: torch.Tensor) -> torch.Tensor:
    dev = _cuda(src, dst)
    if src.shape != dst.shape or src.dim() != 4 or src.dtype != dst.dtype:
        raise ValueError("copy4d: 4-D tensors of one shape and dtype")
    with _On(dev) as s:
        L.check(L.load().bi_copy4d(_p(src), L.i64arr(src.stride()), _p(dst), L.i64arr(dst.stride()),
                                   L.i64arr(src.shape), _dt(src), s), "bi_copy4d")
    return dst


# ------------------------------------------------------------------ status

def last_device_error(device=None):
    """Synchronise the current stream and read+clear the device error word: (status, code)."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    code = ctypes.c_uint32(0)
    with _On(dev) as s:
        st = L.load().bi_last_device_error(s, ctypes.byref(code))
    return st, code.value


def launch_count() -> int:
    return int(L.load().bi_launch_count())


def version() -> int:
    return int(L.load().bi_version())


def debug_wait_probe(limit_us: int, device=None):
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    with _On(dev) as s:
        L.check(L.load().bi_debug_wait_probe(int(limit_us), s), "bi_debug_wait_probe")
