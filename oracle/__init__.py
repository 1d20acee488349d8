"""fp64 CPU oracle for the batch-invariant GEMM / attention path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only users.  The product package never
imports this module, and this module never imports the product package.

The arithmetic lives in ``oracle.c`` (plain C, fp64, natural summation order,
OpenMP over independent output rows).  This file only builds it with gcc,
loads it with ctypes and marshals numpy float64 arrays.  GEMM and attention
functions return ``(result, normaliser)`` where the normaliser is the sum of
the magnitudes of the terms, the quantity the tolerances are stated against.

Definitions follow the "mlx-batch-invariant" README ("Use", "How the kernels
work", "Accuracy"); the readings taken where it is silent are listed in
``oracle.c``'s header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64


def compile_source(src: str, out: str) -> str:
    """gcc -O2 -fopenmp, no FMA contraction (same results on x86-64 and aarch64)."""
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared",
           "-fPIC", "-std=c11", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (skipped when up to date)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _f64(a) -> np.ndarray:
    """Exact conversion to a C-contiguous float64 array (bf16/fp16/fp32 embed exactly)."""
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


class Oracle:
    """The oracle bound to one compiled library (the real one, or a test variant)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_linear.argtypes = [_I64, _I64, _I64, _D, _D, _D, _D, _D]
        lib.oracle_matmul.argtypes = [_I64, _I64, _I64, _D, _D, _D, _D]
        lib.oracle_addmm.argtypes = [_I64, _I64, _I64, _D, ctypes.c_int, _D, _D,
                                     ctypes.c_double, ctypes.c_double, _D, _D]
        lib.oracle_sdpa.argtypes = [_I64, _I64, _I64, _I64, _I64, _I64, _D, _D, _D,
                                    ctypes.c_double, ctypes.c_int, _I64, _D, _D]
        lib.oracle_sdpa_ex.argtypes = [_I64, _I64, _I64, _I64, _I64, _I64, _D, _D, _D,
                                       ctypes.c_double, ctypes.c_int, _I64, _D,
                                       ctypes.POINTER(ctypes.c_ubyte), _D, _D]
        lib.oracle_qlinear.argtypes = [_I64, _I64, _I64, _D, ctypes.POINTER(ctypes.c_uint32),
                                       _I64, _D, _D, _I64, ctypes.c_int, _I64, _D, _D, _D]
        lib.oracle_rmsnorm.argtypes = [_I64, _I64, _D, _D, ctypes.c_double, _D]
        lib.oracle_rope.argtypes = [_I64, _I64, _I64, _D, ctypes.POINTER(ctypes.c_int64),
                                    ctypes.c_double, _D]
        lib.oracle_swiglu.argtypes = [_I64, _I64, _D, _D]
        self.lib = lib

    def num_threads(self) -> int:
        """OpenMP threads the oracle uses (OMP_NUM_THREADS, else the host's cores)."""
        return int(self.lib.oracle_num_threads())

    def linear(self, x, w, bias=None):
        """y = x . w^T + bias, x[M,K], w[N,K], bias[N] or None."""
        x, w = _f64(x), _f64(w)
        bias = None if bias is None else _f64(bias)
        M, K = x.shape
        N = w.shape[0]
        assert w.shape == (N, K) and (bias is None or bias.shape == (N,))
        y = np.empty((M, N)); nrm = np.empty((M, N))
        self.lib.oracle_linear(M, N, K, _p(x), _p(w), _p(bias), _p(y), _p(nrm))
        return y, nrm

    def matmul(self, a, b):
        """y = a . b, a[M,K], b[K,N]."""
        a, b = _f64(a), _f64(b)
        M, K = a.shape
        N = b.shape[1]
        assert b.shape == (K, N)
        y = np.empty((M, N)); nrm = np.empty((M, N))
        self.lib.oracle_matmul(M, N, K, _p(a), _p(b), _p(y), _p(nrm))
        return y, nrm

    def addmm(self, c, a, b, alpha=1.0, beta=1.0):
        """y = beta*c + alpha*(a . b); c is [M,N] or a row [N]."""
        c, a, b = _f64(c), _f64(a), _f64(b)
        M, K = a.shape
        N = b.shape[1]
        c_row = 1 if c.ndim == 1 else 0
        assert c.shape == ((N,) if c_row else (M, N))
        y = np.empty((M, N)); nrm = np.empty((M, N))
        self.lib.oracle_addmm(M, N, K, _p(c), c_row, _p(a), _p(b), float(alpha),
                              float(beta), _p(y), _p(nrm))
        return y, nrm

    def sdpa(self, q, k, v, causal=True, q_offset=None, scale=None):
        """Attention with GQA: q[B,H,Lq,D], k/v[B,Hkv,Lkv,D] -> o[B,H,Lq,D].

        q_offset defaults to Lkv - Lq (the last query sees the whole cache);
        scale defaults to 1/sqrt(D).
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, Lq, D = q.shape
        Hkv, Lkv = k.shape[1], k.shape[2]
        assert k.shape == (B, Hkv, Lkv, D) and v.shape == k.shape and H % Hkv == 0
        if q_offset is None:
            q_offset = Lkv - Lq
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        o = np.empty((B, H, Lq, D)); nrm = np.empty((B, H, Lq, D))
        self.lib.oracle_sdpa(B, H, Hkv, Lq, Lkv, D, _p(q), _p(k), _p(v), float(scale),
                             1 if causal else 0, int(q_offset), _p(o), _p(nrm))
        return o, nrm

    def sdpa_ex(self, q, k, v, causal=True, q_offset=None, scale=None, sinks=None, mask=None):
        """sdpa with optional attention sinks (sinks[H], logits in the units of the scaled
        scores) and an optional boolean array mask [B,H,Lq,Lkv] (or broadcastable to it),
        nonzero = visible; a mask overrides `causal`."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, Lq, D = q.shape
        Hkv, Lkv = k.shape[1], k.shape[2]
        assert k.shape == (B, Hkv, Lkv, D) and v.shape == k.shape and H % Hkv == 0
        if q_offset is None:
            q_offset = Lkv - Lq
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        sk = None if sinks is None else _f64(sinks).reshape(H)
        mk = None
        if mask is not None:
            if hasattr(mask, "detach"):
                mask = mask.detach().to("cpu").numpy()
            mk = np.ascontiguousarray(np.broadcast_to(np.asarray(mask) != 0, (B, H, Lq, Lkv)),
                                      dtype=np.uint8)
        o = np.empty((B, H, Lq, D)); nrm = np.empty((B, H, Lq, D))
        self.lib.oracle_sdpa_ex(B, H, Hkv, Lq, Lkv, D, _p(q), _p(k), _p(v), float(scale),
                                1 if causal else 0, int(q_offset), _p(sk),
                                None if mk is None else mk.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)),
                                _p(o), _p(nrm))
        return o, nrm

    def qlinear(self, x, wq, scales, biases, bits, group_size, bias=None):
        """Group-wise affine quantized linear: x[M,K], wq uint32 [N, K*bits/32] (packed
        along K, lowest field first), scales/biases [N, K/group_size]; y = x . w^T + bias."""
        x, scales, biases = _f64(x), _f64(scales), _f64(biases)
        if hasattr(wq, "detach"):
            wq = wq.detach().to("cpu").numpy()
        wq = np.ascontiguousarray(np.asarray(wq).view(np.uint32))
        bias = None if bias is None else _f64(bias)
        M, K = x.shape
        N = wq.shape[0]
        assert bits in (2, 4, 8) and K % group_size == 0 and K * bits % 32 == 0
        assert wq.shape == (N, K * bits // 32) and scales.shape == (N, K // group_size)
        assert biases.shape == scales.shape and (bias is None or bias.shape == (N,))
        y = np.empty((M, N)); nrm = np.empty((M, N))
        self.lib.oracle_qlinear(M, N, K, _p(x), wq.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)),
                                wq.shape[1], _p(scales), _p(biases), scales.shape[1], int(bits),
                                int(group_size), _p(bias), _p(y), _p(nrm))
        return y, nrm

    def rmsnorm(self, x, w, eps=1e-6):
        """y = x / sqrt(mean(x^2) + eps) * w over the last dim; x[M,N], w[N]."""
        x, w = _f64(x), _f64(w)
        M, N = x.shape
        y = np.empty((M, N))
        self.lib.oracle_rmsnorm(M, N, _p(x), _p(w), float(eps), _p(y))
        return y

    def rope(self, x, pos, base=10000.0):
        """Rotate-half RoPE: x[T,nh,D], pos[T] absolute positions."""
        x = _f64(x)
        T, nh, D = x.shape
        pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64))
        assert pos.shape == (T,) and D % 2 == 0
        y = np.empty_like(x)
        self.lib.oracle_rope(T, nh, D, _p(x),
                             pos.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                             float(base), _p(y))
        return y

    def swiglu(self, gu):
        """gu[M, 2I] = [gate | up] -> silu(gate) * up, [M, I]."""
        gu = _f64(gu)
        M, I2 = gu.shape
        assert I2 % 2 == 0
        y = np.empty((M, I2 // 2))
        self.lib.oracle_swiglu(M, I2 // 2, _p(gu), _p(y))
        return y


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def num_threads():
    return default().num_threads()


def linear(x, w, bias=None):
    return default().linear(x, w, bias)


def matmul(a, b):
    return default().matmul(a, b)


def addmm(c, a, b, alpha=1.0, beta=1.0):
    return default().addmm(c, a, b, alpha, beta)


def sdpa(q, k, v, causal=True, q_offset=None, scale=None):
    return default().sdpa(q, k, v, causal, q_offset, scale)


def sdpa_ex(q, k, v, causal=True, q_offset=None, scale=None, sinks=None, mask=None):
    return default().sdpa_ex(q, k, v, causal, q_offset, scale, sinks, mask)


def qlinear(x, wq, scales, biases, bits, group_size, bias=None):
    return default().qlinear(x, wq, scales, biases, bits, group_size, bias)


def rmsnorm(x, w, eps=1e-6):
    return default().rmsnorm(x, w, eps)


def rope(x, pos, base=10000.0):
    return default().rope(x, pos, base)


def swiglu(gu):
    return default().swiglu(gu)
