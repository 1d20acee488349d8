"""ctypes binding of ``libbi.so`` (include/bi.h).  Argument marshalling only.

The library is loaded on first use.  If it has not been built, loading fails
with an error: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbi.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "bi.h")

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i64p = ctypes.POINTER(ctypes.c_int64)
_f = ctypes.c_float
_int = ctypes.c_int
_st = ctypes.c_int  # bi_status

# name -> (restype, argtypes); the order follows include/bi.h
SIGNATURES = {
    "bi_linear": (_st, [_vp, _i64, _vp, _i64, _vp, _vp, _i64, _i64, _i64, _i64, _int, _vp]),
    "bi_matmul": (_st, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _i64, _int, _vp]),
    "bi_matmul_batched": (_st, [_vp, _i64, _i64, _vp, _i64, _i64, _int, _vp, _i64, _i64, _i64,
                                _i64, _i64, _i64, _int, _vp]),
    "bi_qlinear": (_st, [_vp, _i64, _vp, _i64, _vp, _vp, _i64, _vp, _vp, _i64, _i64, _i64, _i64,
                         _int, _int, _int, _vp]),
    "bi_addmm": (_st, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _i64, _f, _f,
                       _int, _vp]),
    "bi_gemm_config": (_st, [_i64, _i64, _int, _int, ctypes.POINTER(_int),
                             ctypes.POINTER(_int)]),
    "bi_sdpa": (_st, [_vp, _i64p, _vp, _i64p, _vp, _i64p, _vp, _i64p, _i64, _i64, _i64, _i64,
                      _i64, _i64, _f, _int, _i64, _int, _vp]),
    "bi_sdpa_ex": (_st, [_vp, _i64p, _vp, _i64p, _vp, _i64p, _vp, _i64p, _i64, _i64, _i64, _i64,
                         _i64, _i64, _f, _int, _i64, _vp, _vp, _i64p, _int, _vp]),
    "bi_rmsnorm": (_st, [_vp, _i64, _vp, _vp, _i64, _i64, _i64, _f, _int, _vp]),
    "bi_rope": (_st, [_vp, _i64p, _vp, _i64p, _i64, _i64, _i64, _i64, _i64, _f, _int, _vp]),
    "bi_swiglu": (_st, [_vp, _i64, _vp, _i64, _i64, _i64, _int, _vp]),
    "bi_add": (_st, [_vp, _vp, _vp, _i64, _int, _vp]),
    "bi_embedding": (_st, [_vp, _i64, _vp, _i64, _i64, _vp, _i64, _i64, _int, _vp]),
    "bi_copy4d": (_st, [_vp, _i64p, _vp, _i64p, _i64p, _int, _vp]),
    "bi_status_string": (ctypes.c_char_p, [_int]),
    "bi_version": (_int, []),
    "bi_last_device_error": (_st, [_vp, ctypes.POINTER(ctypes.c_uint32)]),
    "bi_launch_count": (_i64, []),
    "bi_debug_wait_probe": (_st, [_i64, _vp]),
}

BI_OK, BI_ERR_INVALID_ARG, BI_ERR_UNSUPPORTED, BI_ERR_ALIGNMENT, BI_ERR_CUDA, BI_ERR_TIMEOUT = range(6)
BI_F32, BI_F16, BI_BF16 = 0, 1, 2
BI_MASK_NONE, BI_MASK_CAUSAL, BI_MASK_ARRAY = 0, 1, 2

_lib = None


class BiError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s" % (what, status_string(status)))


def header_functions() -> list[str]:
    """Names of the functions include/bi.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"\b(bi_[a-z0-9_]+)\s*\(", text)


def load(path: str | None = None):
    """Load libbi.so (once) and declare every signature.  Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError("libbi.so is not built (%s); run __graft_entry__.build() or "
                          "python -m attention_bi_matmul_gb300.build" % p)
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().bi_status_string(int(status)).decode()
    except ImportError:
        return "bi_status %d" % status


def check(status: int, what: str):
    if status != BI_OK:
        raise BiError(status, what)


def i64arr(vals):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])
