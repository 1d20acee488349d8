"""The C-ABI library builds, loads, exports every declared symbol, and rejects bad
arguments on the host (CPU only: no call here reaches a kernel launch)."""
import ctypes
import subprocess

import pytest

from attention_bi_matmul_gb300 import _lib as L
from attention_bi_matmul_gb300 import build as B


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def test_header_matches_binding():
    declared = L.header_functions()
    assert sorted(set(declared)) == sorted(L.SIGNATURES), (
        "include/bi.h and the ctypes signatures disagree")


def test_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], stdout=subprocess.PIPE,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in L.header_functions():
        assert name in exported, "%s is declared in include/bi.h but not exported" % name
        assert getattr(lib, name) is not None


def test_status_strings_and_version(lib):
    for st in range(6):
        s = lib.bi_status_string(st).decode()
        assert s.startswith("BI_"), s
    assert lib.bi_version() == 100


def test_gemm_config_ignores_M_and_is_host_only(lib):
    bn, st = ctypes.c_int(), ctypes.c_int()
    for N in (8, 512, 4096, 11008, 14336, 38912):
        for K in (8, 4096, 8192, 16384):
            for layout in (0, 1):
                assert lib.bi_gemm_config(N, K, L.BI_BF16, layout, ctypes.byref(bn),
                                          ctypes.byref(st)) == L.BI_OK
                assert bn.value == (256 if K >= 8192 else 128)
                assert st.value == (4 if bn.value == 256 else 3)
    assert lib.bi_gemm_config(0, 4096, L.BI_BF16, 0, None, None) == L.BI_ERR_INVALID_ARG
    assert lib.bi_gemm_config(64, 64, 7, 0, None, None) == L.BI_ERR_UNSUPPORTED


def test_host_validation_rejects_before_launch(lib):
    nul = None
    p = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    s = ctypes.c_void_p(0)
    # null pointers / bad sizes
    assert lib.bi_linear(nul, 8, p, 8, nul, p, 8, 1, 8, 8, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG
    assert lib.bi_linear(p, 8, p, 8, nul, p, 8, 1, 0, 8, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG
    assert lib.bi_linear(p, 8, p, 8, nul, p, 8, 1, 8, 0, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG
    assert lib.bi_linear(p, 4, p, 8, nul, p, 8, 1, 8, 8, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG
    # alignment of 16-bit operands: a pointer off by 2 bytes, a row stride not a multiple of 8
    q = ctypes.c_void_p(4096 + 2)
    assert lib.bi_matmul(q, 16, p, 16, p, 16, 2, 16, 16, L.BI_BF16, s) == L.BI_ERR_ALIGNMENT
    assert lib.bi_matmul(p, 20, p, 16, p, 16, 2, 16, 20, L.BI_F16, s) == L.BI_ERR_ALIGNMENT
    # unknown dtype
    assert lib.bi_matmul(p, 16, p, 16, p, 16, 2, 16, 16, 9, s) == L.BI_ERR_UNSUPPORTED
    # addmm: c must be given; ldc in (0, N) is invalid
    assert lib.bi_addmm(nul, 0, p, 16, p, 16, p, 16, 2, 16, 16, 1.0, 1.0, L.BI_BF16, s) \
        == L.BI_ERR_INVALID_ARG
    assert lib.bi_addmm(p, 8, p, 16, p, 16, p, 16, 2, 16, 16, 1.0, 1.0, L.BI_BF16, s) \
        == L.BI_ERR_INVALID_ARG
    # M == 0 is a no-op
    assert lib.bi_linear(p, 8, p, 8, nul, p, 8, 0, 8, 8, L.BI_BF16, s) == L.BI_OK


def test_matmul_batched_validation(lib):
    p = ctypes.c_void_p(4096)
    s = ctypes.c_void_p(0)

    def call(sa=64 * 64, sb=64 * 64, sy=64 * 64, batch=3, layout=1, dt=L.BI_BF16, M=64):
        return lib.bi_matmul_batched(p, 64, sa, p, 64, sb, layout, p, 64, sy, batch, M, 64, 64,
                                     dt, s)

    assert call(layout=2) == L.BI_ERR_INVALID_ARG
    assert call(batch=-1) == L.BI_ERR_INVALID_ARG
    assert call(sa=-8) == L.BI_ERR_INVALID_ARG
    assert call(sy=63 * 64) == L.BI_ERR_INVALID_ARG           # entries of y overlap
    assert call(sa=12) == L.BI_ERR_ALIGNMENT                   # 16-bit: multiples of 8
    assert call(batch=70000) == L.BI_ERR_UNSUPPORTED
    assert call(batch=0) == L.BI_OK                            # empty: no-op
    assert call(M=0) == L.BI_OK
    assert call(sa=12, dt=L.BI_F32) != L.BI_ERR_ALIGNMENT      # fp32 takes any stride


def test_qlinear_validation(lib):
    p = ctypes.c_void_p(4096)
    s = ctypes.c_void_p(0)

    def call(bits=4, gs=64, K=256, ldq=None, ldx=256, dt=L.BI_BF16, ldsb=None, M=8, xp=p):
        ldq = K * bits // 32 if ldq is None else ldq
        ldsb = max(8, K // gs) if ldsb is None else ldsb
        return lib.bi_qlinear(xp, ldx, p, ldq, p, p, ldsb, None, p, 64, M, 64, K, bits, gs, dt, s)

    assert call(bits=3) == L.BI_ERR_UNSUPPORTED               # 3-bit packing not built
    assert call(gs=16) == L.BI_ERR_UNSUPPORTED
    assert call(dt=L.BI_F32) == L.BI_ERR_UNSUPPORTED
    assert call(K=96, ldx=96, gs=32) == L.BI_ERR_UNSUPPORTED   # K not a multiple of 64
    assert call(K=192, ldx=192, gs=128) == L.BI_ERR_INVALID_ARG   # K not a multiple of gs
    assert call(ldq=16) == L.BI_ERR_INVALID_ARG                # row shorter than K*bits/32
    assert call(ldsb=3) == L.BI_ERR_INVALID_ARG
    assert call(ldsb=12) == L.BI_ERR_ALIGNMENT                 # scale rows in 16-byte boxes
    assert call(ldq=34) == L.BI_ERR_ALIGNMENT                  # 16-byte rows for the copy
    assert call(xp=ctypes.c_void_p(4104)) == L.BI_ERR_ALIGNMENT
    assert call(M=0) == L.BI_OK


def test_sdpa_validation(lib):
    p = ctypes.c_void_p(4096)
    s = ctypes.c_void_p(0)
    st4 = L.i64arr([32 * 9 * 128, 9 * 128, 128, 1])
    args = lambda **kw: dict(dict(B=1, H=4, Hkv=2, Lq=1, Lkv=9, D=128, scale=0.0,
                                  mask=L.BI_MASK_CAUSAL, q_offset=-1, dt=L.BI_BF16), **kw)

    def call(**kw):
        a = args(**kw)
        return lib.bi_sdpa(p, st4, p, st4, p, st4, p, st4, a["B"], a["H"], a["Hkv"], a["Lq"],
                           a["Lkv"], a["D"], a["scale"], a["mask"], a["q_offset"], a["dt"], s)

    assert call(H=3) == L.BI_ERR_INVALID_ARG                  # H % Hkv != 0
    assert call(q_offset=9) == L.BI_ERR_INVALID_ARG           # q_offset + Lq > Lkv
    assert call(Lq=10) == L.BI_ERR_INVALID_ARG                # default offset negative
    assert call(mask=5) == L.BI_ERR_UNSUPPORTED
    assert call(dt=L.BI_F32) == L.BI_ERR_UNSUPPORTED
    assert call(D=80) == L.BI_ERR_UNSUPPORTED                 # head dim not built
    assert call(D=288) == L.BI_ERR_UNSUPPORTED
    assert call(D=32) == L.BI_ERR_UNSUPPORTED
    # Without the causal rule the positions only align the tiles: more queries than
    # keys pass validation; no keys at all do not.
    assert call(Lq=10, mask=L.BI_MASK_NONE) != L.BI_ERR_INVALID_ARG
    assert call(Lkv=0, q_offset=0, mask=L.BI_MASK_NONE) == L.BI_ERR_INVALID_ARG
    assert call(H=64, Hkv=2) == L.BI_ERR_UNSUPPORTED          # group of 32 not built
    assert call(Lq=0) == L.BI_OK                              # empty: no-op
    bad = L.i64arr([32 * 9 * 128, 9 * 128, 128, 2])
    assert lib.bi_sdpa(p, bad, p, st4, p, st4, p, st4, 1, 4, 2, 1, 9, 128, 0.0,
                       L.BI_MASK_CAUSAL, -1, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG


def test_sdpa_ex_validation(lib):
    p = ctypes.c_void_p(4096)
    s = ctypes.c_void_p(0)
    st4 = L.i64arr([32 * 9 * 128, 9 * 128, 128, 1])
    ms_ok = L.i64arr([0, 0, 9, 1])

    def call(mask=L.BI_MASK_ARRAY, sinks=None, marr=p, ms=ms_ok):
        return lib.bi_sdpa_ex(p, st4, p, st4, p, st4, p, st4, 1, 4, 2, 1, 9, 128, 0.0, mask, -1,
                              sinks, marr, ms, L.BI_BF16, s)

    assert call(marr=None) == L.BI_ERR_INVALID_ARG            # array mode without a mask
    assert call(ms=None) == L.BI_ERR_INVALID_ARG
    assert call(ms=L.i64arr([0, 0, 9, 2])) == L.BI_ERR_INVALID_ARG   # last dim not contiguous
    assert call(ms=L.i64arr([0, -1, 9, 1])) == L.BI_ERR_INVALID_ARG
    assert call(mask=L.BI_MASK_CAUSAL) == L.BI_ERR_INVALID_ARG        # mask given, mode causal
    assert call(mask=L.BI_MASK_CAUSAL, marr=None, sinks=ctypes.c_void_p(4098)) == L.BI_ERR_ALIGNMENT
    # bi_sdpa has no mask argument: the array form is refused there.
    assert lib.bi_sdpa(p, st4, p, st4, p, st4, p, st4, 1, 4, 2, 1, 9, 128, 0.0,
                       L.BI_MASK_ARRAY, -1, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG


def test_glue_validation(lib):
    p = ctypes.c_void_p(4096)
    s = ctypes.c_void_p(0)
    assert lib.bi_rmsnorm(p, 8, p, p, 8, 1, 16, 1e-6, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG
    assert lib.bi_rmsnorm(p, 16, p, p, 16, 1, 16, -1.0, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG
    assert lib.bi_swiglu(p, 10, p, 8, 1, 8, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG
    x4 = L.i64arr([1024, 256, 128, 1])
    assert lib.bi_rope(p, x4, p, x4, 1, 2, 2, 127, 0, 1e4, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG
    assert lib.bi_rope(p, x4, p, x4, 1, 2, 2, 128, 0, 1e4, L.BI_F32, s) == L.BI_ERR_UNSUPPORTED
    assert lib.bi_embedding(None, 4, p, 8, 10, p, 8, 8, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG
    assert lib.bi_add(p, p, p, -1, L.BI_BF16, s) == L.BI_ERR_INVALID_ARG
    assert lib.bi_debug_wait_probe(0, s) == L.BI_ERR_INVALID_ARG
    assert lib.bi_debug_wait_probe(3000000, s) == L.BI_ERR_INVALID_ARG


def test_element_alignment_of_per_element_operands(lib):
    """Pointers the kernels read or write one element at a time (the bias, addmm's c, the
    glue ops' tensors) must be aligned to their element size, and the embedding ids to 8
    bytes; a misaligned one is refused on the host, before any launch."""
    p = ctypes.c_void_p(4096)
    odd = ctypes.c_void_p(4096 + 1)          # misaligned for 16-bit elements
    half = ctypes.c_void_p(4096 + 2)         # 2-byte aligned: fine for 16-bit, not for fp32
    s = ctypes.c_void_p(0)
    # bias of bi_linear
    assert lib.bi_linear(p, 16, p, 16, odd, p, 16, 2, 16, 16, L.BI_BF16, s) == L.BI_ERR_ALIGNMENT
    assert lib.bi_linear(p, 16, p, 16, half, p, 16, 2, 16, 16, L.BI_F32, s) == L.BI_ERR_ALIGNMENT
    # c of bi_addmm, full and broadcast row
    for ldc in (16, 0):
        assert lib.bi_addmm(odd, ldc, p, 16, p, 16, p, 16, 2, 16, 16, 1.0, 1.0, L.BI_F16, s) \
            == L.BI_ERR_ALIGNMENT
        assert lib.bi_addmm(half, ldc, p, 16, p, 16, p, 16, 2, 16, 16, 1.0, 1.0, L.BI_F32, s) \
            == L.BI_ERR_ALIGNMENT
    # glue ops
    assert lib.bi_rmsnorm(odd, 16, p, p, 16, 1, 16, 1e-6, L.BI_BF16, s) == L.BI_ERR_ALIGNMENT
    assert lib.bi_rmsnorm(p, 16, half, p, 16, 1, 16, 1e-6, L.BI_F32, s) == L.BI_ERR_ALIGNMENT
    assert lib.bi_swiglu(p, 16, odd, 8, 1, 8, L.BI_BF16, s) == L.BI_ERR_ALIGNMENT
    assert lib.bi_add(p, odd, p, 4, L.BI_F16, s) == L.BI_ERR_ALIGNMENT
    x4 = L.i64arr([1024, 256, 128, 1])
    assert lib.bi_rope(odd, x4, p, x4, 1, 2, 2, 128, 0, 1e4, L.BI_BF16, s) == L.BI_ERR_ALIGNMENT
    n4 = L.i64arr([1, 1, 1, 4])
    assert lib.bi_copy4d(p, x4, odd, x4, n4, L.BI_BF16, s) == L.BI_ERR_ALIGNMENT
    # embedding: int64 ids 8-byte aligned; at most 2^31 - 1 ids (one block each)
    assert lib.bi_embedding(ctypes.c_void_p(4096 + 4), 4, p, 8, 10, p, 8, 8, L.BI_BF16, s) \
        == L.BI_ERR_ALIGNMENT
    assert lib.bi_embedding(p, 1 << 31, p, 8, 10, p, 8, 8, L.BI_BF16, s) == L.BI_ERR_UNSUPPORTED
