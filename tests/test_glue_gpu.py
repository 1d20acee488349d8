"""Decoder glue kernels against the fp64 oracle, and the device status machinery (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from attention_bi_matmul_gb300 import synth
from tolerances import assert_same_bits, check_close

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


@pytest.fixture(scope="module")
def bi():
    import __graft_entry__
    __graft_entry__.build()
    import attention_bi_matmul_gb300 as m
    torch.cuda.set_device(0)
    return m


@pytest.mark.parametrize("dt", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("M,N", [(1, 2048), (37, 1000), (300, 5632)])
def test_rmsnorm(bi, dt, M, N):
    x = synth.normal((M, N), 1, 1.0, dt)
    w = synth.normal((N,), 2, 1.0, dt)
    y = bi.rmsnorm(x.cuda(), w.cuda(), 1e-6)
    ref = oracle.rmsnorm(x, w, 1e-6)
    check_close(y, ref, np.abs(ref), DT[dt], "rmsnorm", floor=1e-30)
    # a row's bits do not depend on the other rows
    y1 = bi.rmsnorm(x[M - 1:].cuda(), w.cuda(), 1e-6)
    assert_same_bits(y1, y[M - 1:], "rmsnorm last row alone")


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("pos0", [0, 5, 4095, 8190])
def test_rope(bi, dt, pos0):
    B, L, nh, D = 2, 7, 6, 128
    x = synth.normal((B, L, nh, D), 3, 1.0, dt)
    y = bi.rope(x.cuda(), pos0)
    pos = np.tile(np.arange(pos0, pos0 + L), B)
    xf = x.reshape(B * L, nh, D)
    ref = oracle.rope(xf, pos).reshape(B, L, nh, D)
    xd = xf.double().numpy()
    half = D // 2
    mag = np.concatenate([np.abs(xd[..., :half]) + np.abs(xd[..., half:])] * 2, -1)
    check_close(y, ref, mag.reshape(B, L, nh, D), DT[dt], "rope pos0=%d" % pos0)
    # written through strides into a [B, nh, Lmax, D] cache slice
    cache = torch.zeros((B, nh, pos0 + L + 3, D), dtype=DT[dt], device="cuda")
    bi.rope(x.cuda(), pos0, out=cache[:, :, pos0:pos0 + L].transpose(1, 2))
    assert_same_bits(cache[:, :, pos0:pos0 + L].transpose(1, 2), y, "rope into cache view")


@pytest.mark.parametrize("dt", ["bf16", "fp16", "fp32"])
def test_swiglu(bi, dt):
    M, I = 33, 5632
    gu = synth.normal((M, 2 * I), 4, 2.0, dt)
    y = bi.swiglu(gu.cuda())
    ref = oracle.swiglu(gu)
    check_close(y, ref, np.abs(ref), DT[dt], "swiglu", floor=1e-30)


@pytest.mark.parametrize("dt", ["bf16", "fp16", "fp32"])
def test_add_embedding_copy(bi, dt):
    a = synth.normal((1000,), 5, 1.0, dt)
    b = synth.normal((1000,), 6, 1.0, dt)
    y = bi.add(a.cuda(), b.cuda()).cpu().double()
    ref = a.double() + b.double()
    check_close(y, ref.numpy(), np.abs(ref.numpy()), DT[dt], "add", floor=1e-30)
    table = synth.normal((100, 64), 7, 1.0, dt)
    ids = synth.uniform_ids((3, 5), 100, 8)
    e = bi.embedding(ids.cuda(), table.cuda())
    assert torch.equal(e.cpu(), table[ids]), "embedding gather"
    src = synth.normal((2, 5, 3, 64), 9, 1.0, dt)
    dst = torch.zeros((2, 3, 9, 64), dtype=DT[dt], device="cuda")
    bi.copy4d(src.cuda(), dst[:, :, 2:7].transpose(1, 2))
    assert torch.equal(dst[:, :, 2:7].transpose(1, 2).cpu(), src)
    assert torch.count_nonzero(dst[:, :, :2]) == 0 and torch.count_nonzero(dst[:, :, 7:]) == 0


def test_embedding_bad_id_sets_error_word(bi):
    bi.last_device_error()  # clear
    table = synth.normal((10, 16), 1, 1.0, "bf16").cuda()
    ids = torch.tensor([1, 10, -1, 3], dtype=torch.int64, device="cuda")
    e = bi.embedding(ids, table)
    st, code = bi.last_device_error()
    assert st == 1 and code & 2, (st, code)       # BI_ERR_INVALID_ARG, bad-index bit
    assert torch.count_nonzero(e[1]) == 0 and torch.count_nonzero(e[2]) == 0
    assert torch.equal(e[0], table[1])
    assert bi.last_device_error()[0] == 0         # cleared by the read


def test_bounded_wait_reports_timeout_and_context_survives(bi):
    """A barrier wait that nothing completes runs out after its limit; the kernel records
    BI_ERR_TIMEOUT and returns; the context stays usable."""
    bi.last_device_error()
    bi.debug_wait_probe(100000)   # 0.1 s
    st, code = bi.last_device_error()
    assert st == 5 and code & 1, (st, code)       # BI_ERR_TIMEOUT
    x, w = synth.gemm16(4, 64, 64, "bf16", seed=1, layout="linear")
    y = bi.linear(x.cuda(), w.cuda())
    ref, nrm = oracle.linear(x, w)
    check_close(y, ref, nrm, torch.bfloat16, "linear after timeout")
    assert bi.last_device_error()[0] == 0


def test_python_errors(bi):
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bi.BiError):
        bi.linear(x[:, 1:], w[:, 1:])      # misaligned row start -> BI_ERR_ALIGNMENT
    with pytest.raises(ValueError):
        bi.linear(x.cpu(), w.cpu())
    q = torch.zeros((1, 4, 1, 80), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bi.BiError):
        bi.sdpa(q, q[:, :1], q[:, :1])     # head dim 80 not built
