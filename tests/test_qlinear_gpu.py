"""Quantized linear (group-wise affine 2/4/8-bit weights): parity with the fp64 oracle,
the exact dequantised value, and batch invariance (GPU, through bi_qlinear)."""
import numpy as np
import pytest
import torch

import oracle
from attention_bi_matmul_gb300 import synth
from tolerances import assert_same_bits, check_close

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(scope="module")
def bi():
    import __graft_entry__
    __graft_entry__.build()
    import attention_bi_matmul_gb300 as m
    torch.cuda.set_device(0)
    return m


def _no_device_error(bi):
    st, code = bi.last_device_error()
    assert st == 0, "device error word %#x" % code


def _fields(wq, bits):
    """[N, W] packed words -> [N, W*32/bits] fields (lowest first), via numpy bit unpacking."""
    w = np.ascontiguousarray(wq.cpu().numpy()).view("<u4")
    b = np.unpackbits(w.view(np.uint8), axis=1, bitorder="little").astype(np.int64)
    return (b.reshape(w.shape[0], -1, bits) * (1 << np.arange(bits))).sum(axis=2)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("gs", [32, 64, 128])
def test_parity(bi, dt, bits, gs):
    M, N, K = 37, 300, 512
    x = synth.normal((M, K), bits + gs, 1.0, dt)
    wq, sc, bs = synth.qweights(N, K, bits, gs, dt, seed=bits * gs)
    bias = synth.normal((N,), 3, 0.1, dt)
    for b in (None, bias):
        y = bi.qlinear(x.cuda(), wq.cuda(), sc.cuda(), bs.cuda(), bits, gs,
                       None if b is None else b.cuda())
        ref, nrm = oracle.qlinear(x, wq, sc, bs, bits, gs, b)
        check_close(y, ref, nrm, DT[dt], "qlinear %s %d-bit gs%d bias=%s" % (dt, bits, gs, b is not None))
    _no_device_error(bi)


@pytest.mark.parametrize("M", [1, 3, 16, 64, 65, 130])
@pytest.mark.parametrize("N", [64, 200, 257])
def test_ragged_shapes(bi, M, N):
    K, bits, gs = 256, 4, 64
    x = synth.normal((M, K), M, 1.0, "bf16")
    wq, sc, bs = synth.qweights(N, K, bits, gs, "bf16", seed=N)
    y = bi.qlinear(x.cuda(), wq.cuda(), sc.cuda(), bs.cuda(), bits, gs)
    ref, nrm = oracle.qlinear(x, wq, sc, bs, bits, gs)
    check_close(y, ref, nrm, torch.bfloat16, "qlinear M=%d N=%d" % (M, N))


def test_unaligned_scale_rows_are_padded(bi):
    """K / group_size = 172 groups (K = 11008): rows not a multiple of 8 elements take the
    wrapper's padded copy and give the same bits as an aligned layout of the same values."""
    M, N, K, bits, gs = 5, 256, 11008, 4, 64
    x = synth.normal((M, K), 21, 1.0, "bf16").cuda()
    wq, sc, bs = (t.cuda() for t in synth.qweights(N, K, bits, gs, "bf16", seed=22))
    assert sc.stride(0) % 8 != 0
    y = bi.qlinear(x, wq, sc, bs, bits, gs)
    pad = torch.zeros((N, 2, 176), dtype=sc.dtype, device="cuda")
    pad[:, 0, :172] = sc
    pad[:, 1, :172] = bs
    y2 = bi.qlinear(x, wq, pad[:, 0, :172], pad[:, 1, :172], bits, gs)
    assert_same_bits(y, y2, "padded vs aligned scale rows")
    ref, nrm = oracle.qlinear(x.cpu(), wq.cpu(), sc.cpu(), bs.cpu(), bits, gs)
    check_close(y, ref, nrm, torch.bfloat16, "qlinear K=11008")


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_dequantised_value_is_rounded_once(bi, dt, bits):
    """One-hot activations read the dequantised weights out: they must equal s*q + b,
    computed exactly, rounded once to the activation dtype."""
    N, K, gs = 130, 128, 32
    wq, sc, bs = synth.qweights(N, K, bits, gs, dt, seed=7 + bits)
    x = torch.eye(K, dtype=DT[dt])
    y = bi.qlinear(x.cuda(), wq.cuda(), sc.cuda(), bs.cuda(), bits, gs).cpu()   # [K, N] = w^T
    q = torch.from_numpy(_fields(wq, bits)).double()
    s = sc.double().repeat_interleave(gs, dim=1)
    b = bs.double().repeat_interleave(gs, dim=1)
    exact = s * q + b                        # exact in fp64
    # torch rounds fp64 -> 16-bit through fp32: make sure that first step is exact, so
    # the reference is the single rounding of the exact value.
    assert torch.equal(exact.float().double(), exact)
    want = exact.to(DT[dt])
    assert_same_bits(y.t().contiguous(), want, "dequantised %s %d-bit" % (dt, bits))


def test_integer_exact(bi):
    """scale 1, bias 0, activations in {-1, 0, 1}: every sum is a small integer, exact."""
    # |y| stays within the dtype's exact integers: fp16 2048, bf16 256.
    for dt, bits, K, nnz in (("fp16", 4, 128, 128), ("bf16", 2, 64, 64), ("fp16", 8, 64, 8)):
        M, N, gs = 9, 140, 32
        rng = np.random.default_rng(bits)
        xv = rng.integers(-1, 2, size=(M, K)).astype(np.float32)
        for m in range(M):
            xv[m, rng.permutation(K)[nnz:]] = 0.0
        x = torch.from_numpy(xv).to(DT[dt])
        wq = synth.qweights(N, K, bits, gs, dt, seed=bits)[0]
        sc = torch.ones((N, K // gs), dtype=DT[dt])
        bs = torch.zeros((N, K // gs), dtype=DT[dt])
        y = bi.qlinear(x.cuda(), wq.cuda(), sc.cuda(), bs.cuda(), bits, gs).cpu().double()
        want = x.double() @ torch.from_numpy(_fields(wq, bits)).double().t()
        assert torch.equal(y, want), (dt, bits)


@pytest.mark.parametrize("N", [4096, 14336])
def test_row_bits_independent_of_batch(bi, N):
    """C2's rule for the quantized layer: row 0's bits at every M from 1 to 512."""
    K, bits, gs = 4096, 4, 64
    x = synth.normal((512, K), 5, 1.0, "bf16", device="cuda")
    wq, sc, bs = (t.cuda() for t in synth.qweights(N, K, bits, gs, "bf16", seed=N))
    ref = bi.qlinear(x[:1], wq, sc, bs, bits, gs)
    full = bi.qlinear(x, wq, sc, bs, bits, gs)
    for M in (2, 3, 4, 8, 16, 32, 63, 64, 65, 128, 256, 512):
        y = bi.qlinear(x[:M], wq, sc, bs, bits, gs)
        assert_same_bits(y[:1], ref, "N=%d M=%d row 0" % (N, M))
        assert_same_bits(y, full[:M], "N=%d M=%d all rows vs M=512" % (N, M))
    # neighbours changed: row 0 keeps its bits
    x2 = x.clone()
    x2[1:] = torch.randn_like(x2[1:])
    assert_same_bits(bi.qlinear(x2[:64], wq, sc, bs, bits, gs)[:1], ref, "other neighbours")
    _no_device_error(bi)


def test_full_size_decode_sampled(bi):
    """Decode shape (N = 14336, K = 4096, 4-bit, group 64) against the oracle on sampled rows."""
    N, K, bits, gs = 14336, 4096, 4, 64
    x = synth.normal((16, K), 8, 1.0, "bf16")
    wq, sc, bs = synth.qweights(N, K, bits, gs, "bf16", seed=9)
    y = bi.qlinear(x.cuda(), wq.cuda(), sc.cuda(), bs.cuda(), bits, gs).cpu()
    rows = torch.arange(0, N, 97)
    ref, nrm = oracle.qlinear(x, wq[rows], sc[rows], bs[rows], bits, gs)
    check_close(y[:, rows], ref, nrm, torch.bfloat16, "decode qlinear sampled columns")


def test_graph_capture_same_bits(bi):
    M, N, K, bits, gs = 24, 512, 1024, 4, 64
    x = synth.normal((M, K), 1, 1.0, "bf16", device="cuda")
    wq, sc, bs = (t.cuda() for t in synth.qweights(N, K, bits, gs, "bf16", seed=2))
    eager = bi.qlinear(x, wq, sc, bs, bits, gs)
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        bi.qlinear(x, wq, sc, bs, bits, gs, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bi.qlinear(x, wq, sc, bs, bits, gs, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_same_bits(eager, out, "graph vs eager qlinear")
