"""Stacked (batched) matmul: parity with the fp64 oracle per entry, and each entry's bits
equal to the unbatched call on that entry (GPU, through bi_matmul_batched)."""
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


def _operands(Bt, M, N, K, dt, seed):
    s = K ** -0.5
    a = synth.normal((Bt, M, K), seed, s, dt)
    b = synth.normal((Bt, K, N), seed + 1, s, dt)
    return a, b


@pytest.mark.parametrize("dt", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("Bt,M,N,K", [(3, 37, 200, 136), (2, 130, 256, 512), (4, 1, 64, 4096),
                                      (5, 16, 4096, 64)])
def test_parity_and_entry_bits_kn(bi, dt, Bt, M, N, K):
    a, b = _operands(Bt, M, N, K, dt, seed=M + N)
    y = bi.bmm(a.cuda(), b.cuda())
    for e in range(Bt):
        ref, nrm = oracle.matmul(a[e], b[e])
        check_close(y[e], ref, nrm, DT[dt], "bmm %s entry %d" % (dt, e))
        assert_same_bits(y[e], bi.matmul(a[e].cuda(), b[e].cuda()), "entry %d vs matmul" % e)


@pytest.mark.parametrize("dt", ["bf16", "fp16", "fp32"])
def test_parity_and_entry_bits_nk(bi, dt):
    """b given as w.transpose(-1, -2) with w[Bt, N, K] contiguous: each entry is linear(a, w)."""
    Bt, M, N, K = 3, 45, 320, 256
    a = synth.normal((Bt, M, K), 1, K ** -0.5, dt)
    w = synth.normal((Bt, N, K), 2, K ** -0.5, dt)
    y = bi.bmm(a.cuda(), w.cuda().transpose(-1, -2))
    for e in range(Bt):
        ref, nrm = oracle.linear(a[e], w[e])
        check_close(y[e], ref, nrm, DT[dt], "bmm nk %s entry %d" % (dt, e))
        assert_same_bits(y[e], bi.linear(a[e].cuda(), w[e].cuda()), "entry %d vs linear" % e)


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_entry_bits_independent_of_batch(bi, dt):
    a, b = (t.cuda() for t in _operands(6, 77, 384, 1024, dt, seed=5))
    full = bi.bmm(a, b)
    for n in (1, 2, 5):
        part = bi.bmm(a[:n], b[:n])
        assert_same_bits(full[:n], part, "batch %d vs 6" % n)
    # neighbours changed: entry 0 keeps its bits
    a2, b2 = a.clone(), b.clone()
    a2[1:] = torch.randn_like(a2[1:])
    b2[1:] = torch.randn_like(b2[1:])
    assert_same_bits(full[0], bi.bmm(a2, b2)[0], "entry 0 with other neighbours")


def test_broadcast_and_leading_dims(bi):
    M, N, K = 20, 192, 256
    a = synth.normal((2, 3, M, K), 7, K ** -0.5, "bf16").cuda()
    b1 = synth.normal((K, N), 8, K ** -0.5, "bf16").cuda()
    b3 = synth.normal((3, K, N), 9, K ** -0.5, "bf16").cuda()
    y = bi.bmm(a, b1.expand(2, 3, K, N))                  # b shared (stride 0)
    assert_same_bits(y, bi.matmul(a, b1), "shared b vs flattened matmul")
    y = bi.bmm(a, b3)                                     # b broadcast over the first dim
    for i in range(2):
        for j in range(3):
            assert_same_bits(y[i, j], bi.matmul(a[i, j], b3[j]), "entry (%d,%d)" % (i, j))
    a1 = a[0, 0]
    y = bi.bmm(a1, b3)                                    # a shared (stride 0)
    for j in range(3):
        assert_same_bits(y[j], bi.matmul(a1, b3[j]), "shared a entry %d" % j)


def test_attention_scores_pattern_in_strict_mode(bi):
    """q @ k.transpose(-1, -2) inside batch_invariant_mode runs the batched GEMM."""
    q = synth.normal((2, 4, 33, 128), 10, 1.0, "bf16").cuda()
    k = synth.normal((2, 4, 70, 128), 11, 1.0, "bf16").cuda()
    n0 = bi.launch_count()
    with bi.batch_invariant_mode():
        s = torch.matmul(q, k.transpose(-1, -2))
        s2 = q @ k.transpose(-1, -2)
    assert bi.launch_count() - n0 == 2
    assert_same_bits(s, s2, "matmul vs @")
    for i in range(2):
        for h in range(4):
            assert_same_bits(s[i, h], bi.linear(q[i, h], k[i, h]), "scores (%d,%d)" % (i, h))
    ref = torch.matmul(q.double(), k.double().transpose(-1, -2))
    assert (s.double() - ref).abs().max().item() < 0.25


def test_graph_capture_same_bits(bi):
    a, b = (t.cuda() for t in _operands(4, 50, 256, 512, "bf16", seed=12))
    eager = bi.bmm(a, b)
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        bi.bmm(a, b, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bi.bmm(a, b, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_same_bits(eager, out, "graph vs eager bmm")
