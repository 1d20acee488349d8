"""Attention at head dims 64, 96, 160, 192 and 256 (the kernel's 64-, 128- and 256-column
forms; 96 and 160-224 are loaded with zero fill past the head dim; the 256-column form
keeps the output in tensor memory and visits keys in chunks of 64): parity with the fp64
oracle and invariance."""
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


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [64, 96, 160, 192, 256])
@pytest.mark.parametrize("G", [1, 4, 16])
def test_parity_head_dims(bi, dt, D, G):
    Hkv = 2
    q, k, v = synth.sdpa_qkv(2, G * Hkv, Hkv, 45, 333, D, dt, seed=D + G)
    for causal in (True, False):
        o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), causal=causal, q_offset=270)
        ref, nrm = oracle.sdpa(q, k, v, causal=causal, q_offset=270)
        check_close(o, ref, nrm, DT[dt], "sdpa D=%d G=%d causal=%s" % (D, G, causal))
    _no_device_error(bi)


@pytest.mark.parametrize("D", [64, 96, 192, 256])
@pytest.mark.parametrize("Lq,Lkv,off", [(1, 1, 0), (1, 4097, 4096), (130, 130, 0), (7, 900, 500),
                                        (65, 65, 0), (1, 63, 62)])
def test_parity_shapes_head_dims(bi, D, Lq, Lkv, off):
    q, k, v = synth.sdpa_qkv(1, 8, 2, Lq, Lkv, D, "bf16", seed=Lq + Lkv + D)
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), causal=True, q_offset=off)
    ref, nrm = oracle.sdpa(q, k, v, causal=True, q_offset=off)
    check_close(o, ref, nrm, torch.bfloat16, "sdpa D=%d Lq=%d Lkv=%d" % (D, Lq, Lkv))


@pytest.mark.parametrize("D", [64, 96, 160, 256])
def test_mask_and_sinks_head_dims(bi, D):
    B, H, Hkv, Lq, Lkv = 2, 8, 2, 40, 700
    q, k, v = synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, D, "bf16", seed=3 * D)
    m = synth.bernoulli_mask((B, H, Lq, Lkv), 0.5, seed=D)
    m[..., 7] = True
    sk = synth.normal((H,), D + 1, 2.0, "f32")
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), mask=m.cuda(), sinks=sk.cuda())
    ref, nrm = oracle.sdpa_ex(q, k, v, mask=m, sinks=sk)
    check_close(o, ref, nrm, torch.bfloat16, "sdpa D=%d mask + sinks" % D)


@pytest.mark.parametrize("D", [64, 96, 160, 256])
def test_single_visible_key_is_exact_head_dims(bi, D):
    q, k, v = synth.sdpa_qkv(1, 4, 1, 1, 50, D, "bf16", seed=D)
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), causal=True, q_offset=0)
    for h in range(4):
        assert torch.equal(o[0, h, 0].cpu(), v[0, 0, 0]), "head %d" % h


@pytest.mark.parametrize("D", [64, 96, 160, 224, 256])
def test_columns_past_the_head_dim_untouched(bi, D):
    """The output is written for d < D only: a wider buffer keeps its other columns."""
    B, H, Hkv, Lq, Lkv = 1, 4, 2, 20, 300
    q, k, v = (t.cuda() for t in synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, D, "bf16", seed=9))
    wide = torch.full((B, H, Lq, D + 64), 7.0, dtype=torch.bfloat16, device="cuda")
    bi.sdpa(q, k, v, causal=True, out=wide[..., :D])
    assert (wide[..., D:] == 7.0).all()
    assert_same_bits(wide[..., :D], bi.sdpa(q, k, v, causal=True), "strided out D=%d" % D)


@pytest.mark.parametrize("D", [64, 96, 256])
@pytest.mark.parametrize("L0", [4095, 4097])
def test_decode_equals_prefill_bits_head_dims(bi, D, L0):
    """C3's rule at the other head dims: a token's bits are the same in a 64-token prefill,
    as a single-token decode, and with keys appended past it."""
    B, H, Hkv, n = 2, 32, 8, 64
    Lkv = L0 + n
    q, k, v = (t.cuda() for t in synth.sdpa_qkv(B, H, Hkv, n, Lkv + 130, D, "bf16", seed=L0))
    pre = bi.sdpa(q, k[:, :, :Lkv], v[:, :, :Lkv], causal=True, q_offset=L0)
    for t in (0, 9, 63):
        Lt = L0 + t + 1
        one = bi.sdpa(q[:, :, t:t + 1], k[:, :, :Lt], v[:, :, :Lt], causal=True, q_offset=L0 + t)
        assert_same_bits(pre[:, :, t:t + 1], one, "D=%d decode t=%d" % (D, t))
        more = bi.sdpa(q[:, :, t:t + 1], k, v, causal=True, q_offset=L0 + t)
        assert_same_bits(pre[:, :, t:t + 1], more, "D=%d appended keys t=%d" % (D, t))
    one_b = bi.sdpa(q[1:2], k[1:2, :, :Lkv], v[1:2, :, :Lkv], causal=True, q_offset=L0)
    assert_same_bits(pre[1:2], one_b, "D=%d B=2 vs B=1" % D)


def test_d256_graph_capture_and_long_decode(bi):
    """256-column kernel: graph replay gives the eager bits; a longer decode (8192 keys,
    sliding window + sinks) matches the oracle."""
    B, H, Hkv, Lkv, D = 2, 8, 2, 8192, 256
    q, k, v = synth.sdpa_qkv(B, H, Hkv, 1, Lkv, D, "bf16", seed=77)
    pos = torch.arange(Lkv)
    m = ((pos <= Lkv - 1) & (pos > Lkv - 1 - 3000)).view(1, Lkv)
    sk = synth.normal((H,), 78, 2.0, "f32")
    qc, kc, vc, mc, skc = q.cuda(), k.cuda(), v.cuda(), m.cuda(), sk.cuda()
    eager = bi.sdpa(qc, kc, vc, mask=mc, sinks=skc)
    ref, nrm = oracle.sdpa_ex(q, k, v, mask=m, sinks=sk)
    check_close(eager, ref, nrm, torch.bfloat16, "D=256 decode window + sinks")
    out = torch.empty_like(eager)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        bi.sdpa(qc, kc, vc, mask=mc, sinks=skc, out=out)
    torch.cuda.current_stream().wait_stream(st)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bi.sdpa(qc, kc, vc, mask=mc, sinks=skc, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_same_bits(eager, out, "D=256 graph vs eager")
    _no_device_error(bi)
