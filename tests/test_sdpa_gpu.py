"""Causal GQA attention: parity with the fp64 oracle and invariance across query length,
context length, appended masked keys, batch, and graph capture (GPU, through the C ABI)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from attention_bi_matmul_gb300 import synth
from tolerances import assert_same_bits, check_close, count_bit_diffs

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
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_parity_group_sizes(bi, dt, G):
    Hkv = 2
    q, k, v = synth.sdpa_qkv(2, G * Hkv, Hkv, 37, 301, 128, dt, seed=G)
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), causal=True, q_offset=250)
    ref, nrm = oracle.sdpa(q, k, v, causal=True, q_offset=250)
    check_close(o, ref, nrm, DT[dt], "sdpa G=%d" % G)
    _no_device_error(bi)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("Lq,Lkv,q_offset", [(1, 1, 0), (1, 129, 128), (3, 3, 0), (40, 300, 100),
                                             (130, 130, 0), (200, 520, 320), (5, 1000, 7)])
def test_parity_shapes(bi, dt, Lq, Lkv, q_offset):
    q, k, v = synth.sdpa_qkv(2, 8, 2, Lq, Lkv, 128, dt, seed=Lq + Lkv)
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), causal=True, q_offset=q_offset)
    ref, nrm = oracle.sdpa(q, k, v, causal=True, q_offset=q_offset)
    check_close(o, ref, nrm, DT[dt], "sdpa Lq=%d Lkv=%d off=%d" % (Lq, Lkv, q_offset))
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), causal=False, q_offset=q_offset)
    ref, nrm = oracle.sdpa(q, k, v, causal=False)
    check_close(o, ref, nrm, DT[dt], "sdpa no mask Lq=%d Lkv=%d" % (Lq, Lkv))
    _no_device_error(bi)


def test_single_visible_key_is_exact(bi):
    """Query at position 0 sees only key 0: p = 1 and the output is v_0 exactly."""
    q, k, v = synth.sdpa_qkv(1, 4, 1, 1, 50, 128, "bf16", seed=3)
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), causal=True, q_offset=0)
    for h in range(4):
        assert torch.equal(o[0, h, 0].cpu(), v[0, 0, 0]), "head %d" % h


def test_strided_layouts(bi):
    """q/k/v/o as strided views ([B, L, H, D] storage), as a decoder produces them."""
    B, H, Hkv, Lq, Lkv = 2, 8, 2, 20, 150
    qs = synth.normal((B, Lq, H, 128), 1, 1.0, "bf16")
    ks = synth.normal((B, Lkv, Hkv, 128), 2, 1.0, "bf16")
    vs = synth.normal((B, Lkv, Hkv, 128), 3, 1.0, "bf16")
    q, k, v = (t.cuda().transpose(1, 2) for t in (qs, ks, vs))
    o = torch.empty((B, Lq, H, 128), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    bi.sdpa(q, k, v, causal=True, out=o)
    ref, nrm = oracle.sdpa(qs.transpose(1, 2), ks.transpose(1, 2), vs.transpose(1, 2))
    check_close(o, ref, nrm, torch.bfloat16, "strided sdpa")


# ------------------------------------------------------------------ the invariance config

C3_LQ = (1, 2, 4, 8, 9, 16, 32, 64, 128)
C3_L0 = (4095, 4096, 4097, 8192)


@pytest.mark.parametrize("L0", C3_L0)
def test_c3_token_bits_independent_of_query_length(bi, L0):
    """B=4, H=32, Hkv=8, D=128: a token's output is bit-identical whether it is decoded alone
    (Lq=1), sits anywhere in a prefill chunk of Lq in {1,..,128}, or has fully masked keys
    appended after it; and the same at B=1 as at B=4."""
    B, H, Hkv, D, EXTRA = 4, 32, 8, 128, 128
    Lmax = L0 + 128 + EXTRA
    q, k, v = synth.sdpa_qkv(B, H, Hkv, 128, Lmax, D, "bf16", seed=L0, device="cuda")
    # reference: each new token decoded alone with exactly its prefix
    dec = torch.empty((B, H, 128, D), dtype=torch.bfloat16, device="cuda")
    for i in range(128):
        pos = L0 + i
        dec[:, :, i:i + 1] = bi.sdpa(q[:, :, i:i + 1], k[:, :, :pos + 1], v[:, :, :pos + 1],
                                     causal=True, q_offset=pos)
    for Lq in C3_LQ:
        for start in range(0, 128, Lq):
            n = min(Lq, 128 - start)
            pos0 = L0 + start
            for extra in (0, 1, EXTRA):
                Lkv = pos0 + n + extra
                o = bi.sdpa(q[:, :, start:start + n], k[:, :, :Lkv], v[:, :, :Lkv], causal=True,
                            q_offset=pos0)
                assert_same_bits(o, dec[:, :, start:start + n],
                                 "L0=%d Lq=%d start=%d extra=%d" % (L0, Lq, start, extra))
            if Lq >= 64:
                break
    # batch of one vs batch of four
    o1 = bi.sdpa(q[1:2, :, :9], k[1:2, :, :L0 + 9], v[1:2, :, :L0 + 9], causal=True, q_offset=L0)
    assert_same_bits(o1, dec[1:2, :, :9], "B=1 vs B=4")
    # accuracy of sampled tokens against the oracle
    for (b, i) in ((0, 0), (3, 127), (2, 64)):
        pos = L0 + i
        ref, nrm = oracle.sdpa(q[b:b + 1, :, i:i + 1].cpu(), k[b:b + 1, :, :pos + 1].cpu(),
                               v[b:b + 1, :, :pos + 1].cpu(), causal=True, q_offset=pos)
        check_close(dec[b:b + 1, :, i:i + 1], ref, nrm, torch.bfloat16, "C3 sample")
    _no_device_error(bi)


def test_c3_torch_sdpa_control_differs(bi):
    """The negative control: torch's SDPA gives a token different bits in decode vs in a
    prefill chunk (the library's kernel does not)."""
    B, H, Hkv, D, L0 = 4, 32, 8, 128, 4096
    q, k, v = synth.sdpa_qkv(B, H, Hkv, 128, L0 + 128, D, "bf16", seed=5, device="cuda")
    kr = k.repeat_interleave(H // Hkv, 1)
    vr = v.repeat_interleave(H // Hkv, 1)
    diffs = 0
    for Lq in (2, 8, 9, 64, 128):
        mask = torch.ones(Lq, L0 + Lq, dtype=torch.bool, device="cuda").tril(L0)
        chunk = F.scaled_dot_product_attention(q[:, :, :Lq], kr[:, :, :L0 + Lq], vr[:, :, :L0 + Lq],
                                               attn_mask=mask)
        for i in (0, Lq - 1):
            one = F.scaled_dot_product_attention(q[:, :, i:i + 1], kr[:, :, :L0 + i + 1],
                                                 vr[:, :, :L0 + i + 1])
            diffs += count_bit_diffs(chunk[:, :, i:i + 1], one)
    print("torch SDPA control: %d differing bit patterns" % diffs)
    assert diffs > 0


def test_sdpa_graph_capture_same_bits(bi):
    q, k, v = synth.sdpa_qkv(2, 16, 4, 9, 700, 128, "bf16", seed=8, device="cuda")
    eager = bi.sdpa(q, k, v, causal=True)
    o = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        bi.sdpa(q, k, v, causal=True, out=o)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bi.sdpa(q, k, v, causal=True, out=o)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_same_bits(o, eager, "sdpa graph vs eager")


def test_decode_full_size_sampled(bi):
    """The decode workload B=32, H=32, Hkv=8, KV 32768 in the benchmark's launch shape;
    sampled (b, h) rows against the oracle."""
    B, H, Hkv, D, L = 32, 32, 8, 128, 32768
    q, k, v = synth.sdpa_qkv(B, H, Hkv, 1, L, D, "bf16", seed=0, device="cuda")
    o = bi.sdpa(q, k, v, causal=True)
    for b in (0, 17, 31):
        ref, nrm = oracle.sdpa(q[b:b + 1].cpu(), k[b:b + 1].cpu(), v[b:b + 1].cpu(), causal=True)
        check_close(o[b:b + 1], ref, nrm, torch.bfloat16, "decode b=%d" % b)
    _no_device_error(bi)


@pytest.mark.parametrize("B,H,Hkv,L,D", [(4, 32, 8, 4096, 128), (1, 16, 8, 8192, 256)])
def test_prefill_full_size_sampled(bi, B, H, Hkv, L, D):
    """Causal prefill at the sizes its throughput is quoted on, in one call: sampled query
    positions (first, chunk edges, a ragged middle, last) of two batch entries against the
    oracle, each position with every head."""
    q, k, v = synth.sdpa_qkv(B, H, Hkv, L, L, D, "bf16", seed=3, device="cuda")
    o = bi.sdpa(q, k, v, causal=True)
    torch.cuda.synchronize()
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    for b in sorted({0, B - 1}):
        for p in (0, 127, 128, 1000, L // 2 + 63, L - 1):
            ref, nrm = oracle.sdpa(qc[b:b + 1, :, p:p + 1], kc[b:b + 1, :, :p + 1], vc[b:b + 1, :, :p + 1],
                                   causal=True)
            check_close(o[b:b + 1, :, p:p + 1], ref, nrm, torch.bfloat16,
                        "prefill B%d L%d D%d b=%d row %d" % (B, L, D, b, p))
    _no_device_error(bi)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_growing_scores_move_the_shift(bi, dt):
    """Keys whose scale grows along the sequence, so a row's chunk maxima keep rising far
    past its shift (the shift must move many times, by more than 2^8 each): parity with
    the oracle, and a token's bits are the same alone (decode), inside a 256-row chunk
    and inside the whole prefill."""
    B, H, Hkv, L, D = 1, 8, 2, 1024, 128
    g = torch.Generator().manual_seed(41)
    q = torch.randn(B, H, L, D, generator=g)
    grow = (1.0 + torch.arange(L, dtype=torch.float32) / 32.0).view(1, 1, L, 1)
    k = torch.randn(B, Hkv, L, D, generator=g) * grow
    v = torch.randn(B, Hkv, L, D, generator=g)
    q, k, v = (t.to(DT[dt]) for t in (q, k, v))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = bi.sdpa(qd, kd, vd, causal=True)
    for p in (0, 1, 127, 128, 500, 1000, 1023):
        # row p sees keys 0..p: the oracle on that prefix with q_offset = p
        ref, nrm = oracle.sdpa(q[:, :, p:p + 1], k[:, :, :p + 1], v[:, :, :p + 1], causal=True)
        check_close(o[:, :, p:p + 1], ref, nrm, DT[dt], "growing scores, row %d" % p)
    for p in (700, 1023):
        one = bi.sdpa(qd[:, :, p:p + 1], kd[:, :, :p + 1], vd[:, :, :p + 1], causal=True)
        assert_same_bits(one, o[:, :, p:p + 1], "token %d alone vs in the prefill" % p)
        tile = bi.sdpa(qd[:, :, p - 255:p + 1], kd[:, :, :p + 1], vd[:, :, :p + 1], causal=True)
        assert_same_bits(tile[:, :, -1:], o[:, :, p:p + 1], "token %d in a 256-row chunk" % p)
    _no_device_error(bi)


def test_two_chunk_decode_many_ctas_repeated(bi):
    """Decode where every block sees exactly two key chunks (the last step of the key/value
    pipeline then carries only values), with 256 blocks in flight and the call repeated:
    every launch gives the same bits, and sampled rows match the oracle."""
    B, H, Hkv, Lkv, D = 32, 32, 8, 200, 128
    q, k, v = synth.sdpa_qkv(B, H, Hkv, 1, Lkv, D, "bf16", seed=51)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    first = bi.sdpa(qd, kd, vd, causal=True)
    for _ in range(20):
        assert_same_bits(bi.sdpa(qd, kd, vd, causal=True), first, "repeated two-chunk decode")
    for b in (0, 17, 31):
        ref, nrm = oracle.sdpa(q[b:b + 1], k[b:b + 1], v[b:b + 1], causal=True)
        check_close(first[b:b + 1], ref, nrm, torch.bfloat16, "two-chunk decode b=%d" % b)
    _no_device_error(bi)
