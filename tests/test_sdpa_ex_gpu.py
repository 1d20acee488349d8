"""Attention with boolean array masks and attention sinks: parity with the fp64 oracle,
the degenerate rows, and invariance (GPU, through the C ABI's bi_sdpa_ex)."""
import math

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


def _sinks(H, seed, std=2.0):
    """Sink logits in the units of the scaled scores (those are ~N(0,1) here)."""
    return synth.normal((H,), seed, std, "f32")


def _window_mask(Lq, Lkv, q_offset, window):
    """Sliding window: query i (position q_offset+i) sees keys (pos-window, pos]."""
    pos = torch.arange(Lq).view(-1, 1) + q_offset
    j = torch.arange(Lkv).view(1, -1)
    return (j <= pos) & (j > pos - window)


# ------------------------------------------------------------------ parity

@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("G", [1, 4, 8, 16])
def test_sinks_parity_causal(bi, dt, G):
    Hkv = 2
    H = G * Hkv
    q, k, v = synth.sdpa_qkv(2, H, Hkv, 37, 301, 128, dt, seed=40 + G)
    sk = _sinks(H, 7 + G)
    sk[0] = 6.0          # a sink that dominates every key
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), causal=True, q_offset=250, sinks=sk.cuda())
    ref, nrm = oracle.sdpa_ex(q, k, v, causal=True, q_offset=250, sinks=sk)
    check_close(o, ref, nrm, DT[dt], "sdpa sinks G=%d" % G)
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), causal=False, q_offset=250, sinks=sk.cuda())
    ref, nrm = oracle.sdpa_ex(q, k, v, causal=False, q_offset=250, sinks=sk)
    check_close(o, ref, nrm, DT[dt], "sdpa sinks no mask G=%d" % G)
    _no_device_error(bi)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("Lq,Lkv,p", [(1, 1, 1.0), (3, 70, 0.5), (40, 300, 0.7), (130, 512, 0.3),
                                      (129, 1000, 0.9), (17, 257, 0.05)])
def test_array_mask_parity(bi, dt, Lq, Lkv, p):
    B, H, Hkv = 2, 8, 2
    q, k, v = synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, 128, dt, seed=Lq * 7 + Lkv)
    m = synth.bernoulli_mask((B, H, Lq, Lkv), p, seed=Lq + 3 * Lkv)
    m[..., Lkv // 2] = True              # at least one visible key in every row
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), mask=m.cuda())
    ref, nrm = oracle.sdpa_ex(q, k, v, mask=m)
    check_close(o, ref, nrm, DT[dt], "sdpa array mask Lq=%d Lkv=%d p=%g" % (Lq, Lkv, p))
    sk = _sinks(H, Lq)
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), mask=m.cuda(), sinks=sk.cuda())
    ref, nrm = oracle.sdpa_ex(q, k, v, mask=m, sinks=sk)
    check_close(o, ref, nrm, DT[dt], "sdpa array mask + sinks Lq=%d Lkv=%d" % (Lq, Lkv))
    _no_device_error(bi)


@pytest.mark.parametrize("shape", ["LqLkv", "B1LqLkv", "1H1Lkv"])
def test_broadcast_masks(bi, shape):
    """Masks with stride-0 dimensions: [Lq,Lkv], [B,1,Lq,Lkv], [1,H,1,Lkv]."""
    B, H, Hkv, Lq, Lkv = 2, 8, 4, 50, 384
    q, k, v = synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, 128, "bf16", seed=5)
    dims = {"LqLkv": (Lq, Lkv), "B1LqLkv": (B, 1, Lq, Lkv), "1H1Lkv": (1, H, 1, Lkv)}[shape]
    m = synth.bernoulli_mask(dims, 0.6, seed=9)
    m[..., 0] = True
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), mask=m.cuda())
    ref, nrm = oracle.sdpa_ex(q, k, v, mask=m.expand(B, H, Lq, Lkv))
    check_close(o, ref, nrm, torch.bfloat16, "sdpa broadcast mask %s" % shape)


def test_sliding_window_parity(bi):
    B, H, Hkv, Lq, Lkv = 1, 16, 2, 200, 1500
    q, k, v = synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, 128, "bf16", seed=11)
    m = _window_mask(Lq, Lkv, Lkv - Lq, 256)
    sk = _sinks(H, 12)
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), mask=m.cuda(), sinks=sk.cuda())
    ref, nrm = oracle.sdpa_ex(q, k, v, mask=m, sinks=sk)
    check_close(o, ref, nrm, torch.bfloat16, "sdpa sliding window + sinks")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("with_sinks", [False, True])
def test_late_rescales_parity_and_repeat(bi, causal, with_sinks):
    """Keys whose scores grow along the sequence, so that a row's shift moves up again
    and again in late chunks and O is rescaled between P V steps near the end of the
    call -- the case where a wait for the last P V could pass before an earlier one
    finished.  Parity with the oracle, and two calls bit for bit equal."""
    B, H, Hkv, Lq, Lkv = 2, 8, 2, 300, 1000
    q, k, v = synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, 128, "bf16", seed=77)
    grow = 1.0 + 8.0 * torch.arange(Lkv, dtype=torch.float32).view(1, 1, Lkv, 1) / Lkv
    k = (k.float() * grow).to(torch.bfloat16)
    sk = _sinks(H, 5) if with_sinks else None
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    skc = sk.cuda() if with_sinks else None
    o1 = bi.sdpa(qc, kc, vc, causal=causal, sinks=skc)
    o2 = bi.sdpa(qc, kc, vc, causal=causal, sinks=skc)
    assert_same_bits(o1, o2, "late rescales, two calls")
    ref, nrm = oracle.sdpa_ex(q, k, v, causal=causal, sinks=sk)
    check_close(o1, ref, nrm, torch.bfloat16, "late rescales causal=%s sinks=%s" % (causal, with_sinks))
    _no_device_error(bi)


# ------------------------------------------------------------------ degenerate rows

def test_fully_masked_rows(bi):
    """No visible key: NaN without a sink (as the oracle); exactly 0 with one (p_sink = 1)."""
    B, H, Hkv, Lq, Lkv = 1, 4, 2, 6, 200
    q, k, v = synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, 128, "bf16", seed=2)
    m = synth.bernoulli_mask((B, H, Lq, Lkv), 0.5, seed=3)
    m[0, 1, 2, :] = False
    m[0, 3, 5, :] = False
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), mask=m.cuda()).cpu()
    assert torch.isnan(o[0, 1, 2]).all() and torch.isnan(o[0, 3, 5]).all()
    ref, nrm = oracle.sdpa_ex(q, k, v, mask=m)
    keep = ~torch.isnan(torch.from_numpy(ref))
    assert torch.isnan(torch.from_numpy(ref)).sum() == 2 * 128
    check_close(torch.where(keep, o.float(), 0.0), np.where(keep.numpy(), ref, 0.0),
                np.where(keep.numpy(), nrm, 0.0), torch.bfloat16, "masked rows, others")
    sk = _sinks(H, 4)
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), mask=m.cuda(), sinks=sk.cuda()).cpu()
    assert (o[0, 1, 2] == 0).all() and (o[0, 3, 5] == 0).all()
    ref, nrm = oracle.sdpa_ex(q, k, v, mask=m, sinks=sk)
    check_close(o, ref, nrm, torch.bfloat16, "masked rows with sinks")
    _no_device_error(bi)


def test_single_visible_key_is_exact(bi):
    """One visible key and no sink: p = 1 and the output is that key's value exactly."""
    B, H, Hkv, Lq, Lkv = 1, 4, 1, 3, 700
    q, k, v = synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, 128, "bf16", seed=8)
    m = torch.zeros((B, H, Lq, Lkv), dtype=torch.bool)
    keys = [0, 129, 699]
    for i, j in enumerate(keys):
        m[0, :, i, j] = True
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), mask=m.cuda()).cpu()
    for i, j in enumerate(keys):
        for h in range(H):
            assert torch.equal(o[0, h, i], v[0, 0, j]), (i, j, h)


def test_dominant_sink_takes_the_mass(bi):
    """A sink far above every score takes all the mass: the output is ~e^-60 (not 0)."""
    B, H, Hkv, Lq, Lkv = 1, 2, 1, 4, 130
    q, k, v = synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, 128, "bf16", seed=13)
    sk = torch.full((H,), 60.0)
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), causal=False, sinks=sk.cuda()).cpu().float()
    ref, nrm = oracle.sdpa_ex(q, k, v, causal=False, sinks=sk)
    assert np.abs(ref).max() < 1e-20
    assert o.abs().max() < 1e-20


# ------------------------------------------------------------------ invariance

def test_causal_pattern_array_equals_causal_bits(bi):
    """An array mask holding the causal pattern gives the causal mode's bits; an all-True
    mask gives the unmasked mode's bits (fully masked chunks are exact no-ops)."""
    B, H, Hkv, Lq, Lkv, off = 2, 16, 2, 150, 700, 550
    q, k, v = (t.cuda() for t in synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, 128, "bf16", seed=21))
    causal = _window_mask(Lq, Lkv, off, Lkv + 1).cuda()
    a = bi.sdpa(q, k, v, causal=True, q_offset=off)
    b = bi.sdpa(q, k, v, mask=causal, q_offset=off)
    assert_same_bits(a, b, "causal vs causal-pattern array mask")
    a = bi.sdpa(q, k, v, causal=False)
    b = bi.sdpa(q, k, v, mask=torch.ones((Lq, Lkv), dtype=torch.bool, device="cuda"))
    assert_same_bits(a, b, "no mask vs all-True array mask")
    sk = _sinks(H, 22).cuda()
    a = bi.sdpa(q, k, v, causal=True, q_offset=off, sinks=sk)
    b = bi.sdpa(q, k, v, mask=causal, q_offset=off, sinks=sk)
    assert_same_bits(a, b, "causal vs causal-pattern array mask, with sinks")


@pytest.mark.parametrize("L0", [4095, 4096])
def test_window_mask_decode_equals_prefill_bits(bi, L0):
    """Sliding-window mask + sinks: a token's bits are the same whether it is computed in a
    64-token prefill or one token at a time against the growing cache."""
    B, H, Hkv, n, win = 1, 32, 8, 64, 1000
    Lkv = L0 + n
    q, k, v = (t.cuda() for t in synth.sdpa_qkv(B, H, Hkv, n, Lkv, 128, "bf16", seed=L0))
    sk = _sinks(H, 23).cuda()
    m = _window_mask(n, Lkv, L0, win).cuda()
    pre = bi.sdpa(q, k, v, q_offset=L0, mask=m, sinks=sk)
    for t in (0, 1, 31, 63):
        Lt = L0 + t + 1
        mt = _window_mask(1, Lt, L0 + t, win).cuda()
        one = bi.sdpa(q[:, :, t:t + 1], k[:, :, :Lt], v[:, :, :Lt], q_offset=L0 + t, mask=mt,
                      sinks=sk)
        assert_same_bits(pre[:, :, t:t + 1], one, "window decode t=%d" % t)


def test_batch_invariance_with_mask_and_sinks(bi):
    H, Hkv, Lq, Lkv = 8, 2, 33, 600
    q, k, v = (t.cuda() for t in synth.sdpa_qkv(4, H, Hkv, Lq, Lkv, 128, "fp16", seed=31))
    m = synth.bernoulli_mask((4, H, Lq, Lkv), 0.7, seed=32).cuda()
    sk = _sinks(H, 33).cuda()
    full = bi.sdpa(q, k, v, mask=m, sinks=sk)
    one = bi.sdpa(q[2:3], k[2:3], v[2:3], mask=m[2:3], sinks=sk)
    assert_same_bits(full[2:3], one, "B=4 vs B=1 with array mask + sinks")


def test_graph_capture_same_bits(bi):
    H, Hkv, Lq, Lkv = 8, 2, 16, 1000
    q, k, v = (t.cuda() for t in synth.sdpa_qkv(2, H, Hkv, Lq, Lkv, 128, "bf16", seed=41))
    m = synth.bernoulli_mask((2, H, Lq, Lkv), 0.5, seed=42).cuda()
    sk = _sinks(H, 43).cuda()
    eager = bi.sdpa(q, k, v, mask=m, sinks=sk)
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        bi.sdpa(q, k, v, mask=m, sinks=sk, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bi.sdpa(q, k, v, mask=m, sinks=sk, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_same_bits(eager, out, "graph vs eager, array mask + sinks")


def test_decode_with_window_and_sinks_medium(bi):
    """A decode batch at a longer context: B=4, H=32, Hkv=8, Lkv=8192, window 4096 + sinks."""
    B, H, Hkv, Lkv = 4, 32, 8, 8192
    q, k, v = synth.sdpa_qkv(B, H, Hkv, 1, Lkv, 128, "bf16", seed=51)
    m = _window_mask(1, Lkv, Lkv - 1, 4096)
    sk = _sinks(H, 52)
    o = bi.sdpa(q.cuda(), k.cuda(), v.cuda(), mask=m.cuda(), sinks=sk.cuda())
    ref, nrm = oracle.sdpa_ex(q, k, v, mask=m, sinks=sk)
    check_close(o, ref, nrm, torch.bfloat16, "decode window + sinks")
    assert math.isfinite(float(o.float().abs().max()))
