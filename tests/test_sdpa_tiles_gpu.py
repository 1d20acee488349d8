"""Query-length invariance of attention across head dims, group sizes, dtypes and every
mask form: the rows of a call spanning several query tiles (both ends ragged) against the
same rows computed one query tile per call, bit for bit; and a prefill's parity with the
oracle (GPU)."""
import pytest
import torch

import oracle
from attention_bi_matmul_gb300 import synth
from tolerances import assert_same_bits, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import attention_bi_matmul_gb300 as mod
    torch.cuda.set_device(0)
    return mod


def _no_device_error(bi):
    st, code = bi.last_device_error()
    assert st == 0 and code == 0, (st, code)


def _tilewise(bi, q, k, v, q_offset, G, causal, mask=None, sinks=None):
    """The same rows, each query tile (128 // G aligned positions) computed by its own
    one-tile call."""
    Qt = 128 // G
    Lq = q.shape[2]
    out = torch.empty_like(q)
    p = q_offset
    while p < q_offset + Lq:
        end = min((p // Qt + 1) * Qt, q_offset + Lq)
        i0, i1 = p - q_offset, end - q_offset
        kw = {}
        if mask is not None:
            kw["mask"] = mask[:, :, i0:i1]
        if sinks is not None:
            kw["sinks"] = sinks
        if mask is None:
            kw["causal"] = causal
        out[:, :, i0:i1] = bi.sdpa(q[:, :, i0:i1], k, v, q_offset=p, **kw)
        p = end
    return out


@pytest.mark.parametrize("D", [64, 96, 128])
@pytest.mark.parametrize("G", [1, 4, 16])
@pytest.mark.parametrize("causal", [True, False])
def test_rows_same_bits_as_one_tile_calls(bi, D, G, causal):
    B, Hkv = 2, 2
    Qt = 128 // G
    Lq = 3 * Qt + Qt // 2 + 1            # four query tiles, the last ragged
    q_offset = 5 * Qt - 3                # not tile-aligned: the first tile is ragged too
    Lkv = q_offset + Lq + 17
    q, k, v = synth.sdpa_qkv(B, G * Hkv, Hkv, Lq, Lkv, D, "bf16", seed=D * 31 + G, device="cuda")
    o = bi.sdpa(q, k, v, causal=causal, q_offset=q_offset)
    ref = _tilewise(bi, q, k, v, q_offset, G, causal)
    assert_same_bits(o, ref, "D=%d G=%d causal=%s: several tiles vs one per call" % (D, G, causal))
    _no_device_error(bi)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_mask_array_and_sinks_same_bits(bi, dt):
    B, H, Hkv, D, G = 2, 8, 2, 128, 4
    Qt = 128 // G
    Lq, q_offset = 5 * Qt, 40
    Lkv = q_offset + Lq + 9
    q, k, v = synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, D, dt, seed=77, device="cuda")
    m = synth.bernoulli_mask((B, H, Lq, Lkv), 0.6, seed=78).cuda()
    m[..., 0] = True
    sk = synth.normal((H,), 79, 2.0, "f32").cuda()
    o = bi.sdpa(q, k, v, mask=m, sinks=sk, q_offset=q_offset)
    ref = _tilewise(bi, q, k, v, q_offset, G, None, mask=m, sinks=sk)
    assert_same_bits(o, ref, "array mask + sinks: several tiles vs one per call")
    _no_device_error(bi)


def test_prefill_parity_and_repeat(bi):
    """A causal prefill of many query tiles: sampled rows against the oracle, and the
    same bits on a second call."""
    B, H, Hkv, L, D = 1, 8, 2, 600, 128
    q, k, v = synth.sdpa_qkv(B, H, Hkv, L, L, D, "bf16", seed=5, device="cuda")
    o = bi.sdpa(q, k, v, causal=True, q_offset=0)
    assert_same_bits(bi.sdpa(q, k, v, causal=True, q_offset=0), o, "second call")
    ref, nrm = oracle.sdpa(q.cpu(), k.cpu(), v.cpu(), causal=True, q_offset=0)
    rows = [0, 1, 31, 32, 300, 598, 599]
    check_close(o[:, :, rows], ref[:, :, rows], nrm[:, :, rows], torch.bfloat16, "prefill sampled")
    _no_device_error(bi)
