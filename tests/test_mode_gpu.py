"""batch_invariant_mode on the GPU: the patched torch ops run the library's kernels and give
the same bits as the direct calls."""
import pytest
import torch
import torch.nn.functional as F

from attention_bi_matmul_gb300 import synth
from tolerances import assert_same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    import __graft_entry__
    __graft_entry__.build()
    import attention_bi_matmul_gb300 as m
    torch.cuda.set_device(0)
    return m


def test_gemm_ops_route_to_the_library(bi):
    a, b, c = (t.cuda() for t in synth.gemm16(24, 512, 256, "bf16", seed=1, with_c=True))
    w = b.t().contiguous()                       # [N, K]
    bias = c[0].contiguous()
    n0 = bi.launch_count()
    with bi.batch_invariant_mode():
        y_mm = torch.matmul(a, b)
        y_at = a @ b
        y_lin = F.linear(a, w, bias)
        y_wt = a @ w.t()                          # the nn.Linear layout, transposed view
        y_add = torch.addmm(c, a, b, beta=0.5, alpha=2.0)
    assert bi.launch_count() - n0 == 5
    assert_same_bits(y_mm, bi.matmul(a, b), "torch.matmul")
    assert_same_bits(y_at, bi.matmul(a, b), "@")
    assert_same_bits(y_lin, bi.linear(a, w, bias), "F.linear")
    assert_same_bits(y_wt, bi.linear(a, w), "a @ w.t()")
    assert_same_bits(y_add, bi.addmm(c, a, b, alpha=2.0, beta=0.5), "torch.addmm")


def test_sdpa_routes_causal_and_boolean_masks(bi):
    q, k, v = (t.cuda() for t in synth.sdpa_qkv(2, 8, 2, 64, 64, 128, "bf16", seed=2))
    m = synth.bernoulli_mask((64, 64), 0.5, seed=3).cuda()
    m[:, 0] = True
    with bi.batch_invariant_mode():
        o_c = F.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
        o_m = F.scaled_dot_product_attention(q, k, v, attn_mask=m, enable_gqa=True)
        with pytest.raises(NotImplementedError):
            F.scaled_dot_product_attention(q, k, v, attn_mask=m.to(q.dtype), enable_gqa=True)
        with pytest.raises(NotImplementedError):
            F.scaled_dot_product_attention(q.float(), k.float(), v.float(), is_causal=True,
                                           enable_gqa=True)
    assert_same_bits(o_c, bi.sdpa(q, k, v, causal=True, q_offset=0), "is_causal")
    assert_same_bits(o_m, bi.sdpa(q, k, v, mask=m), "boolean attn_mask")
    ref = F.scaled_dot_product_attention(q.float(), k.float().repeat_interleave(4, 1),
                                         v.float().repeat_interleave(4, 1), attn_mask=m)
    assert (o_m.float() - ref).abs().max().item() < 3e-2


def test_unaligned_gemm_is_refused_in_strict_mode(bi):
    a = torch.randn(4, 100, device="cuda", dtype=torch.bfloat16)[:, :99]   # K = 99: no TMA rows
    b = torch.randn(99, 64, device="cuda", dtype=torch.bfloat16)
    with bi.batch_invariant_mode():
        with pytest.raises(NotImplementedError):
            torch.matmul(a, b)
    with bi.batch_invariant_mode(strict=False):
        y = torch.matmul(a, b)
    assert y.shape == (4, 64)
