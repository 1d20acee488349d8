"""batch_invariant_mode on the host: strict refusal, fallback, and restoring torch's ops."""
import pytest
import torch
import torch.nn.functional as F

from attention_bi_matmul_gb300.mode import batch_invariant_mode


def _ops():
    return (torch.matmul, torch.Tensor.__matmul__, torch.addmm, F.linear,
            F.scaled_dot_product_attention)


def test_strict_refuses_what_has_no_kernel():
    a, b = torch.randn(3, 8), torch.randn(8, 5)
    before = _ops()
    with batch_invariant_mode():
        with pytest.raises(NotImplementedError):
            torch.matmul(a, b)                       # host tensors: no kernel
        with pytest.raises(NotImplementedError):
            a @ b
        with pytest.raises(NotImplementedError):
            F.linear(a, b.t().contiguous())
        with pytest.raises(NotImplementedError):
            torch.addmm(torch.zeros(5), a, b)
        q = torch.randn(1, 2, 4, 16)
        with pytest.raises(NotImplementedError):
            F.scaled_dot_product_attention(q, q, q, is_causal=True)
    assert _ops() == before


def test_non_strict_falls_back_to_torch():
    a, b = torch.randn(3, 8), torch.randn(8, 5)
    with batch_invariant_mode(strict=False):
        y = torch.matmul(a, b)
        z = F.linear(a, b.t().contiguous())
    assert torch.equal(y, a.matmul(b))
    assert torch.allclose(z, y, rtol=1e-5, atol=1e-6)


def test_ops_restored_after_an_exception():
    before = _ops()
    with pytest.raises(RuntimeError):
        with batch_invariant_mode():
            raise RuntimeError("boom")
    assert _ops() == before
