"""Batch-invariant GEMM and causal GQA attention for GB300 (sm_103a).

The kernels live in ``libbi.so`` (C ABI, include/bi.h); this package is its
Python binding:

    import attention_bi_matmul_gb300 as bi
    y = bi.linear(x, w, bias)                 # w is [N, K], the nn.Linear layout
    y = bi.matmul(a, b)                       # b is [K, N]
    y = bi.addmm(c, a, b, alpha=1.0, beta=1.0)
    o = bi.sdpa(q, k, v, causal=True)         # q[B,H,Lq,D], k/v[B,Hkv,Lkv,D]
    with bi.batch_invariant_mode():           # reroute torch ops to the kernels
        logits = model(tokens)

The bits of one output row do not depend on batch size, batch neighbours,
query length, KV-cache length, or eager vs CUDA-graph execution.
"""
from .api import (add, addmm, bmm, copy4d, debug_wait_probe, embedding, gemm_config,  # noqa: F401
                  last_device_error, launch_count, linear, matmul, qlinear, rmsnorm, rope, sdpa,
                  swiglu, version)
from ._lib import BiError  # noqa: F401
from .mode import batch_invariant_mode  # noqa: F401

scaled_dot_product_attention = sdpa
