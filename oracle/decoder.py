"""fp64 reference of the random-init decoder, composed from the oracle's ops.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Each op is the fp64
definition from oracle.c; between ops the activations are rounded to bf16 at
the same points where the decoder stores bf16 tensors, so the comparison
measures the kernels' arithmetic, not the storage format.  The final logits
are left in fp64.  Architecture readings: pre-norm blocks, RMSNorm, rotate-half
RoPE, GQA attention with fused QKV ([q | k | v] heads), SwiGLU with fused
[gate | up], untied LM head, no biases.
"""
from __future__ import annotations

import numpy as np
import torch

from . import default


def _bf16(a: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 (ties to even), returned as float64."""
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


def logits(weights: dict, ids, d, H, Hkv, D, inter, eps=1e-6, rope_base=10000.0):
    """weights: host tensors emb, lnf, lm_head and layers[i] = {ln1, wqkv, wo, ln2, wgu, wdown}.
    ids: the token ids of ONE request at positions 0..L-1.  Returns logits[L, vocab] (fp64)."""
    O = default()
    f = lambda t: t.detach().to("cpu").double().numpy()
    ids = np.asarray(ids.cpu() if hasattr(ids, "cpu") else ids, dtype=np.int64)
    L = ids.shape[0]
    pos = np.arange(L)
    h = f(weights["emb"])[ids]
    for lw in weights["layers"]:
        n = _bf16(O.rmsnorm(h, f(lw["ln1"]), eps))
        qkv = _bf16(O.linear(n, f(lw["wqkv"]))[0]).reshape(L, H + 2 * Hkv, D)
        q = _bf16(O.rope(qkv[:, :H].copy(), pos, rope_base))
        k = _bf16(O.rope(qkv[:, H:H + Hkv].copy(), pos, rope_base))
        v = qkv[:, H + Hkv:]
        att = O.sdpa(q.transpose(1, 0, 2)[None], k.transpose(1, 0, 2)[None],
                     np.ascontiguousarray(v.transpose(1, 0, 2))[None], causal=True, q_offset=0)[0]
        att = _bf16(att[0].transpose(1, 0, 2).reshape(L, H * D))
        h = _bf16(h + _bf16(O.linear(att, f(lw["wo"]))[0]))
        n = _bf16(O.rmsnorm(h, f(lw["ln2"]), eps))
        a = _bf16(O.swiglu(_bf16(O.linear(n, f(lw["wgu"]))[0])))
        h = _bf16(h + _bf16(O.linear(a, f(lw["wdown"]))[0]))
    n = _bf16(O.rmsnorm(h, f(weights["lnf"]), eps))
    return O.linear(n, f(weights["lm_head"]))[0]
