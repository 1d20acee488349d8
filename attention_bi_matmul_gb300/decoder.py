"""A random-initialised Llama-style decoder whose every op runs in the library's kernels.

Used to check the end-to-end property the "mlx-batch-invariant" README opens
with: request 0's logits are bit-identical whether it runs alone or batched
with other requests, and whether the forward runs eagerly or is replayed from
a CUDA graph.  Architecture (readings where nothing is specified): pre-norm
blocks, RMSNorm (eps 1e-6, weight 1), rotate-half RoPE (base 10000), GQA
attention with a fused QKV projection, SwiGLU MLP ([gate | up] fused), no
biases, untied LM head, bf16 weights ~ N(0, 0.02).

Every step -- embedding gather, RMSNorm, the QKV/O/MLP/LM-head GEMMs, RoPE,
KV-cache writes, causal GQA attention, SwiGLU and residual adds -- is a call
into libbi.so; torch only allocates memory and provides the stream.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import api as bi
from . import synth


@dataclass(frozen=True)
class DecoderConfig:
    d: int = 2048
    n_layers: int = 4
    H: int = 16
    Hkv: int = 4
    D: int = 128
    inter: int = 5632
    vocab: int = 32000
    eps: float = 1e-6
    rope_base: float = 10000.0
    std: float = 0.02


class Decoder:
    def __init__(self, cfg: DecoderConfig = DecoderConfig(), seed: int = 0, device="cuda",
                 dtype=torch.bfloat16):
        self.cfg = cfg
        self.device = torch.device(device)
        self.dtype = dtype
        c = cfg
        nq = (c.H + 2 * c.Hkv) * c.D

        def w(shape, s):
            return synth.normal(shape, seed * 1000 + s, c.std, dtype, self.device)

        ones = lambda: torch.ones((c.d,), dtype=dtype, device=self.device)
        self.emb = w((c.vocab, c.d), 1)
        self.layers = []
        for i in range(c.n_layers):
            b = 10 * (i + 1)
            self.layers.append(dict(
                ln1=ones(), wqkv=w((nq, c.d), b + 1), wo=w((c.d, c.H * c.D), b + 2),
                ln2=ones(), wgu=w((2 * c.inter, c.d), b + 3), wdown=w((c.d, c.inter), b + 4)))
        self.lnf = ones()
        self.lm_head = w((c.vocab, c.d), 2)

    def new_cache(self, B: int, max_len: int):
        c = self.cfg
        shape = (B, c.Hkv, max_len, c.D)
        return [(torch.zeros(shape, dtype=self.dtype, device=self.device),
                 torch.zeros(shape, dtype=self.dtype, device=self.device))
                for _ in range(c.n_layers)]

    def forward(self, ids: torch.Tensor, cache, pos0: int, trace: dict | None = None) -> torch.Tensor:
        """ids[B, L] at absolute positions pos0 .. pos0+L-1 -> logits[B, L, vocab].

        Writes the new keys/values into ``cache`` at those positions.  With ``trace``
        (a dict), every intermediate tensor is also stored there under "<layer>.<name>"
        (layer "f" for the final norm and LM head), so that each op can be checked on
        its own inputs; nothing else changes."""
        c = self.cfg
        B, L = ids.shape
        T = B * L
        h = bi.embedding(ids.reshape(-1).contiguous(), self.emb)            # [T, d]
        for i, (lw, (kc, vc)) in enumerate(zip(self.layers, cache)):
            n = bi.rmsnorm(h, lw["ln1"], c.eps)
            qkv = bi.linear(n, lw["wqkv"]).view(B, L, c.H + 2 * c.Hkv, c.D)
            q = bi.rope(qkv[:, :, :c.H], pos0, c.rope_base)                 # [B, L, H, D]
            bi.rope(qkv[:, :, c.H:c.H + c.Hkv], pos0, c.rope_base,
                    out=kc[:, :, pos0:pos0 + L].transpose(1, 2))
            bi.copy4d(qkv[:, :, c.H + c.Hkv:], vc[:, :, pos0:pos0 + L].transpose(1, 2))
            att = torch.empty((B, L, c.H, c.D), dtype=self.dtype, device=self.device)
            bi.sdpa(q.transpose(1, 2), kc[:, :, :pos0 + L], vc[:, :, :pos0 + L], causal=True,
                    q_offset=pos0, out=att.transpose(1, 2))
            o = bi.linear(att.view(T, c.H * c.D), lw["wo"])
            h1 = bi.add(h, o)
            n2 = bi.rmsnorm(h1, lw["ln2"], c.eps)
            gu = bi.linear(n2, lw["wgu"])
            a = bi.swiglu(gu)
            down = bi.linear(a, lw["wdown"])
            h2 = bi.add(h1, down)
            if trace is not None:
                for name, t in (("h_in", h), ("n1", n), ("qkv", qkv), ("q", q),
                                ("k_cache", kc[:, :, :pos0 + L]), ("v_cache", vc[:, :, :pos0 + L]),
                                ("att", att), ("o", o), ("h1", h1), ("n2", n2), ("gu", gu),
                                ("a", a), ("down", down), ("h_out", h2)):
                    trace["%d.%s" % (i, name)] = t.clone()
            h = h2
        n = bi.rmsnorm(h, self.lnf, c.eps)
        logits = bi.linear(n, self.lm_head).view(B, L, c.vocab)
        if trace is not None:
            trace.update({"f.h_in": h, "f.n": n, "f.logits": logits})
        return logits

    __call__ = forward
