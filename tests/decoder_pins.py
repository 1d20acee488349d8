"""Pins of the oracle's decoder composition (``oracle/decoder.py``) on CPU.

``oracle/decoder.py`` composes the oracle's per-op functions into the
random-init decoder used by the end-to-end batch-invariance check (the
"mlx-batch-invariant" README opens with request 0's 32000 logits at batch 8
against batch 1).  The pages give only dimensions for that model; the readings
are: pre-norm blocks, RMSNorm, rotate-half RoPE on q and k only, GQA attention
with a fused [q | k | v] projection and a causal mask from position 0, SwiGLU
with a fused [gate | up] projection, residual adds, untied LM head, no biases,
bf16 storage between ops.

Each ``pin_*`` takes a decoder module (the oracle's, or a copy with a planted
mistake) and raises ``AssertionError`` when its ``logits`` disagree with:
  * an independent float64 forward written here from those readings with torch
    library routines (``F.rms_norm``, ``F.scaled_dot_product_attention`` with an
    explicit boolean mask, ``F.silu``, RoPE as a complex rotation), rounding to
    bf16 at the same storage points;
  * causality: the logits of a prefix are the first rows of the full logits;
  * a closed form: with every block's output projections zero, the blocks add
    nothing and the logits are the LM head of the normalised embeddings.
The model is tiny and its weights non-symmetric (random norm weights, distinct
per layer) so that a swapped slice, a dropped term or a wrong position fails.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

CFG = dict(d=64, H=4, Hkv=2, D=16, inter=96, vocab=97, eps=1e-6, rope_base=10000.0)
N_LAYERS = 2
L = 7


def _weights(seed: int = 5, zero_out: bool = False):
    """bf16 weights of a tiny decoder with random (non-unit) norm weights."""
    g = torch.Generator().manual_seed(seed)
    c = CFG
    nq = (c["H"] + 2 * c["Hkv"]) * c["D"]

    def w(shape, std):
        return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)

    def ln():
        return (1.0 + 0.3 * torch.randn((c["d"],), generator=g)).to(torch.bfloat16)

    layers = []
    for _ in range(N_LAYERS):
        lw = dict(ln1=ln(), wqkv=w((nq, c["d"]), 0.25), wo=w((c["d"], c["H"] * c["D"]), 0.2),
                  ln2=ln(), wgu=w((2 * c["inter"], c["d"]), 0.2),
                  wdown=w((c["d"], c["inter"]), 0.2))
        if zero_out:
            lw["wo"] = torch.zeros_like(lw["wo"])
            lw["wdown"] = torch.zeros_like(lw["wdown"])
        layers.append(lw)
    return {"emb": w((c["vocab"], c["d"]), 1.0), "lnf": ln(), "lm_head": w((c["vocab"], c["d"]), 0.2),
            "layers": layers}


def _ids(seed: int = 6, n: int = L):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, CFG["vocab"], (n,), generator=g, dtype=torch.int64)


def _call(mod, weights, ids):
    c = CFG
    return np.asarray(mod.logits(weights, ids, c["d"], c["H"], c["Hkv"], c["D"], c["inter"],
                                 c["eps"], c["rope_base"]), dtype=np.float64)


def independent_logits(weights, ids) -> np.ndarray:
    """The decoder forward in torch float64, written from the architecture readings."""
    c = CFG
    d, H, Hkv, D, inter = c["d"], c["H"], c["Hkv"], c["D"], c["inter"]
    f64 = lambda t: t.double()
    bf = lambda t: t.to(torch.bfloat16).double()      # a bf16 storage point
    n_tok = ids.shape[0]
    half = D // 2
    # RoPE (rotate-half pairing: element i pairs with i + D/2) as the rotation of the
    # complex number x_i + j x_{i+half} by the angle pos * base^(-2i/D)
    inv = c["rope_base"] ** (-2.0 * torch.arange(half, dtype=torch.float64) / D)
    ang = torch.arange(n_tok, dtype=torch.float64)[:, None] * inv[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]          # [T, 1, half]

    def rope(x):                                                      # [T, n, D]
        z = torch.complex(x[..., :half], x[..., half:]) * rot
        return torch.cat([z.real, z.imag], dim=-1)

    visible = torch.ones((n_tok, n_tok), dtype=torch.bool).tril()     # key j <= query i
    h = f64(weights["emb"])[ids]
    for lw in weights["layers"]:
        n = bf(F.rms_norm(h, (d,), f64(lw["ln1"]), c["eps"]))
        qkv = bf(n @ f64(lw["wqkv"]).T).view(n_tok, H + 2 * Hkv, D)
        q, k, v = torch.split(qkv, [H, Hkv, Hkv], dim=1)
        q, k = bf(rope(q)), bf(rope(k))
        rep = H // Hkv                                                # query head h -> kv head h // rep
        att = F.scaled_dot_product_attention(
            q.transpose(0, 1), k.transpose(0, 1).repeat_interleave(rep, 0),
            v.transpose(0, 1).repeat_interleave(rep, 0), attn_mask=visible)
        att = bf(att.transpose(0, 1).reshape(n_tok, H * D))
        h = bf(h + bf(att @ f64(lw["wo"]).T))
        n = bf(F.rms_norm(h, (d,), f64(lw["ln2"]), c["eps"]))
        gu = bf(n @ f64(lw["wgu"]).T)
        a = bf(F.silu(gu[:, :inter]) * gu[:, inter:])
        h = bf(h + bf(a @ f64(lw["wdown"]).T))
    n = bf(F.rms_norm(h, (d,), f64(weights["lnf"]), c["eps"]))
    return (n @ f64(weights["lm_head"]).T).numpy()


def _close(got, want, rel, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, "%s: shape %s vs %s" % (what, got.shape, want.shape)
    scale = float(np.abs(want).max())
    err = float(np.abs(got - want).max())
    assert np.isfinite(got).all() and err <= rel * scale, \
        "%s: max |err| %.3e against %.3e x max|ref| %.3e" % (what, err, rel, scale)


def pin_decoder_matches_independent_forward(mod):
    """All positions of a 2-layer decoder; both sides round to bf16 at the same points, so
    they agree to fp64 rounding unless a value lands on a bf16 rounding boundary (for
    these seeds none does)."""
    w = _weights()
    for seed in (6, 7):
        ids = _ids(seed)
        _close(_call(mod, w, ids), independent_logits(w, ids), 1e-9,
               "decoder logits vs independent float64 forward (ids seed %d)" % seed)


def pin_decoder_prefix_is_causal(mod):
    """Position t sees tokens 0..t only: the logits of every prefix are the first rows of
    the logits of the whole sequence, and changing a later token changes no earlier row."""
    w = _weights()
    ids = _ids(8)
    full = _call(mod, w, ids)
    for t in (1, 3, L - 1):
        _close(_call(mod, w, ids[:t]), full[:t], 1e-12, "prefix of %d tokens" % t)
    other = ids.clone()
    other[-1] = (other[-1] + 1) % CFG["vocab"]
    changed = _call(mod, w, other)
    _close(changed[:-1], full[:-1], 1e-12, "earlier rows after changing the last token")
    assert np.abs(changed[-1] - full[-1]).max() > 0, "the last token must reach its own row"


def pin_decoder_zero_blocks_closed_form(mod):
    """With wo = wdown = 0 each block adds exact zeros to the residual stream, so
    logits = bf16(rmsnorm(emb[ids]) * lnf) . lm_head^T, computed here with numpy."""
    w = _weights(zero_out=True)
    ids = _ids(9)
    e = w["emb"].double().numpy()[ids.numpy()]
    g = w["lnf"].double().numpy()
    n = e / np.sqrt((e * e).mean(axis=1, keepdims=True) + CFG["eps"]) * g
    n = torch.from_numpy(n).to(torch.bfloat16).double().numpy()
    want = n @ w["lm_head"].double().numpy().T
    _close(_call(mod, w, ids), want, 1e-12, "zero blocks: closed form")


DECODER_PINS = [pin_decoder_matches_independent_forward, pin_decoder_prefix_is_causal,
                pin_decoder_zero_blocks_closed_form]
