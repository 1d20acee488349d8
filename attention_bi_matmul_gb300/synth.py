"""Seeded synthetic inputs for the GEMM / attention / decoder workloads.

This module only draws random numbers; it holds none of the method's
arithmetic.  The same tensors feed the CUDA library and the fp64 oracle.

Two sources, both seeded:
  * ``device="cpu"``: a CPU ``torch.Generator`` (used for every size the oracle
    checks element by element);
  * ``device="cuda"``: a CUDA ``torch.Generator`` (used for the full-size
    workloads, whose inputs are too large to draw on the host in reasonable
    time).  The oracle then receives host copies of the slices it checks.

Distributions follow the workloads in the design notes: GEMM operands
N(0,1)/sqrt(K) (fp32 linear: N(0,1)/16, bias N(0,0.1)), attention q/k/v N(0,1),
decoder weights N(0,0.02), token ids uniform over the vocabulary, quantized
weights as uniformly random packed words with per-group scales and biases.
"""
from __future__ import annotations

import math

import torch

_DT = {"f32": torch.float32, "fp32": torch.float32, "float32": torch.float32,
       "f16": torch.float16, "fp16": torch.float16, "float16": torch.float16,
       "bf16": torch.bfloat16, "bfloat16": torch.bfloat16}


def dtype_of(name) -> torch.dtype:
    if isinstance(name, torch.dtype):
        return name
    return _DT[name]


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, std: float = 1.0, dtype="f32", device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32 from a seeded generator, then cast to ``dtype``."""
    g = generator(seed, device)
    t = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype_of(dtype))


def bernoulli_mask(shape, p_visible: float, seed: int, device="cpu") -> torch.Tensor:
    """Boolean mask, each element True (visible) with probability ``p_visible``."""
    g = generator(seed, device)
    return torch.rand(tuple(shape), generator=g, dtype=torch.float32, device=device) < p_visible


def uniform_ids(shape, vocab: int, seed: int, device="cpu") -> torch.Tensor:
    g = generator(seed, device)
    return torch.randint(0, vocab, tuple(shape), generator=g, dtype=torch.int64, device=device)


# ---------------------------------------------------------------- workloads

def linear_f32(M: int, seed: int = 0, K: int = 256, N: int = 512, device="cpu"):
    """fp32 linear: x[M,K], w[N,K] ~ N(0,1)/16, bias[N] ~ N(0,0.1).

    Row m of x does not depend on M (x is drawn for max(M, 8) rows and sliced),
    so row 0 is the same request at every batch size.
    """
    Mg = max(M, 8)
    x = normal((Mg, K), seed, 1.0 / 16, "f32", device)[:M].contiguous()
    w = normal((N, K), seed + 1, 1.0 / 16, "f32", device)
    bias = normal((N,), seed + 2, 0.1, "f32", device)
    return x, w, bias


def gemm16(M: int, N: int, K: int, dtype="bf16", seed: int = 0, layout="matmul",
           device="cpu", with_c: bool = False, c_row: bool = False):
    """16-bit GEMM operands ~ N(0,1)/sqrt(K).

    layout="matmul": b[K,N];  layout="linear": w[N,K].  With ``with_c`` also
    returns c[M,N] (or a row c[N]) ~ N(0,1)/sqrt(K) for addmm.
    """
    s = 1.0 / math.sqrt(K)
    a = normal((M, K), seed, s, dtype, device)
    if layout == "matmul":
        b = normal((K, N), seed + 1, s, dtype, device)
    else:
        b = normal((N, K), seed + 1, s, dtype, device)
    if not with_c:
        return a, b
    c = normal((N,) if c_row else (M, N), seed + 2, s, dtype, device)
    return a, b, c


def qweights(N: int, K: int, bits: int, group_size: int, dtype="bf16", seed: int = 0,
             device="cpu"):
    """Synthetic group-wise affine quantized weights of an [N, K] layer.

    wq: int32 [N, K*bits/32], uniformly random words (every bit pattern is a valid
    packing of 32/bits fields); scales ~ U(0.5, 1.5) * 6 sigma / (2^bits - 1) and
    biases ~ -3 sigma * U(0.8, 1.2) per group, sigma = 1/sqrt(K), so the weights
    span about [-3 sigma, 3 sigma] as a quantized N(0, sigma^2) layer would.
    """
    g = generator(seed, device)
    wq = torch.randint(-2 ** 31, 2 ** 31, (N, K * bits // 32), generator=g, dtype=torch.int64,
                       device=device).to(torch.int32)
    sigma = 1.0 / math.sqrt(K)
    G = K // group_size
    u = torch.rand((N, G), generator=g, dtype=torch.float32, device=device)
    scales = (0.5 + u) * (6.0 * sigma / (2 ** bits - 1))
    v = torch.rand((N, G), generator=g, dtype=torch.float32, device=device)
    biases = -3.0 * sigma * (0.8 + 0.4 * v)
    return wq, scales.to(dtype_of(dtype)), biases.to(dtype_of(dtype))


def sdpa_qkv(B: int, H: int, Hkv: int, Lq: int, Lkv: int, D: int = 128, dtype="bf16",
             seed: int = 0, device="cpu"):
    """q[B,H,Lq,D], k/v[B,Hkv,Lkv,D] ~ N(0,1)."""
    q = normal((B, H, Lq, D), seed, 1.0, dtype, device)
    k = normal((B, Hkv, Lkv, D), seed + 1, 1.0, dtype, device)
    v = normal((B, Hkv, Lkv, D), seed + 2, 1.0, dtype, device)
    return q, k, v
