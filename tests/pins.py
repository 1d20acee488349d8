"""Pins of the fp64 oracle to facts it does not compute itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when
the oracle disagrees with:
  * exact rational brute force (``fractions.Fraction``, ``decimal`` at 60
    digits) on tiny inputs,
  * integer-exact cases, closed forms and invariants of the definitions,
  * independent library routines (numpy float64 matmul, torch CPU float64
    scaled_dot_product_attention / rms_norm / silu).
The shapes are non-square and the data non-symmetric so that a transposed
operand, a wrong index or sign, or a dropped term fails at least one pin;
``test_oracle_mutations.py`` plants such mistakes in a copy of the oracle and
checks that they are caught.
"""
from __future__ import annotations

import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import torch
import torch.nn.functional as F

U64 = 2.0 ** -53  # unit roundoff of fp64


def _rng(seed):
    return np.random.default_rng(seed)


def _fp32_vals(rng, shape, scale=1.0):
    """Random values exactly representable in fp32 (so Fraction(x) is the stored value)."""
    return (rng.standard_normal(shape) * scale).astype(np.float32).astype(np.float64)


def _close(got, want, bound, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    bad = ~(err <= bound)
    assert not bad.any(), "%s: max err %.3e, bound %.3e at %s" % (
        what, float(err.max()), float(np.max(bound)), np.argwhere(bad)[0])


# ------------------------------------------------------------------ GEMM pins

GEMM_SHAPES = [(1, 1, 1), (2, 3, 4), (3, 2, 5), (4, 5, 3), (3, 4, 4)]


def pin_linear_bruteforce(O):
    """linear == exact rational sum, within (K+1)*u*nrm; nrm == exact sum of |terms|."""
    rng = _rng(1)
    for (M, N, K) in GEMM_SHAPES:
        for with_bias in (False, True):
            x = _fp32_vals(rng, (M, K)); w = _fp32_vals(rng, (N, K))
            bias = _fp32_vals(rng, (N,)) if with_bias else None
            y, nrm = O.linear(x, w, bias)
            for m in range(M):
                for n in range(N):
                    terms = [Fraction(x[m, k]) * Fraction(w[n, k]) for k in range(K)]
                    if with_bias:
                        terms.append(Fraction(bias[n]))
                    exact = sum(terms, Fraction(0))
                    mag = sum((abs(t) for t in terms), Fraction(0))
                    tol = (K + 2) * U64 * float(mag)
                    assert abs(Fraction(y[m, n]) - exact) <= Fraction(tol), \
                        "linear(%d,%d,%d)[%d,%d]" % (M, N, K, m, n)
                    assert abs(Fraction(nrm[m, n]) - mag) <= Fraction(tol), "linear nrm"


def pin_matmul_bruteforce(O):
    rng = _rng(2)
    for (M, N, K) in GEMM_SHAPES:
        a = _fp32_vals(rng, (M, K)); b = _fp32_vals(rng, (K, N))
        y, nrm = O.matmul(a, b)
        for m in range(M):
            for n in range(N):
                terms = [Fraction(a[m, k]) * Fraction(b[k, n]) for k in range(K)]
                exact = sum(terms, Fraction(0))
                mag = sum((abs(t) for t in terms), Fraction(0))
                tol = (K + 1) * U64 * float(mag)
                assert abs(Fraction(y[m, n]) - exact) <= Fraction(tol), \
                    "matmul(%d,%d,%d)[%d,%d]" % (M, N, K, m, n)
                assert abs(Fraction(nrm[m, n]) - mag) <= Fraction(tol), "matmul nrm"


def pin_addmm_bruteforce(O):
    rng = _rng(3)
    for (M, N, K) in GEMM_SHAPES:
        for (alpha, beta) in ((1.0, 1.0), (0.5, -2.0), (0.0, 1.0), (1.0, 0.0), (-1.5, 0.25)):
            for c_row in (False, True):
                a = _fp32_vals(rng, (M, K)); b = _fp32_vals(rng, (K, N))
                c = _fp32_vals(rng, (N,) if c_row else (M, N))
                y, nrm = O.addmm(c, a, b, alpha, beta)
                for m in range(M):
                    for n in range(N):
                        s = sum((Fraction(a[m, k]) * Fraction(b[k, n]) for k in range(K)),
                                Fraction(0))
                        mag = sum((abs(Fraction(a[m, k]) * Fraction(b[k, n])) for k in range(K)),
                                  Fraction(0))
                        cv = Fraction(c[n] if c_row else c[m, n])
                        exact = Fraction(beta) * cv + Fraction(alpha) * s
                        emag = abs(Fraction(alpha)) * mag + abs(Fraction(beta) * cv)
                        tol = (K + 3) * U64 * float(emag)
                        assert abs(Fraction(y[m, n]) - exact) <= Fraction(tol), \
                            "addmm a=%g b=%g row=%d (%d,%d,%d)[%d,%d]" % (
                                alpha, beta, c_row, M, N, K, m, n)
                        assert abs(Fraction(nrm[m, n]) - emag) <= Fraction(tol), "addmm nrm"


def pin_gemm_integer_exact(O):
    """Small integers: every partial sum is exact in fp64, so the result is the integer product."""
    rng = _rng(4)
    M, N, K = 7, 9, 33
    a = rng.integers(-2, 3, (M, K)).astype(np.float64)
    b = rng.integers(-2, 3, (K, N)).astype(np.float64)
    bias = rng.integers(-3, 4, (N,)).astype(np.float64)
    want = (a.astype(np.int64) @ b.astype(np.int64)).astype(np.float64)
    y, _ = O.matmul(a, b)
    assert np.array_equal(y, want), "matmul integer-exact"
    y, _ = O.linear(a, b.T.copy(), bias)
    assert np.array_equal(y, want + bias), "linear integer-exact"
    y, _ = O.addmm(bias, a, b, 3.0, -2.0)
    assert np.array_equal(y, 3.0 * want - 2.0 * bias), "addmm integer-exact"


def pin_gemm_numpy(O):
    """numpy float64 matmul (BLAS, another summation order): equal within 2*K*u*nrm."""
    rng = _rng(5)
    M, N, K = 37, 53, 129
    a = rng.standard_normal((M, K)); b = rng.standard_normal((K, N))
    y, nrm = O.matmul(a, b)
    _close(y, a @ b, 2 * K * U64 * nrm, "matmul vs numpy")
    w = rng.standard_normal((N, K)); bias = rng.standard_normal(N)
    y, nrm = O.linear(a, w, bias)
    _close(y, a @ w.T + bias, 2 * (K + 1) * U64 * nrm, "linear vs numpy")
    c = rng.standard_normal((M, N))
    y, nrm = O.addmm(c, a, b, 0.75, -1.25)
    _close(y, -1.25 * c + 0.75 * (a @ b), 2 * (K + 2) * U64 * nrm, "addmm vs numpy")


def pin_gemm_identities(O):
    """w = I gives y = x + bias exactly; linear(x, w) == matmul(x, w^T) bit for bit."""
    rng = _rng(6)
    M, K = 5, 8
    x = rng.standard_normal((M, K)); bias = rng.standard_normal(K)
    y, _ = O.linear(x, np.eye(K), bias)
    assert np.array_equal(y, x + bias), "linear with identity weight"
    w = rng.standard_normal((11, K))
    y1, n1 = O.linear(x, w)
    y2, n2 = O.matmul(x, w.T.copy())
    assert np.array_equal(y1, y2) and np.array_equal(n1, n2), "linear == matmul(w^T)"


# ------------------------------------------------------------------ attention pins

def _decimal_sdpa(q, k, v, causal, q_offset, scale, sinks=None, mask=None):
    """Softmax attention in 60-digit decimal arithmetic, straight from the definition
    (optional sink logit per head in the denominator, optional boolean mask)."""
    getcontext().prec = 60
    B, H, Lq, D = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    G = H // Hkv
    out = np.zeros(q.shape)
    mag = np.zeros(q.shape)
    sc = Decimal(scale)
    for b in range(B):
        for h in range(H):
            hk = h // G
            for i in range(Lq):
                if mask is not None:
                    vis = [j for j in range(Lkv) if mask[b, h, i, j]]
                else:
                    last = q_offset + i if causal else Lkv - 1
                    vis = [j for j in range(Lkv) if j <= last]
                s = [sc * sum(Decimal(q[b, h, i, d]) * Decimal(k[b, hk, j, d]) for d in range(D))
                     for j in vis]
                sk = Decimal(sinks[h]) if sinks is not None else None
                mx = max(s + ([sk] if sk is not None else []))
                e = [(x - mx).exp() for x in s]
                den = sum(e) + ((sk - mx).exp() if sk is not None else Decimal(0))
                for d in range(D):
                    out[b, h, i, d] = float(sum(e[t] * Decimal(v[b, hk, j, d])
                                                for t, j in enumerate(vis)) / den)
                    mag[b, h, i, d] = float(sum(e[t] * abs(Decimal(v[b, hk, j, d]))
                                                for t, j in enumerate(vis)) / den)
    return out, mag


def pin_sdpa_bruteforce(O):
    rng = _rng(7)
    B, H, Hkv, Lq, Lkv, D = 2, 4, 2, 3, 5, 3
    q = rng.standard_normal((B, H, Lq, D)); k = rng.standard_normal((B, Hkv, Lkv, D))
    v = rng.standard_normal((B, Hkv, Lkv, D))
    for causal, q_offset, scale in ((True, 2, None), (True, 0, None), (True, 1, 0.7),
                                    (False, 2, None), (False, 0, 1.3)):
        sc = 1.0 / math.sqrt(D) if scale is None else scale
        o, nrm = O.sdpa(q, k, v, causal=causal, q_offset=q_offset, scale=scale)
        want, wmag = _decimal_sdpa(q, k, v, causal, q_offset, sc)
        _close(o, want, 1e-13 * wmag, "sdpa brute force c=%s off=%d" % (causal, q_offset))
        _close(nrm, wmag, 1e-13 * wmag, "sdpa normaliser c=%s off=%d" % (causal, q_offset))


def _torch_sdpa_f64(q, k, v, causal, q_offset, scale):
    """torch CPU float64 attention with an explicit boolean mask and repeated K/V heads."""
    q, k, v = (torch.from_numpy(np.asarray(t, dtype=np.float64)) for t in (q, k, v))
    B, H, Lq, D = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    G = H // Hkv
    k = k.repeat_interleave(G, dim=1); v = v.repeat_interleave(G, dim=1)
    i = torch.arange(Lq)[:, None]; j = torch.arange(Lkv)[None, :]
    mask = (j <= q_offset + i) if causal else torch.ones(Lq, Lkv, dtype=torch.bool)
    return F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale).numpy()


def pin_sdpa_torch(O):
    rng = _rng(8)
    B, H, Hkv, Lq, Lkv, D = 2, 6, 2, 7, 23, 16
    q = rng.standard_normal((B, H, Lq, D)); k = rng.standard_normal((B, Hkv, Lkv, D))
    v = rng.standard_normal((B, Hkv, Lkv, D))
    for causal, q_offset in ((True, Lkv - Lq), (True, 3), (False, 0)):
        sc = 1.0 / math.sqrt(D)
        o, nrm = O.sdpa(q, k, v, causal=causal, q_offset=q_offset)
        want = _torch_sdpa_f64(q, k, v, causal, q_offset, sc)
        _close(o, want, 1e-12 * nrm + 1e-300, "sdpa vs torch causal=%s off=%d" % (causal, q_offset))


def pin_sdpa_closed_forms(O):
    rng = _rng(9)
    B, H, Hkv, Lq, Lkv, D = 1, 4, 2, 4, 9, 8
    q = rng.standard_normal((B, H, Lq, D)); k = rng.standard_normal((B, Hkv, Lkv, D))
    v = rng.standard_normal((B, Hkv, Lkv, D))
    # one visible key: query 0 at position 0 sees only key 0 -> o = v_0 exactly
    o, _ = O.sdpa(q, k, v, causal=True, q_offset=0)
    for h in range(H):
        assert np.array_equal(o[0, h, 0], v[0, h // 2, 0]), "single visible key"
    # identical keys -> uniform weights -> mean of the visible values
    kc = np.broadcast_to(k[:, :, :1], k.shape).copy()
    o, _ = O.sdpa(q, kc, v, causal=True, q_offset=3)
    for h in range(H):
        for i in range(Lq):
            want = v[0, h // 2, :3 + i + 1].mean(axis=0)
            _close(o[0, h, i], want, 1e-14 * np.abs(v[0, h // 2]).max(), "identical keys")
    # constant values -> the constant; ones -> softmax weights sum to 1
    for c in (1.0, -2.5):
        vc = np.full(v.shape, c)
        o, _ = O.sdpa(q, k, vc, causal=True, q_offset=5)
        _close(o, np.full(o.shape, c), 4e-15 * abs(c), "constant values %g" % c)


def pin_sdpa_structure(O):
    """GQA == MHA on repeated K/V; no mask == causal at the last position; key order free without mask."""
    rng = _rng(10)
    B, H, Hkv, Lq, Lkv, D = 2, 8, 2, 3, 11, 4
    q = rng.standard_normal((B, H, Lq, D)); k = rng.standard_normal((B, Hkv, Lkv, D))
    v = rng.standard_normal((B, Hkv, Lkv, D))
    o1, _ = O.sdpa(q, k, v, causal=True, q_offset=6)
    kr = np.repeat(k, H // Hkv, axis=1); vr = np.repeat(v, H // Hkv, axis=1)
    o2, _ = O.sdpa(q, kr, vr, causal=True, q_offset=6)
    assert np.array_equal(o1, o2), "GQA == MHA with repeated heads"
    q1 = q[:, :, :1].copy()
    a, _ = O.sdpa(q1, k, v, causal=False, q_offset=0)
    b, _ = O.sdpa(q1, k, v, causal=True, q_offset=Lkv - 1)
    assert np.array_equal(a, b), "no mask == causal at the last position"
    perm = rng.permutation(Lkv)
    a, nrm = O.sdpa(q, k, v, causal=False, q_offset=0)
    b, _ = O.sdpa(q, k[:, :, perm], v[:, :, perm], causal=False, q_offset=0)
    _close(a, b, 8 * Lkv * U64 * nrm + 1e-300, "key permutation without mask")


def pin_sdpa_sinks_and_masks_bruteforce(O):
    rng = _rng(14)
    B, H, Hkv, Lq, Lkv, D = 2, 4, 2, 3, 6, 3
    q = rng.standard_normal((B, H, Lq, D)); k = rng.standard_normal((B, Hkv, Lkv, D))
    v = rng.standard_normal((B, Hkv, Lkv, D))
    sinks = rng.standard_normal(H) * 2
    mask = rng.random((B, H, Lq, Lkv)) < 0.6
    mask[..., 0] |= ~mask.any(-1)            # every row sees at least one key
    sc = 1.0 / math.sqrt(D)
    for sk, mk, causal in ((sinks, None, True), (None, mask, True), (sinks, mask, False)):
        o, nrm = O.sdpa_ex(q, k, v, causal=causal, q_offset=3, sinks=sk, mask=mk)
        want, wmag = _decimal_sdpa(q, k, v, causal, 3, sc, sinks=sk, mask=mk)
        _close(o, want, 1e-13 * wmag + 1e-300, "sdpa sinks/mask brute force")
        _close(nrm, wmag, 1e-13 * wmag + 1e-300, "sdpa sinks/mask normaliser")


def pin_sdpa_sinks_and_masks_torch(O):
    """torch CPU float64 SDPA: a boolean mask directly; a sink as one extra key whose score
    is 0 plus an additive mask value of sink_h, carrying a zero value vector."""
    rng = _rng(15)
    B, H, Hkv, Lq, Lkv, D = 2, 6, 3, 5, 19, 8
    q = rng.standard_normal((B, H, Lq, D)); k = rng.standard_normal((B, Hkv, Lkv, D))
    v = rng.standard_normal((B, Hkv, Lkv, D))
    sinks = rng.standard_normal(H) * 1.5
    mask = rng.random((B, H, Lq, Lkv)) < 0.5
    mask[..., 3] = True
    tq, tk, tv = (torch.from_numpy(t) for t in (q, k, v))
    G = H // Hkv
    tk, tv = tk.repeat_interleave(G, 1), tv.repeat_interleave(G, 1)
    o, nrm = O.sdpa_ex(q, k, v, mask=mask)
    want = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(mask)).numpy()
    _close(o, want, 1e-12 * nrm + 1e-300, "array mask vs torch")
    zk = torch.cat([tk, torch.zeros(B, H, 1, D, dtype=torch.float64)], 2)
    zv = torch.cat([tv, torch.zeros(B, H, 1, D, dtype=torch.float64)], 2)
    add = torch.zeros(B, H, Lq, Lkv + 1, dtype=torch.float64)
    add[..., :Lkv] = torch.where(torch.from_numpy(mask), 0.0, float("-inf"))
    add[..., Lkv] = torch.from_numpy(sinks)[None, :, None]
    o, nrm = O.sdpa_ex(q, k, v, sinks=sinks, mask=mask)
    want = F.scaled_dot_product_attention(tq, zk, zv, attn_mask=add).numpy()
    _close(o, want, 1e-12 * np.maximum(nrm, 1e-3), "sinks vs torch extra-key form")


def pin_sdpa_mask_structure(O):
    """causal == the causal pattern as an array mask; an all-true mask == no mask; a sink of
    -inf == no sink; one visible key with a sink: o = v_j * e^s / (e^s + e^sink)."""
    rng = _rng(16)
    B, H, Hkv, Lq, Lkv, D = 1, 4, 2, 4, 9, 8
    q = rng.standard_normal((B, H, Lq, D)); k = rng.standard_normal((B, Hkv, Lkv, D))
    v = rng.standard_normal((B, Hkv, Lkv, D))
    causal_pat = (np.arange(Lkv)[None, :] <= 5 + np.arange(Lq)[:, None])[None, None]
    a, _ = O.sdpa(q, k, v, causal=True, q_offset=5)
    b, _ = O.sdpa_ex(q, k, v, mask=np.broadcast_to(causal_pat, (B, H, Lq, Lkv)))
    assert np.array_equal(a, b), "causal == causal-pattern array mask"
    a, _ = O.sdpa(q, k, v, causal=False)
    b, _ = O.sdpa_ex(q, k, v, mask=np.ones((B, H, Lq, Lkv), bool))
    assert np.array_equal(a, b), "all-true mask == no mask"
    b, _ = O.sdpa_ex(q, k, v, causal=False, sinks=np.full(H, -np.inf))
    assert np.array_equal(a, b), "sink -inf == no sink"
    one = np.zeros((B, H, Lq, Lkv), bool); one[..., 2] = True
    sk = rng.standard_normal(H)
    o, _ = O.sdpa_ex(q, k, v, sinks=sk, mask=one)
    for h in range(H):
        for i in range(Lq):
            s = (q[0, h, i] @ k[0, h // 2, 2]) / math.sqrt(D)
            w = math.exp(s) / (math.exp(s) + math.exp(sk[h]))
            _close(o[0, h, i], w * v[0, h // 2, 2], 1e-14 * np.abs(v).max(), "one key + sink")


# ------------------------------------------------------------------ glue pins

def pin_rmsnorm(O):
    rng = _rng(11)
    x = rng.standard_normal((6, 40)); w = rng.standard_normal(40)
    y = O.rmsnorm(x, w, 1e-6)
    want = F.rms_norm(torch.from_numpy(x), (40,), torch.from_numpy(w), 1e-6).numpy()
    _close(y, want, 1e-14 * np.abs(want).max(), "rmsnorm vs torch")
    for c in (3.0, -0.5):
        xc = np.full((1, 40), c)
        y = O.rmsnorm(xc, w, 1e-6)
        _close(y[0], c / math.sqrt(c * c + 1e-6) * w, 1e-15 * np.abs(w).max(), "rmsnorm constant row")


def pin_rope(O):
    rng = _rng(12)
    T, nh, D = 5, 3, 16
    x = rng.standard_normal((T, nh, D))
    y = O.rope(x, np.zeros(T, dtype=np.int64))
    assert np.array_equal(y, x), "rope at position 0 is the identity"
    pos = np.array([1, 7, 100, 4095, 8191])
    y = O.rope(x, pos)
    half = D // 2
    z = x[..., :half] + 1j * x[..., half:]
    inv = 10000.0 ** (-2.0 * np.arange(half) / D)
    zr = z * np.exp(1j * pos[:, None, None] * inv[None, None, :])
    _close(y[..., :half], zr.real, 1e-12, "rope real part (complex form)")
    _close(y[..., half:], zr.imag, 1e-12, "rope imaginary part (complex form)")
    y2 = O.rope(O.rope(x, np.full(T, 3)), np.full(T, 4))
    _close(y2, O.rope(x, np.full(T, 7)), 1e-13, "rope composition 3+4 == 7")


def pin_swiglu(O):
    rng = _rng(13)
    gu = rng.standard_normal((4, 2 * 24)) * 3
    y = O.swiglu(gu)
    g = torch.from_numpy(gu[:, :24]); u = torch.from_numpy(gu[:, 24:])
    want = (F.silu(g) * u).numpy()
    _close(y, want, 1e-15 * np.abs(want).max() + 1e-300, "swiglu vs torch silu")
    gu0 = gu.copy(); gu0[:, :24] = 0.0
    assert np.array_equal(O.swiglu(gu0), np.zeros((4, 24))), "silu(0) == 0"


# ------------------------------------------------------------------ quantized linear pins

def _fields_by_bitstring(words, bits):
    """Unpack uint32 words into `bits`-wide fields, least significant first, by reading
    each word's binary string (a method independent of shifts and masks)."""
    out = []
    for w in np.asarray(words, dtype=np.uint64).ravel():
        s = format(int(w), "032b")[::-1]           # s[i] = bit i
        for j in range(32 // bits):
            out.append(int(s[j * bits:(j + 1) * bits][::-1], 2))
    return out


def _fields_by_unpackbits(wq, bits):
    """[N, W] uint32 -> [N, W*32/bits] fields, via numpy's little-endian bit unpacking."""
    b = np.unpackbits(np.ascontiguousarray(wq, dtype="<u4").view(np.uint8), axis=1,
                      bitorder="little").astype(np.int64)
    b = b.reshape(wq.shape[0], -1, bits)
    return (b * (1 << np.arange(bits))).sum(axis=2)


def _qweights(rng, N, K, bits, gs, full_range=True):
    wq = rng.integers(0, 2 ** 32, size=(N, K * bits // 32), dtype=np.uint64).astype(np.uint32)
    scales = np.abs(_fp32_vals(rng, (N, K // gs), 0.1)) + 0.01
    biases = _fp32_vals(rng, (N, K // gs), 0.5)
    return wq, scales, biases


def pin_qlinear_bruteforce(O):
    """qlinear == exact rational sum over the bit-string unpacking, within (K+1)*u*nrm."""
    rng = _rng(41)
    for bits in (2, 4, 8):
        for gs in (32, 64):
            M, N, K = 2, 3, 128
            wq, sc, bi = _qweights(rng, N, K, bits, gs)
            x = _fp32_vals(rng, (M, K))
            bias = _fp32_vals(rng, (N,))
            y, nrm = O.qlinear(x, wq, sc, bi, bits, gs, bias)
            for n in range(N):
                q = _fields_by_bitstring(wq[n], bits)
                w = [Fraction(sc[n, k // gs]) * q[k] + Fraction(bi[n, k // gs]) for k in range(K)]
                for m in range(M):
                    exact = sum(Fraction(x[m, k]) * w[k] for k in range(K)) + Fraction(bias[n])
                    mag = sum(abs(Fraction(x[m, k]) * w[k]) for k in range(K)) + abs(Fraction(bias[n]))
                    bound = (K + 2) * U64 * float(mag)
                    assert abs(y[m, n] - float(exact)) <= bound, ("qlinear", bits, gs, m, n)
                    assert abs(nrm[m, n] - float(mag)) <= bound, ("qlinear nrm", bits, gs, m, n)


def pin_qlinear_integer_exact(O):
    """Integer scales, biases and activations: every term and sum is an exact integer, so
    y equals an int64 matmul over numpy's bit unpacking exactly."""
    rng = _rng(42)
    for bits in (2, 4, 8):
        for gs in (32, 128):
            M, N, K = 3, 5, 256
            wq = rng.integers(0, 2 ** 32, size=(N, K * bits // 32), dtype=np.uint64).astype(np.uint32)
            sc = rng.integers(1, 4, size=(N, K // gs)).astype(np.float64)
            bi = rng.integers(-8, 8, size=(N, K // gs)).astype(np.float64)
            x = rng.integers(-2, 3, size=(M, K))
            q = _fields_by_unpackbits(wq, bits)
            w = q * np.repeat(sc, gs, axis=1).astype(np.int64) + np.repeat(bi, gs, axis=1).astype(np.int64)
            want = x @ w.T
            y, _ = O.qlinear(x.astype(np.float64), wq, sc, bi, bits, gs)
            assert np.array_equal(y, want.astype(np.float64)), ("qlinear integer", bits, gs)


def pin_qlinear_closed_forms(O):
    """All fields 0: w = the group's bias; all fields 2^bits - 1: w = s (2^bits - 1) + b."""
    rng = _rng(43)
    M, N, K, gs = 2, 4, 192, 64
    x = _fp32_vals(rng, (M, K))
    for bits in (2, 4, 8):
        _, sc, bi = _qweights(rng, N, K, bits, gs)
        for fill, qv in ((0, 0), (0xFFFFFFFF, 2 ** bits - 1)):
            wq = np.full((N, K * bits // 32), fill, dtype=np.uint32)
            y, _ = O.qlinear(x, wq, sc, bi, bits, gs)
            w = np.repeat(sc * qv + bi, gs, axis=1)
            want = np.array([[math.fsum(x[m] * w[n]) for n in range(N)] for m in range(M)])
            _close(y, want, 4 * K * U64 * (np.abs(x) @ np.abs(w).T), "qlinear closed form %d" % bits)


def pin_qlinear_group_locality(O):
    """With x zero outside group g, y depends on group g's scale and bias only."""
    rng = _rng(44)
    M, N, K, gs, bits = 2, 3, 256, 64, 4
    wq, sc, bi = _qweights(rng, N, K, bits, gs)
    for g in range(K // gs):
        x = np.zeros((M, K))
        x[:, g * gs:(g + 1) * gs] = _fp32_vals(rng, (M, gs))
        y0, _ = O.qlinear(x, wq, sc, bi, bits, gs)
        sc2, bi2 = sc.copy(), bi.copy()
        others = [h for h in range(K // gs) if h != g]
        sc2[:, others] *= 3.0
        bi2[:, others] += 1.0
        y1, _ = O.qlinear(x, wq, sc2, bi2, bits, gs)
        assert np.array_equal(y0, y1), ("group locality", g)
        sc3 = sc.copy()
        sc3[:, g] *= 2.0
        y2, _ = O.qlinear(x, wq, sc3, bi, bits, gs)
        assert not np.array_equal(y0, y2), ("group's own scale matters", g)


ALL_PINS = [pin_linear_bruteforce, pin_matmul_bruteforce, pin_addmm_bruteforce,
            pin_gemm_integer_exact, pin_gemm_numpy, pin_gemm_identities,
            pin_sdpa_bruteforce, pin_sdpa_torch, pin_sdpa_closed_forms, pin_sdpa_structure,
            pin_sdpa_sinks_and_masks_bruteforce, pin_sdpa_sinks_and_masks_torch,
            pin_sdpa_mask_structure,
            pin_qlinear_bruteforce, pin_qlinear_integer_exact, pin_qlinear_closed_forms,
            pin_qlinear_group_locality,
            pin_rmsnorm, pin_rope, pin_swiglu]
