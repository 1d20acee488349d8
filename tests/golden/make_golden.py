"""Write the drift fixtures in this folder from the fp64 oracle.

Calls only ``oracle/`` (and the seeded input generators).  The fixtures detect
drift of the oracle itself: a later change to its arithmetic that moves any of
these values must be deliberate (and regenerate them with a reason).  Each
fixture records the README section whose definition it exercises.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from attention_bi_matmul_gb300 import synth  # noqa: E402


def _l(t):
    return t.double().tolist() if hasattr(t, "double") else t.tolist()


def main():
    fixtures = {}
    x, w, bias = synth.linear_f32(3, seed=7, K=8, N=5)
    y, nrm = oracle.linear(x, w, bias)
    fixtures["linear_f32_small"] = dict(
        cite="mlx-batch-invariant README, 'Use' (linear) and 'How the kernels work' / GEMM "
             "(bias added to the accumulator)",
        inputs=dict(x=_l(x), w=_l(w), bias=_l(bias)), y=y.tolist(), nrm=nrm.tolist())
    a, b, c = synth.gemm16(4, 6, 16, "bf16", seed=8, with_c=True)
    y, nrm = oracle.addmm(c, a, b, 0.5, -1.25)
    fixtures["addmm_bf16_small"] = dict(
        cite="mlx-batch-invariant README, 'Use' (addmm(c, a, b, alpha, beta))",
        inputs=dict(c=_l(c), a=_l(a), b=_l(b), alpha=0.5, beta=-1.25), y=y.tolist(),
        nrm=nrm.tolist())
    q, k, v = synth.sdpa_qkv(1, 4, 2, 3, 7, 8, "bf16", seed=9)
    o, nrm = oracle.sdpa(q, k, v, causal=True, q_offset=3)
    fixtures["sdpa_causal_gqa_small"] = dict(
        cite="mlx-batch-invariant README, 'Use' (scaled_dot_product_attention, mask='causal') "
             "and 'How the kernels work' / Attention",
        inputs=dict(q=_l(q), k=_l(k), v=_l(v), causal=True, q_offset=3), o=o.tolist(),
        nrm=nrm.tolist())
    x = synth.normal((3, 64), 10, 1.0, "bf16")
    wq, sc, bi = synth.qweights(5, 64, 4, 32, "bf16", seed=11)
    bias = synth.normal((5,), 12, 0.1, "bf16")
    y, nrm = oracle.qlinear(x, wq, sc, bi, 4, 32, bias)
    fixtures["qlinear_4bit_small"] = dict(
        cite="mlx-batch-invariant README, 'Quantized models' (2, 4 and 8-bit affine weights "
             "unpacked inside the K loop)",
        inputs=dict(x=_l(x), wq=wq.tolist(), scales=_l(sc), biases=_l(bi), bias=_l(bias),
                    bits=4, group_size=32), y=y.tolist(), nrm=nrm.tolist())
    for name, fx in fixtures.items():
        with open(os.path.join(HERE, name + ".json"), "w") as f:
            json.dump(fx, f, indent=1)
            f.write("\n")
    print("wrote", ", ".join(sorted(fixtures)))


if __name__ == "__main__":
    main()
