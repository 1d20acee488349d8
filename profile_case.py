"""Run one kernel case a few times, for profilers (ncu) and quick timing.

  python profile_case.py linear M N K [--reps R]
  python profile_case.py matmul M N K [--reps R]
  python profile_case.py sdpa B H Hkv Lq Lkv [--reps R]
  python profile_case.py qlinear M N K BITS GROUP [--reps R]
      (bf16 activations; each call on one of 8 quantized weight copies, so the
      packed weights come from HBM)
  python profile_case.py sweep [--reps R]
      (bf16 linear, K=4096, N in {4096, 11008, 14336}, M in {1,..,512}, each call
      on one of 4 weight copies, as in the benchmark's batch sweep)

Inputs are seeded synthetic bf16 tensors on cuda:0.  Prints the CUDA-event
time per call of the last repetitions (not meaningful under a profiler).
"""
from __future__ import annotations

import argparse
import math
import os
import sys

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=("linear", "matmul", "sdpa", "sweep", "qlinear"))
    ap.add_argument("dims", type=int, nargs="*")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()

    import attention_bi_matmul_gb300 as bi
    from attention_bi_matmul_gb300 import synth
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    if args.op in ("linear", "matmul"):
        M, N, K = args.dims
        a, b = synth.gemm16(M, N, K, "bf16", seed=0, layout=args.op, device=dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = (lambda: bi.linear(a, b, out=y)) if args.op == "linear" else (lambda: bi.matmul(a, b, out=y))
        work = "%.3f GFLOP" % (2.0 * M * N * K / 1e9)
    elif args.op == "qlinear":
        M, N, K, bits, gs = args.dims
        x = synth.normal((M, K), 0, 1.0, "bf16", dev)
        copies = [synth.qweights(N, K, bits, gs, "bf16", seed=i, device=dev) for i in range(8)]
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        state = {"i": 0}

        def fn():
            wq, sc, bs = copies[state["i"] % 8]
            state["i"] += 1
            bi.qlinear(x, wq, sc, bs, bits, gs, out=y)
        nbytes = N * K * bits / 8 + 2 * 2 * N * K / gs + 2 * M * K + 2 * M * N
        work = "%.4f GB (packed weights, scales, biases, x, y)" % (nbytes / 1e9)
    elif args.op == "sweep":
        Ns, Ms, K = (4096, 11008, 14336), (1, 2, 3, 4, 8, 16, 32, 64, 128, 256, 512), 4096
        x = synth.normal((512, K), 0, 1.0 / math.sqrt(K), "bf16", dev)
        ws = {N: [synth.normal((N, K), 10 * N + i, 1.0 / math.sqrt(K), "bf16", dev) for i in range(4)]
              for N in Ns}
        ys = {N: torch.empty((512, N), dtype=torch.bfloat16, device=dev) for N in Ns}

        def fn():
            i = 0
            for N in Ns:
                for M in Ms:
                    bi.linear(x[:M], ws[N][i % 4], out=ys[N][:M])
                    i += 1
        work = "%.3f GB of weights" % (2.0 * len(Ms) * K * sum(Ns) / 1e9)
    else:
        B, H, Hkv, Lq, Lkv = args.dims
        q, k, v = synth.sdpa_qkv(B, H, Hkv, Lq, Lkv, 128, "bf16", seed=0, device=dev)
        o = torch.empty_like(q)
        fn = lambda: bi.sdpa(q, k, v, causal=True, out=o)
        work = "%.3f GB of K/V" % (4.0 * B * Hkv * Lkv * 128 / 1e9)
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    st, code = bi.last_device_error()
    print("%s %s: %s, %.4f ms per call, device status %d" % (
        args.op, args.dims, work, e0.elapsed_time(e1) / args.reps, st))
    if st != 0:
        sys.exit(1)


if __name__ == "__main__":
    main()
