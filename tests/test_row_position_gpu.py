"""A row's bits do not depend on where it sits in the batch (GPU).

"mlx-batch-invariant" README, "What batch-invariant means here": the bits of a
request must not depend on the batch size or on which rows are its batch
neighbours.  The batch-size sweeps keep the request at row 0; here one request
row is placed at many indices of batches of random other rows -- inside a tile,
on both sides of the 128-row tile boundary, of the 128-row split between the
two CTAs of a pair tile, of the 256-row pair-tile boundary, of the 64-token
tile of the quantized kernel -- and its output row must equal, bit for bit,
the result of the same call on that row alone.  Every GEMM form is covered:
the fp32 SIMT kernel, the one-CTA 128-row tiles (both weight layouts), the
256-row CTA-pair tile (K >= 8192), the quantized linear and the batched matmul.
"""
import pytest
import torch

from attention_bi_matmul_gb300 import synth
from tolerances import assert_same_bits

pytestmark = pytest.mark.gpu

POSITIONS = (0, 1, 63, 64, 65, 77, 127, 128, 129, 255, 256, 257, 383, 384, 511)
BATCH = 512


@pytest.fixture(scope="module")
def bi():
    import __graft_entry__
    __graft_entry__.build()
    import attention_bi_matmul_gb300 as m
    torch.cuda.set_device(0)
    return m


def _no_device_error(bi):
    st, code = bi.last_device_error()
    assert st == 0, "device error word %#x" % code


def _check_positions(fn, request, others, what):
    """fn(rows [M, K]) -> [M, N].  The request alone, then at each position of a batch of
    `others` (random rows), and at the last row of a batch cut just after it."""
    alone = fn(request[None])
    for p in POSITIONS:
        batch = others.clone()
        batch[p] = request
        y = fn(batch)
        assert_same_bits(y[p:p + 1], alone, "%s: row at index %d of %d" % (what, p, BATCH))
        y = fn(batch[:p + 1])
        assert_same_bits(y[p:p + 1], alone, "%s: last row of a batch of %d" % (what, p + 1))


def test_fp32_simt_row_position(bi):
    x, w, bias = synth.linear_f32(BATCH + 1, seed=40, device="cuda")
    _check_positions(lambda r: bi.linear(r, w, bias), x[BATCH], x[:BATCH], "fp32 linear K=256")
    a, b = synth.gemm16(BATCH + 1, 300, 130, "fp32", seed=41, device="cuda")
    _check_positions(lambda r: bi.matmul(r, b), a[BATCH], a[:BATCH], "fp32 matmul ragged")
    _no_device_error(bi)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("N", [4096, 11008, 14336])
def test_one_cta_tile_row_position(bi, dt, N):
    """K = 4096, the batch-size config's shapes: 128-row tiles on one CTA."""
    K = 4096
    x, w = synth.gemm16(BATCH + 1, N, K, dt, seed=42, layout="linear", device="cuda")
    bias = synth.normal((N,), 43, 0.1, dt, "cuda")
    _check_positions(lambda r: bi.linear(r, w, bias), x[BATCH], x[:BATCH], "linear N=%d" % N)
    a, b, c = synth.gemm16(BATCH + 1, N, K, dt, seed=44, with_c=True, c_row=True, device="cuda")
    _check_positions(lambda r: bi.addmm(c, r, b, alpha=0.5, beta=2.0), a[BATCH], a[:BATCH],
                     "addmm (row c) N=%d" % N)
    _no_device_error(bi)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("layout", ["linear", "matmul"])
def test_pair_tile_row_position(bi, dt, layout):
    """K = 8192: 256-row tiles on a CTA pair (rows 0-127 of a tile on the even CTA,
    128-255 on the odd one)."""
    K, N = 8192, 1000
    a, b = synth.gemm16(BATCH + 1, N, K, dt, seed=45, layout=layout, device="cuda")
    fn = (lambda r: bi.linear(r, b)) if layout == "linear" else (lambda r: bi.matmul(r, b))
    _check_positions(fn, a[BATCH], a[:BATCH], "pair %s K=8192" % layout)
    _no_device_error(bi)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_qlinear_row_position(bi, bits):
    """The quantized linear: tiles of 64 token rows."""
    N, K, gs = 1024, 4096, 64
    x = synth.normal((BATCH + 1, K), 46, 1.0, "bf16", "cuda")
    wq, sc, bz = synth.qweights(N, K, bits, gs, "bf16", seed=47, device="cuda")
    bias = synth.normal((N,), 48, 0.1, "bf16", "cuda")
    _check_positions(lambda r: bi.qlinear(r, wq, sc, bz, bits, gs, bias), x[BATCH], x[:BATCH],
                     "qlinear %d-bit" % bits)
    _no_device_error(bi)


@pytest.mark.parametrize("K", [4096, 8192])
def test_bmm_row_position(bi, K):
    """The batched matmul: the request row in entry 1 of 3, at every position."""
    N = 640
    g = torch.Generator(device="cuda").manual_seed(49)
    a = (torch.randn((3, BATCH + 1, K), generator=g, device="cuda") / K ** 0.5).to(torch.bfloat16)
    b = (torch.randn((3, K, N), generator=g, device="cuda") / K ** 0.5).to(torch.bfloat16)
    request = a[1, BATCH].clone()
    alone = bi.matmul(request[None], b[1])
    for p in POSITIONS:
        batch = a[:, :BATCH].clone()
        batch[1, p] = request
        y = bi.bmm(batch, b)
        assert_same_bits(y[1, p:p + 1], alone, "bmm K=%d: entry 1 row %d" % (K, p))
    _no_device_error(bi)
