"""GEMM parity against the fp64 oracle and batch invariance, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from attention_bi_matmul_gb300 import synth
from tolerances import assert_same_bits, bits, check_close, count_bit_diffs

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


@pytest.fixture(scope="module")
def bi():
    import __graft_entry__
    __graft_entry__.build()
    import attention_bi_matmul_gb300 as m
    torch.cuda.set_device(0)
    return m


def _dev(*ts):
    return [t.cuda() for t in ts]


def _no_device_error(bi):
    st, code = bi.last_device_error()
    assert st == 0, "device error word %#x" % code


# ------------------------------------------------------------------ fp32 linear (small config)

def test_fp32_linear_rows_invariant_and_accurate(bi):
    """x[M,256] . w[512,256]^T + bias, M in {1,2,3,4,8}: row 0 bit-identical across M,
    every row within 1e-5 * sum|x w| of the fp64 oracle."""
    outs = {}
    for M in (1, 2, 3, 4, 8):
        x, w, bias = synth.linear_f32(M, seed=0)
        y = bi.linear(*_dev(x, w, bias))
        ref, nrm = oracle.linear(x, w, bias)
        check_close(y, ref, nrm, torch.float32, "fp32 linear M=%d" % M)
        outs[M] = y
    for M in (2, 3, 4, 8):
        assert_same_bits(outs[M][:1], outs[1], "fp32 linear row 0, M=%d vs M=1" % M)
        assert_same_bits(outs[M], outs[8][:M], "fp32 linear rows, M=%d vs M=8" % M)
    _no_device_error(bi)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (70, 130, 90), (129, 65, 257), (5, 300, 33)])
def test_fp32_matmul_addmm_ragged(bi, M, N, K):
    a, b, c = synth.gemm16(M, N, K, "fp32", seed=3, with_c=True)
    y = bi.matmul(*_dev(a, b))
    ref, nrm = oracle.matmul(a, b)
    check_close(y, ref, nrm, torch.float32, "fp32 matmul %s" % ((M, N, K),))
    ya = bi.addmm(*_dev(c, a, b), alpha=0.5, beta=-1.5)
    ref, nrm = oracle.addmm(c, a, b, 0.5, -1.5)
    check_close(ya, ref, nrm, torch.float32, "fp32 addmm")
    crow = c[0].contiguous()
    yr = bi.addmm(*_dev(crow, a, b))
    ref, nrm = oracle.addmm(crow, a, b)
    check_close(yr, ref, nrm, torch.float32, "fp32 addmm row c")


# ------------------------------------------------------------------ 16-bit parity, every tile width

def _k_for_width(bi, layout, bn):
    """A K that selects the built tile width `bn` (the width is a function of K)."""
    for K in (256, 4096, 8192, 16384):
        if bi.gemm_config(4096, K, torch.bfloat16, layout)[0] == bn:
            return K
    raise AssertionError("no K selects width %d" % bn)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_tile_widths_depend_on_K_only(bi, dt):
    for layout in ("linear", "matmul"):
        widths = {bi.gemm_config(N, K, DT[dt], layout)[0]
                  for N in (8, 4096, 11008, 14336, 38912) for K in (64, 4096)}
        assert widths == {128}
        assert bi.gemm_config(4096, 8192, DT[dt], layout)[0] == 256


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("layout_bn", ["linear-128", "linear-256", "matmul-128", "matmul-256"])
def test_16bit_parity_each_width(bi, dt, layout_bn):
    layout, bn = layout_bn.split("-")
    K = _k_for_width(bi, layout, int(bn))
    M, N = 300, 1000          # three row tiles (ragged), several column tiles (ragged)
    a, b, c = synth.gemm16(M, N, K, dt, seed=5, layout=layout, with_c=True)
    ad, bd, cd = _dev(a, b, c)
    cols = np.r_[0:300, 600:1000]
    if layout == "linear":
        bias = synth.normal((N,), 6, 0.1, dt)
        y = bi.linear(ad, bd, bias.cuda())
        ref, nrm = oracle.linear(a, b[cols], bias[cols])
        check_close(y[:, cols], ref, nrm, DT[dt], "linear bn=%s K=%d" % (bn, K))
    else:
        y = bi.matmul(ad, bd)
        bs = b[:, cols].contiguous()
        ref, nrm = oracle.matmul(a, bs)
        check_close(y[:, cols], ref, nrm, DT[dt], "matmul bn=%s K=%d" % (bn, K))
        ya = bi.addmm(cd, ad, bd, alpha=1.0, beta=1.0)
        ref, nrm = oracle.addmm(c[:, cols].contiguous(), a, bs, 1.0, 1.0)
        check_close(ya[:, cols], ref, nrm, DT[dt], "addmm bn=%s" % bn)
        ya = bi.addmm(cd[0].contiguous(), ad, bd, alpha=-0.75, beta=2.0)
        ref, nrm = oracle.addmm(c[0, cols].contiguous(), a, bs, -0.75, 2.0)
        check_close(ya[:, cols], ref, nrm, DT[dt], "addmm row-c bn=%s" % bn)
    _no_device_error(bi)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (1, 40, 72), (17, 520, 1000), (128, 256, 64),
                                   (129, 96, 4096), (3, 2056, 136)])
def test_16bit_ragged_shapes(bi, dt, M, N, K):
    """Sizes that are not multiples of the tiles: tails in M, N and K, tiny N and K."""
    x, w = synth.gemm16(M, N, K, dt, seed=7, layout="linear")
    y = bi.linear(*_dev(x, w))
    ref, nrm = oracle.linear(x, w)
    check_close(y, ref, nrm, DT[dt], "linear %s" % ((M, N, K),))
    a, b = synth.gemm16(M, N, K, dt, seed=8, layout="matmul")
    y = bi.matmul(*_dev(a, b))
    ref, nrm = oracle.matmul(a, b)
    check_close(y, ref, nrm, DT[dt], "matmul %s" % ((M, N, K),))


def test_integer_exact_bits(bi):
    """Small-integer operands: every partial sum is exact in fp32, so every dtype path and
    the oracle agree exactly (pins the GEMM and its epilogue bits)."""
    g = torch.Generator().manual_seed(21)
    M, N, K = 130, 200, 96
    a = torch.randint(-2, 3, (M, K), generator=g).float()
    b = torch.randint(-2, 3, (K, N), generator=g).float()
    c = torch.randint(-3, 4, (N,), generator=g).float()
    want = torch.from_numpy(oracle.addmm(c, a, b, 1.0, 1.0)[0])
    assert want.abs().max() <= 256
    for dt in (torch.float32, torch.bfloat16, torch.float16):
        ad, bd, cd = a.to(dt).cuda(), b.to(dt).cuda(), c.to(dt).cuda()
        y = bi.addmm(cd, ad, bd).float().cpu().double()
        assert torch.equal(y, want), "integer-exact addmm %s" % dt
        y = bi.linear(ad, bd.t().contiguous(), cd).float().cpu().double()
        assert torch.equal(y, want), "integer-exact linear %s" % dt


# ------------------------------------------------------------------ the 16-bit batch-size config

C2_M = (1, 2, 3, 4, 8, 16, 32, 64, 128, 256, 512)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("N", [4096, 11008, 14336])
def test_c2_rows_invariant_across_batch(bi, dt, N):
    """K=4096: every row's bits are the same for M in {1..512}, for matmul, addmm and linear,
    and with different batch neighbours; sampled rows/columns match the oracle."""
    K = 4096
    a, b, c = synth.gemm16(512, N, K, dt, seed=1, with_c=True, device="cuda")
    w = b.t().contiguous()
    full_m = bi.matmul(a, b)
    full_a = bi.addmm(c, a, b, alpha=1.0, beta=1.0)
    full_l = bi.linear(a, w)
    for M in C2_M:
        assert_same_bits(bi.matmul(a[:M], b), full_m[:M], "matmul N=%d M=%d" % (N, M))
        assert_same_bits(bi.addmm(c[:M], a[:M], b, alpha=1.0, beta=1.0), full_a[:M],
                         "addmm N=%d M=%d" % (N, M))
        assert_same_bits(bi.linear(a[:M], w), full_l[:M], "linear N=%d M=%d" % (N, M))
    # batch neighbours: row 0 surrounded by other rows
    perm = torch.randperm(511, generator=torch.Generator().manual_seed(2))[:63].cuda() + 1
    mixed = torch.cat([a[:1], a[perm]], 0)
    assert_same_bits(bi.matmul(mixed, b)[:1], full_m[:1], "matmul neighbours")
    # accuracy on sampled rows
    rows = [0, 1, 255, 511]
    cols = np.r_[0:128, N - 128:N]
    ah = a[rows].cpu()
    bh = b[:, cols].contiguous().cpu()
    ref, nrm = oracle.matmul(ah, bh)
    check_close(full_m[rows][:, cols], ref, nrm, DT[dt], "matmul N=%d sampled" % N)
    ref, nrm = oracle.addmm(c[rows][:, cols].cpu(), ah, bh, 1.0, 1.0)
    check_close(full_a[rows][:, cols], ref, nrm, DT[dt], "addmm N=%d sampled" % N)
    _no_device_error(bi)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_rows_invariant_wide_tile_k8192(bi, dt):
    """The same row-bits property on the 256-column tile (K = 8192), M up to 512."""
    a, b = synth.gemm16(512, 8192, 8192, dt, seed=12, device="cuda")
    full = bi.matmul(a, b)
    for M in C2_M:
        assert_same_bits(bi.matmul(a[:M], b), full[:M], "matmul K=8192 M=%d" % M)
    rows = [0, 300, 511]
    cols = np.r_[0:64, 8128:8192]
    ref, nrm = oracle.matmul(a[rows].cpu(), b[:, cols].contiguous().cpu())
    check_close(full[rows][:, cols], ref, nrm, DT[dt], "K=8192 sampled")


def test_linear_8192_cube_full_size_sampled(bi):
    """The bench's large GEMM at full size and in the bench's launch form (bi_linear, CTA
    pairs, two K panels per stage, more tiles than resident pairs): sampled outputs from
    every corner and the middle against the oracle, and the same bits on a second call."""
    x, w = synth.gemm16(8192, 8192, 8192, "bf16", seed=21, layout="linear", device="cuda")
    y = bi.linear(x, w)
    rows = [0, 1, 127, 128, 4095, 4096, 8190, 8191]
    cols = np.r_[0:32, 4080:4112, 8160:8192]
    ref, nrm = oracle.linear(x[rows].cpu(), w[cols].contiguous().cpu())
    check_close(y[rows][:, cols], ref, nrm, torch.bfloat16, "8192^3 linear sampled")
    assert_same_bits(bi.linear(x, w), y, "8192^3 linear, second call")
    _no_device_error(bi)


def test_c2_cublas_control_differs(bi):
    """The negative control: torch.matmul (cuBLAS) changes a row's bits with the batch size
    on at least one of the config's shapes, where the library's do not."""
    K = 4096
    diffs = 0
    for dt in ("bf16", "fp16"):
        for N in (4096, 11008, 14336):
            a, b = synth.gemm16(512, N, K, dt, seed=1, device="cuda")
            ref = torch.matmul(a[:1], b)
            for M in C2_M[1:]:
                diffs += count_bit_diffs(torch.matmul(a[:M], b)[:1], ref)
    print("cuBLAS control: %d differing bit patterns in row 0 across the sweep" % diffs)
    assert diffs > 0, "cuBLAS was batch-invariant on every shape of the sweep"


def test_eager_vs_cuda_graph(bi):
    """The same calls captured in a CUDA graph and replayed give the same bits."""
    a, b, c = synth.gemm16(64, 4096, 4096, "bf16", seed=4, with_c=True, device="cuda")
    w = b.t().contiguous()
    eager = (bi.linear(a, w), bi.addmm(c, a, b))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        bi.linear(a, w)   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    yl = torch.empty_like(eager[0])
    ya = torch.empty_like(eager[1])
    with torch.cuda.graph(g):
        bi.linear(a, w, out=yl)
        bi.addmm(c, a, b, out=ya)
    g.replay()
    torch.cuda.synchronize()
    assert_same_bits(yl, eager[0], "linear graph vs eager")
    assert_same_bits(ya, eager[1], "addmm graph vs eager")
    g.replay()
    torch.cuda.synchronize()
    assert_same_bits(yl, eager[0], "linear graph replay 2")


def test_repeated_runs_identical(bi):
    a, b = synth.gemm16(200, 11008, 4096, "bf16", seed=9, device="cuda")
    y0 = bi.matmul(a, b)
    for _ in range(3):
        assert_same_bits(bi.matmul(a, b), y0, "repeat")


# ------------------------------------------------------------------ the CTA-pair tile (K >= 8192)

@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_pair_tile_linear_rows_invariant(bi, dt):
    """K-major weights on the 256-row pair tile: a row's bits do not depend on M, across
    the 128-row boundary between the pair's CTAs and the 256-row boundary between tiles."""
    K, N = 8192, 1000
    x, w = synth.gemm16(700, N, K, dt, seed=31, layout="linear", device="cuda")
    full = bi.linear(x, w)
    for M in (1, 16, 127, 128, 129, 255, 256, 257, 511, 512, 700):
        assert_same_bits(bi.linear(x[:M], w), full[:M], "linear K=8192 M=%d" % M)
    rows = [0, 127, 128, 255, 256, 383, 384, 699]
    cols = np.r_[0:70, 930:1000]
    ref, nrm = oracle.linear(x[rows].cpu(), w[cols].cpu())
    check_close(full[rows][:, cols], ref, nrm, DT[dt], "pair linear sampled")
    _no_device_error(bi)


@pytest.mark.parametrize("layout", ["linear", "matmul"])
def test_pair_tile_more_tiles_than_pairs(bi, layout):
    """2304 x 2600 outputs at K = 8192: 9 x 11 = 99 pair tiles, more than the pairs the
    device holds at once, so pairs loop over tiles and both accumulator buffers turn over."""
    M, N, K = 2304, 2600, 8192
    a, b = synth.gemm16(M, N, K, "bf16", seed=32, layout=layout, device="cuda")
    y = bi.linear(a, b) if layout == "linear" else bi.matmul(a, b)
    rows = [0, 255, 256, 1151, 2047, 2303]
    cols = np.r_[0:40, 1280:1300, 2560:2600]
    if layout == "linear":
        ref, nrm = oracle.linear(a[rows].cpu(), b[cols].cpu())
    else:
        ref, nrm = oracle.matmul(a[rows].cpu(), b[:, cols].contiguous().cpu())
    check_close(y[rows][:, cols], ref, nrm, torch.bfloat16, "pair %s 2304x2600" % layout)
    # the first 300 rows alone give the same bits
    y2 = bi.linear(a[:300], b) if layout == "linear" else bi.matmul(a[:300], b)
    assert_same_bits(y2, y[:300], "pair %s first 300 rows" % layout)
    _no_device_error(bi)


def test_pair_tile_batched_entries(bi):
    """Batched matmul at K = 8192 (pair tiles with a batch coordinate): each entry equals
    its own unbatched product, bit for bit, for a shared and a per-entry right operand."""
    Bt, M, N, K = 3, 200, 264, 8192
    g = torch.Generator().manual_seed(33)
    a = (torch.randn(Bt, M, K, generator=g) / 64).to(torch.bfloat16).cuda()
    b = (torch.randn(Bt, K, N, generator=g) / 64).to(torch.bfloat16).cuda()
    y = bi.bmm(a, b)
    ys = bi.bmm(a, b[0])
    for e in range(Bt):
        assert_same_bits(y[e], bi.matmul(a[e], b[e]), "entry %d" % e)
        assert_same_bits(ys[e], bi.matmul(a[e], b[0]), "shared b entry %d" % e)
    ref, nrm = oracle.matmul(a[1, :9].cpu(), b[1].cpu())
    check_close(y[1, :9], ref, nrm, torch.bfloat16, "pair bmm entry 1")
    _no_device_error(bi)


@pytest.mark.parametrize("layout", ["linear", "matmul"])
def test_pair_tile_stage_shape_keeps_bits(bi, layout):
    """The pair kernel stages two K panels at a time when every pair has at least two tiles
    (4096 x 2600 at K = 8192: 16 x 11 = 176 tiles) and one otherwise (the first 256 rows
    alone: 11 tiles). The stage shape is scheduling only: the rows' bits must agree."""
    M, N, K = 4096, 2600, 8192
    a, b = synth.gemm16(M, N, K, "bf16", seed=34, layout=layout, device="cuda")
    fn = bi.linear if layout == "linear" else bi.matmul
    full = fn(a, b)
    assert_same_bits(fn(a[:256], b), full[:256], "%s first 256 rows vs all 4096" % layout)
    assert_same_bits(fn(a[3000:3001], b), full[3000:3001], "%s row 3000 alone" % layout)
    rows = [0, 1000, 4095]
    cols = np.r_[0:32, 2568:2600]
    if layout == "linear":
        ref, nrm = oracle.linear(a[rows].cpu(), b[cols].cpu())
    else:
        ref, nrm = oracle.matmul(a[rows].cpu(), b[:, cols].contiguous().cpu())
    check_close(full[rows][:, cols], ref, nrm, torch.bfloat16, "pair %s 4096 rows" % layout)
    _no_device_error(bi)


@pytest.mark.parametrize("layout", ["linear", "matmul"])
def test_pair_tile_odd_panel_count_keeps_bits(bi, layout):
    """K = 8256 has an odd number (129) of 64-wide K panels.  With two panels per stage the
    last stage holds one panel past K; it must not be multiplied, or a row whose
    accumulator is a signed zero would change bits between the two stage shapes (4096 rows:
    256 tiles, two panels per stage; 256 rows: 16 tiles, one).  Rows of +0 and of -0
    are included."""
    M, N, K = 4096, 4096, 8256
    a, b = synth.gemm16(M, N, K, "bf16", seed=35, layout=layout, device="cuda")
    a[5] = 0.0
    a[6] = -0.0
    a[7, : K // 2] = -0.0
    fn = bi.linear if layout == "linear" else bi.matmul
    full = fn(a, b)
    assert_same_bits(fn(a[:256], b), full[:256], "%s K=8256 first 256 rows vs all 4096" % layout)
    for r in (5, 6, 7, 300):
        assert_same_bits(fn(a[r:r + 1], b), full[r:r + 1], "%s K=8256 row %d alone" % (layout, r))
    rows = [0, 5, 7, 4095]
    cols = np.r_[0:32, 4064:4096]
    if layout == "linear":
        ref, nrm = oracle.linear(a[rows].cpu(), b[cols].cpu())
    else:
        ref, nrm = oracle.matmul(a[rows].cpu(), b[:, cols].contiguous().cpu())
    check_close(full[rows][:, cols], ref, nrm, torch.bfloat16, "pair %s K=8256" % layout)
    _no_device_error(bi)
