"""bi_gemm on the GPU: parity with the oracle's sequential fp32 GEMM, exact
results on integer data, and bitwise batch invariance (ybb.press sections
1, 2.2 and 4: the same row must give the same bits for every M, every row
position and every tile plan)."""
import numpy as np
import pytest
import torch

from helpers import bits, f32bits, gamma, sum_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    from deterministic_invariant_bf16_gb300 import binding, build
    build.build()
    binding.lib()
    return binding


def gemm(bi, x, W, kind=None):
    kind = bi.OUT_F32 if kind is None else kind
    M, K = x.shape
    N = W.shape[0]
    if kind == bi.OUT_BF16:
        out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    elif kind == bi.OUT_SWIGLU:
        out = torch.empty(M, N // 2, dtype=torch.bfloat16, device="cuda")
    else:
        out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    nws = bi.bi_gemm_workspace_size(M, N, K)
    ws = torch.empty(max(nws // 4, 1), dtype=torch.float32, device="cuda")
    bi.bi_gemm(x, W, out, kind, ws)
    torch.cuda.synchronize()
    assert bi.bi_device_status() == 0
    return out


def randn_bf16(shape, seed, std=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(
        torch.bfloat16)


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (5, 384, 512),
                                   (130, 256, 1024), (300, 200, 136),
                                   (257, 1000, 264), (300, 40000, 64),
                                   (3, 14336, 4096)])
def test_exact_on_small_integers(bi, M, N, K):
    """Integer data keeps every partial sum exact, so any correct summation
    order gives exactly the integer product (catches a transposed operand,
    a wrong tile offset or a dropped k-block).  (300, 40000, 64) runs
    several units per CTA over two m-tiles; (3, 14336, 4096) takes CTA
    pairs."""
    g = torch.Generator().manual_seed(M * 7 + N + K)
    xi = torch.randint(-4, 5, (M, K), generator=g)
    wi = torch.randint(-4, 5, (N, K), generator=g)
    out = gemm(bi, xi.to(torch.bfloat16).cuda(), wi.to(torch.bfloat16).cuda())
    ref = (xi.double() @ wi.double().T).float()
    assert torch.equal(out.cpu(), ref)


@pytest.mark.parametrize("M,N,K", [(1, 384, 512), (37, 640, 1024),
                                   (200, 256, 2048), (129, 1000, 264)])
def test_parity_with_oracle(bi, orc, M, N, K):
    """Both results lie within the recursive-summation bound of the exact
    sum, hence within twice that bound of each other."""
    x = randn_bf16((M, K), 1)
    W = randn_bf16((N, K), 2)
    out = gemm(bi, x, W).cpu().numpy().astype(np.float64)
    xb, wb = bits(x), bits(W)
    ref = orc.gemm(xb, wb).astype(np.float64)
    bound = 2 * gamma(K) * sum_bound(orc, xb, wb)
    assert np.all(np.abs(out - ref) <= bound)


def _check_rows(bi, orc, x, W, Ms, sample_rows, n_cols=48):
    full = gemm(bi, x, W)
    fb = f32bits(full)
    for M in Ms:
        part = gemm(bi, x[:M].contiguous(), W)
        assert np.array_equal(f32bits(part), fb[:M]), "M=%d" % M
    for m in sample_rows:
        alone = gemm(bi, x[m:m + 1].contiguous(), W)
        assert np.array_equal(f32bits(alone)[0], fb[m]), "row %d" % m
    # row positions: a permuted batch gives permuted rows, bit for bit
    perm = torch.randperm(x.shape[0], generator=torch.Generator().manual_seed(5))
    permuted = gemm(bi, x[perm.cuda()].contiguous(), W)
    assert np.array_equal(f32bits(permuted), fb[perm.numpy()])
    # oracle parity on sampled outputs at full size
    rng = np.random.default_rng(6)
    cols = np.sort(rng.choice(W.shape[0], size=n_cols, replace=False))
    rows = np.array(sorted(set(sample_rows)))
    xb = bits(x[torch.from_numpy(rows).cuda()])
    wb = bits(W[torch.from_numpy(cols).cuda()])
    ref = orc.gemm(xb, wb).astype(np.float64)
    got = full.cpu().numpy()[rows][:, cols].astype(np.float64)
    bound = 2 * gamma(x.shape[1]) * sum_bound(orc, xb, wb)
    assert np.all(np.abs(got - ref) <= bound)


def test_batch_invariance_4096(bi, orc):
    """W 4096x4096 and x ~ N(0,1): every row of every M in 1..256 equals
    its M=1 result bit for bit (the linear-layer experiment of ybb.press
    section 1, which finds >30% of elements differ with a library GEMM)."""
    W = randn_bf16((4096, 4096), 11)
    x = randn_bf16((256, 4096), 12)
    _check_rows(bi, orc, x, W, [1, 2, 4, 8, 16, 32, 64, 128, 129, 200],
                [0, 1, 7, 63, 127, 128, 200, 255])


@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336),
                                 (14336, 14336), (128256, 4096)])
def test_batch_invariance_8b_shapes(bi, orc, N, K):
    """The 8B FFN and LM-head shapes (and the literal N=K=14336 square),
    covering the 128-, 192- and 256-column tile plans."""
    W = randn_bf16((N, K), 21)
    x = randn_bf16((256, K), 22)
    _check_rows(bi, orc, x, W, [1, 64, 128], [0, 5, 128, 255], n_cols=24)


@pytest.mark.parametrize("M", [1, 70, 256, 300])
def test_kernels_agree_across_plans(bi, M):
    """An output depends on its rows of x and W, on K and on the K slices
    only.  At K = 2048 with one slice, N = 8192 runs the 128-column plan of
    single CTAs, N = 20480 the 192-column plan and N = 90112 the 128-column
    CTA pairs (cta_group::2, M = 256 across two SMs); the columns they
    share agree bit for bit."""
    K = 2048
    Ns = (8192, 20480, 90112)
    assert [bi.bi_gemm_splits(n, K) for n in Ns] == [1, 1, 1]
    assert [bi.bi_gemm_tile_n(n, K) for n in Ns] == [128, 192, 128]
    W = randn_bf16((Ns[-1], K), 71)
    x = randn_bf16((M, K), 72 + M)
    outs = [f32bits(gemm(bi, x, W[:n].contiguous()))[:, :Ns[0]] for n in Ns]
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(outs[0], outs[2])


def test_rows_agree_at_prefill_size(bi):
    """M=2048 (eight m-tiles) against the same rows computed at M=64."""
    W = randn_bf16((4096, 4096), 31)
    x = randn_bf16((2048, 4096), 32)
    big = f32bits(gemm(bi, x, W))
    for lo in (0, 640, 1984):
        small = f32bits(gemm(bi, x[lo:lo + 64].contiguous(), W))
        assert np.array_equal(small, big[lo:lo + 64])


def test_bf16_and_swiglu_epilogues(bi, orc):
    M, F, K = 70, 256, 384
    x = randn_bf16((M, K), 41)
    wg = randn_bf16((F, K), 42, 0.05)
    wu = randn_bf16((F, K), 43, 0.05)
    f32 = gemm(bi, x, wg)
    b16 = gemm(bi, x, wg, bi.OUT_BF16)
    assert np.array_equal(bits(b16), bits(f32.to(torch.bfloat16)))
    wgu = torch.empty(2 * F, K, dtype=torch.bfloat16, device="cuda")
    bi.bi_pack_gate_up(wg, wu, wgu)
    torch.cuda.synchronize()
    w0 = bi.bi_gemm_tile_n(2 * F, K) // 2
    assert torch.equal(wgu[w0:2 * w0], wu[:w0]) and torch.equal(
        wgu[2 * w0:3 * w0], wg[w0:2 * w0])
    sw = gemm(bi, x, wgu, bi.OUT_SWIGLU)
    g = gemm(bi, x, wg).cpu().numpy()
    u = gemm(bi, x, wu).cpu().numpy()
    ref = orc.bf16_bits(orc.swiglu(g, u)).astype(np.int32)
    diff = np.abs(bits(sw).astype(np.int32) - ref)
    assert diff.max() <= 1      # at most one bf16 ulp (expf last bit)
    assert (diff == 0).mean() > 0.99


def _swiglu_via_f32(bi, orc, x, wgu, F):
    """SwiGLU of the F32 GEMM on the interleaved weight (the same plan, so
    the same sums), de-interleaved on the host, by the oracle's formula."""
    K = x.shape[1]
    y = gemm(bi, x, wgu).cpu().numpy()
    w0 = bi.bi_gemm_tile_n(2 * F, K) // 2
    g = np.empty((x.shape[0], F), np.float32)
    u = np.empty_like(g)
    for b in range(-(-F // w0)):
        w = min(w0, F - b * w0)
        g[:, b * w0:b * w0 + w] = y[:, 2 * b * w0:2 * b * w0 + w]
        u[:, b * w0:b * w0 + w] = y[:, 2 * b * w0 + w:2 * b * w0 + 2 * w]
    return orc.bf16_bits(orc.swiglu(g, u)).astype(np.int32)


@pytest.mark.parametrize("F,K,M", [(14336, 4096, 5), (256, 4096, 70),
                                   (20480, 128, 300)])
def test_swiglu_tile_interleave(bi, orc, F, K, M):
    """The 8B gate/up shape (192-column tiles: 96 features per tile and a
    last tile of 32), a shape with 8 K slices (partials reduced by the
    second-stage kernel) and a wide, shallow one with several units per CTA
    over two m-tiles: bi_pack_gate_up's interleave and the SwiGLU epilogue
    agree with the de-interleaved F32 GEMM to one bf16 ulp (the last bit of
    the fast exponential and division)."""
    x = randn_bf16((M, K), 61)
    wg = randn_bf16((F, K), 62, 0.02)
    wu = randn_bf16((F, K), 63, 0.02)
    wgu = torch.empty(2 * F, K, dtype=torch.bfloat16, device="cuda")
    bi.bi_pack_gate_up(wg, wu, wgu)
    sw = gemm(bi, x, wgu, bi.OUT_SWIGLU)
    ref = _swiglu_via_f32(bi, orc, x, wgu, F)
    diff = np.abs(bits(sw).astype(np.int32) - ref)
    assert diff.max() <= 1
    assert (diff == 0).mean() > 0.99
