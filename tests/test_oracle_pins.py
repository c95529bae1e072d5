"""Pins of the CPU oracle against things other than itself: values the pages
print, closed forms, invariants, float64 brute force, and numpy / torch
library routines.  Each test is chosen so that a plausible slip in the oracle
(a dropped term, a wrong sign or index, a transposed operand) fails it."""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24  # unit roundoff of fp32


def gamma(n):
    return n * U / (1 - n * U)


def rand_bf16_bits(rng, shape, std=1.0):
    x = torch.from_numpy(rng.normal(0, std, size=shape).astype(np.float32))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(orc, bits):
    return orc.bf16_value(bits).astype(np.float64)


# ---------------------------------------------------------------- bf16 --

def test_bf16_rounding_matches_torch(orc):
    """fp32 -> bf16 RNE against torch's CPU conversion (a library routine)
    over 2^22 random bit patterns plus the hard cases."""
    rng = np.random.default_rng(1)
    pats = rng.integers(0, 2 ** 32, size=2 ** 22, dtype=np.uint64).astype(
        np.uint32)
    special = np.array([0x00000000, 0x80000000, 0x7f800000, 0xff800000,
                        0x3f808000, 0x3f818000, 0x3f80ffff, 0x3f817fff,
                        0x7f7fffff, 0x7f7f8000, 0x00000001, 0x807fffff,
                        0x00008000, 0x00018000], np.uint32)
    pats = np.concatenate([special, pats])
    x = pats.view(np.float32)
    mine = orc.bf16_bits(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all(np.isnan(orc.bf16_value(mine[nan])))
    back = orc.bf16_value(mine[~nan])
    ref_back = torch.from_numpy(ref[~nan].view(np.int16)).view(
        torch.bfloat16).float().numpy()
    assert np.array_equal(back.view(np.uint32), ref_back.view(np.uint32))


# ---------------------------------------------------- non-associativity --

def test_nonassoc_values_printed_on_page(orc):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "nonassoc_fp32.txt"))
            if l.strip() and not l.startswith("#")]
    for a, b, c, left, right in rows:
        got = orc.nonassoc_demo(float(a), float(b), float(c))
        assert got == (float(left), float(right))


# ---------------------------------------------------------------- GEMM --

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 9, 64),
                                   (5, 33, 130)])
def test_gemm_within_higham_bound_of_exact(orc, M, N, K):
    """|fl(sum) - exact| <= gamma_K sum|x||w| (Higham, recursive summation)
    with the exact product taken in float64 (bf16 products are exact)."""
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    x = rand_bf16_bits(rng, (M, K))
    w = rand_bf16_bits(rng, (N, K))
    y = orc.gemm(x, w).astype(np.float64)
    xf, wf = bits_to_f64(orc, x), bits_to_f64(orc, w)
    exact = xf @ wf.T
    bound = gamma(K) * (np.abs(xf) @ np.abs(wf).T)
    assert y.shape == (M, N)
    assert np.all(np.abs(y - exact) <= bound + 1e-300)


def test_gemm_exact_on_small_integers(orc):
    """Small integers make every partial sum exact: the result must equal the
    integer matrix product (catches a transposed W or a dropped k)."""
    rng = np.random.default_rng(3)
    xi = rng.integers(-8, 9, size=(6, 40))
    wi = rng.integers(-8, 9, size=(11, 40))
    x = orc.bf16_bits(xi.astype(np.float32))
    w = orc.bf16_bits(wi.astype(np.float32))
    assert np.array_equal(orc.gemm(x, w), (xi @ wi.T).astype(np.float32))


def test_gemm_rows_independent_of_batch(orc):
    """Row m of a batch equals the same row computed alone, bit for bit."""
    rng = np.random.default_rng(4)
    x = rand_bf16_bits(rng, (9, 96))
    w = rand_bf16_bits(rng, (20, 96))
    full = orc.gemm(x, w)
    for m in range(9):
        assert np.array_equal(orc.gemm(x[m:m + 1], w)[0].view(np.uint32),
                              full[m].view(np.uint32))


# ------------------------------------------------------------- RMSNorm --

def test_rmsnorm_constant_row_closed_form(orc):
    """x == c everywhere gives y = c / sqrt(c^2 + eps) * w."""
    H = 64
    rng = np.random.default_rng(5)
    w = rand_bf16_bits(rng, (H,))
    wf = bits_to_f64(orc, w)
    for c in (0.5, -3.0, 1e-3, 7.25):
        y = orc.rmsnorm(np.full((1, H), c, np.float32), w, 1e-5)
        ref = c / math.sqrt(c * c + 1e-5) * wf
        assert np.allclose(y[0], ref, rtol=4 * U * 8, atol=0)


def test_rmsnorm_float64_reference_and_scale_invariance(orc):
    rng = np.random.default_rng(6)
    T, H = 5, 300
    x = rng.normal(0, 2, size=(T, H)).astype(np.float32)
    w = rand_bf16_bits(rng, (H,))
    y = orc.rmsnorm(x, w, 1e-5).astype(np.float64)
    xd = x.astype(np.float64)
    ref = xd / np.sqrt((xd ** 2).mean(1, keepdims=True) + 1e-5) * bits_to_f64(
        orc, w)
    assert np.allclose(y, ref, rtol=gamma(H) * 4 + 8 * U, atol=1e-12)
    # Scaling a row by a power of two (exact) leaves the output unchanged up
    # to eps: the norm divides it out.
    y4 = orc.rmsnorm(x * 4, w, 1e-5 * 16)
    assert np.array_equal(y4, y.astype(np.float32))


# ---------------------------------------------------------------- RoPE --

def test_rope_identity_at_position_zero(orc):
    rng = np.random.default_rng(7)
    x = rng.normal(size=(3, 2, 32)).astype(np.float32)
    assert np.array_equal(orc.rope(x, np.zeros(3, np.int32), 1e4), x)


def test_rope_is_complex_rotation(orc):
    """Half-split RoPE equals multiplying x_i + i x_{i+D/2} by
    exp(i pos theta^(-2i/D)) (numpy complex arithmetic, float64)."""
    rng = np.random.default_rng(8)
    T, nh, D, theta = 6, 3, 32, 5e5
    x = rng.normal(size=(T, nh, D)).astype(np.float32)
    pos = rng.integers(0, 9000, size=T).astype(np.int32)
    y = orc.rope(x, pos, theta).astype(np.float64)
    half = D // 2
    z = x[..., :half].astype(np.float64) + 1j * x[..., half:]
    ang = pos[:, None].astype(np.float64) * theta ** (
        -2.0 * np.arange(half) / D)[None, :]
    rz = z * np.exp(1j * ang)[:, None, :]
    assert np.allclose(y[..., :half], rz.real, atol=2e-6 * 8, rtol=0)
    assert np.allclose(y[..., half:], rz.imag, atol=2e-6 * 8, rtol=0)


def test_rope_relative_position_property(orc):
    """<rope(q, p1), rope(k, p2)> depends only on p1 - p2."""
    rng = np.random.default_rng(9)
    D = 32
    q = rng.normal(size=(1, 1, D)).astype(np.float32)
    k = rng.normal(size=(1, 1, D)).astype(np.float32)
    dots = []
    for shift in (0, 13, 200, 4000):
        a = orc.rope(q, np.array([50 + shift], np.int32), 1e4)
        b = orc.rope(k, np.array([20 + shift], np.int32), 1e4)
        dots.append(float((a.astype(np.float64) * b).sum()))
    assert np.allclose(dots, dots[0], atol=1e-4)


# ----------------------------------------------------------- attention --

def _attention_f64(q, kc, vc, row_req, row_pos, scale):
    T, Hq, D = q.shape
    Hkv = kc.shape[2]
    out = np.zeros((T, Hq, D))
    for t in range(T):
        n = row_pos[t] + 1
        K = np.repeat(kc[row_req[t], :n].astype(np.float64), Hq // Hkv, axis=1)
        V = np.repeat(vc[row_req[t], :n].astype(np.float64), Hq // Hkv, axis=1)
        s = np.einsum("hd,jhd->hj", q[t].astype(np.float64), K) * scale
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        out[t] = np.einsum("hj,jhd->hd", p, V)
    return out


def test_attention_float64_brute_force(orc):
    rng = np.random.default_rng(10)
    R, L, Hq, Hkv, D = 3, 48, 4, 2, 16
    kc = rng.normal(size=(R, L, Hkv, D)).astype(np.float32)
    vc = rng.normal(size=(R, L, Hkv, D)).astype(np.float32)
    row_req = np.array([0, 0, 1, 2, 2, 1], np.int32)
    row_pos = np.array([0, 47, 20, 5, 31, 3], np.int32)
    q = rng.normal(size=(6, Hq, D)).astype(np.float32)
    scale = np.float32(1 / math.sqrt(D))
    got = orc.attention(q, kc, vc, row_req, row_pos, scale)
    ref = _attention_f64(q, kc, vc, row_req, row_pos, float(scale))
    assert np.allclose(got, ref, atol=2e-5, rtol=1e-4)


def test_attention_special_cases(orc):
    rng = np.random.default_rng(11)
    R, L, Hkv, D = 1, 40, 1, 8
    vc = rng.normal(size=(R, L, Hkv, D)).astype(np.float32)
    kc = rng.normal(size=(R, L, Hkv, D)).astype(np.float32)
    q = rng.normal(size=(1, 2, D)).astype(np.float32)
    # one visible key: the output is that key's value, exactly
    out = orc.attention(q, kc, vc, np.array([0], np.int32),
                        np.array([0], np.int32), np.float32(0.3))
    assert np.array_equal(out[0, 0], vc[0, 0, 0])
    # identical keys: uniform weights, the mean of the visible values
    kc_same = np.repeat(kc[:, :1], L, axis=1)
    out = orc.attention(q, kc_same, vc, np.array([0], np.int32),
                        np.array([24], np.int32), np.float32(0.3))
    assert np.allclose(out[0, 1], vc[0, :25, 0].astype(np.float64).mean(0),
                       atol=1e-6)


# -------------------------------------------------------------- SwiGLU --

def test_swiglu(orc):
    rng = np.random.default_rng(12)
    g = rng.normal(0, 3, size=1000).astype(np.float32)
    u = rng.normal(size=1000).astype(np.float32)
    got = orc.swiglu(g, u).astype(np.float64)
    gd = g.astype(np.float64)
    ref = gd / (1 + np.exp(-gd)) * u
    assert np.allclose(got, ref, rtol=8 * U, atol=1e-30)
    z = orc.swiglu(np.array([0.0, -200.0, 200.0], np.float32),
                   np.array([5.0, 5.0, 2.0], np.float32))
    assert z[0] == 0.0 and z[1] == 0.0 and z[2] == 400.0


# -------------------------------------------------------------- argmax --

def test_argmax_matches_numpy(orc):
    rng = np.random.default_rng(13)
    x = rng.normal(size=(64, 777)).astype(np.float32)
    x[3, [10, 500]] = 9.0          # tie: the first wins
    x[4, 7] = np.nan               # NaN is maximal
    x[5, [20, 30]] = np.nan        # first NaN wins
    x[6] = 0.0
    x[6, 0] = -0.0                 # -0 == +0: index 0 wins
    x[7] = -np.inf
    x[8, -1] = np.inf
    assert np.array_equal(orc.argmax(x), np.argmax(x, axis=1))


# -------------------------------------------------------------- Philox --

def test_philox_matches_numpy():
    """Raw Philox4x64-10 blocks against numpy.random.Philox.  numpy bumps
    its counter before each block, so numpy counter c yields block c+1."""
    import oracle
    rng = np.random.default_rng(14)
    for _ in range(20):
        key = rng.integers(0, 2 ** 63, size=2, dtype=np.uint64) * np.uint64(2)
        ctr = rng.integers(0, 2 ** 63, size=4, dtype=np.uint64)
        ctr[0] = ctr[0] & np.uint64(0x7fffffffffffffff)
        g = np.random.Philox(key=key, counter=ctr)
        ref = g.random_raw(4)
        ctr1 = ctr.copy()
        ctr1[0] += np.uint64(1)
        assert np.array_equal(oracle.philox4x64_10(ctr1, key), ref)
    # counter 0 itself: numpy counter 2^256 - 1 wraps to 0
    key = np.array([12345, 0], np.uint64)
    g = np.random.Philox(key=key, counter=np.full(4, 2 ** 64 - 1, np.uint64))
    assert np.array_equal(oracle.philox4x64_10([0, 0, 0, 0], key),
                          g.random_raw(4))


def test_sample_seed_formula():
    import oracle
    rows = [l.split() for l in open(os.path.join(GOLDEN, "sample_seed.txt"))
            if l.strip() and not l.startswith("#")]
    for rid, step, seed in rows:
        assert oracle.sample_seed(int(rid), int(step)) == int(seed)


def test_sample_uniform_is_top_24_bits():
    import oracle
    for seed in (0, 1, 1000003, 2 ** 64 - 5):
        g = np.random.Philox(key=np.array([seed, 0], np.uint64),
                             counter=np.full(4, 2 ** 64 - 1, np.uint64))
        w0 = int(g.random_raw(1)[0])
        assert oracle.sample_uniform(seed) == (w0 >> 40) / 2 ** 24


def test_philox_sample_reductions(orc):
    """tau = 0 is argmax; a one-hot distribution always returns its index;
    frequencies over many (request, step) pairs follow softmax (chi^2)."""
    rng = np.random.default_rng(15)
    logits = rng.normal(size=(8, 50)).astype(np.float32)
    rid = np.arange(8, dtype=np.uint64)
    st = np.zeros(8, np.uint64)
    assert np.array_equal(orc.philox_sample(logits, rid, st, 0.0),
                          np.argmax(logits, 1))
    onehot = np.full((8, 50), -1e4, np.float32)
    onehot[np.arange(8), np.arange(8) * 3] = 0.0
    assert np.array_equal(orc.philox_sample(onehot, rid, st, 1.0),
                          np.arange(8) * 3)
    V, n = 6, 6000
    row = np.log(np.array([0.05, 0.1, 0.15, 0.2, 0.2, 0.3], np.float32))
    lg = np.tile(row, (n, 1))
    ids = orc.philox_sample(lg, np.full(n, 7, np.uint64),
                            np.arange(n, dtype=np.uint64), 1.0)
    counts = np.bincount(ids, minlength=V)
    exp = np.exp(row.astype(np.float64)) / np.exp(row).sum() * n
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 20.5  # 99.9% quantile of chi^2 with 5 degrees of freedom


def test_philox_sample_inverse_cdf_brute_force(orc):
    """The chosen token is the first i with cdf_i > u * total, cdf and total
    in exact float64 arithmetic, whenever u * total is not within rounding
    of a cdf boundary."""
    import oracle
    rng = np.random.default_rng(16)
    T, V = 40, 30
    logits = rng.normal(0, 2, size=(T, V)).astype(np.float32)
    rid = rng.integers(0, 2 ** 40, size=T).astype(np.uint64)
    st = rng.integers(0, 1000, size=T).astype(np.uint64)
    ids = orc.philox_sample(logits, rid, st, 0.7)
    for t in range(T):
        p = np.exp((logits[t].astype(np.float64) - logits[t].max()) / 0.7)
        u = oracle.sample_uniform(oracle.sample_seed(int(rid[t]), int(st[t])))
        cdf = np.cumsum(p)
        target = u * cdf[-1]
        if np.min(np.abs(cdf - target)) < 1e-4 * cdf[-1]:
            continue
        assert ids[t] == int(np.argmax(cdf > target))


# ------------------------------------------------------- decoder stack --

def _tiny_weights(seed=0, layers=2):
    from deterministic_invariant_bf16_gb300 import synth
    import oracle
    w = synth.make_weights(synth.TINY, seed, "cpu", n_layers=layers)

    def np16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    out = dict(embed=np16(w["embed"]), final_norm=np16(w["final_norm"]),
               lm_head=np16(w["lm_head"]),
               layers=[{k: np16(v) for k, v in lw.items()}
                       for lw in w["layers"]])
    return out, oracle.Cfg(n_layers=layers)


def test_layer_is_identity_without_output_projections(orc):
    """Zero Wo and Wd make both residual branches vanish exactly."""
    w, cfg = _tiny_weights()
    lw = dict(w["layers"][0])
    lw["wo"] = np.zeros_like(lw["wo"])
    lw["wd"] = np.zeros_like(lw["wd"])
    rng = np.random.default_rng(17)
    h = orc.bf16r(rng.normal(size=(5, cfg.hidden)).astype(np.float32))
    kc, vc = orc.new_caches(cfg, 1, 8)[0]
    out = orc.decoder_layer(h, np.zeros(5, np.int32),
                            np.arange(5, dtype=np.int32), lw, kc, vc, cfg)
    assert np.array_equal(out, h)


def test_layer_branch_is_scale_free(orc):
    """Pre-norm placement: scaling the input by 4 (exact) leaves the residual
    branch's output unchanged when eps scales by 16."""
    w, cfg = _tiny_weights()
    rng = np.random.default_rng(18)
    h = orc.bf16r(rng.normal(size=(4, cfg.hidden)).astype(np.float32))
    req = np.zeros(4, np.int32)
    pos = np.arange(4, dtype=np.int32)
    lw = dict(w["layers"][0])
    lw["wd"] = np.zeros_like(lw["wd"])
    import dataclasses
    cfg4 = dataclasses.replace(cfg, eps=cfg.eps * 16)
    kc, vc = orc.new_caches(cfg, 1, 8)[0]
    a = orc.decoder_layer(h, req, pos, lw, kc, vc, cfg) - h
    kc, vc = orc.new_caches(cfg, 1, 8)[0]
    b = orc.decoder_layer(h * 4, req, pos, lw, kc, vc, cfg4) - h * 4
    # the branch output is the same up to one bf16 rounding of h + branch
    assert np.allclose(a, b, atol=4 * 2 ** -8 * np.abs(h * 4).max())


def test_causality_and_incremental_decode(orc):
    """Logits at position p ignore later tokens, and a prompt processed in
    one call equals the same prompt fed one token per call."""
    w, cfg = _tiny_weights()
    rng = np.random.default_rng(19)
    ids = rng.integers(0, cfg.vocab, size=10)
    caches = orc.new_caches(cfg, 1, 16)
    full = orc.model_forward(ids, np.zeros(10, np.int32),
                             np.arange(10, dtype=np.int32), w, caches, cfg)
    ids2 = ids.copy()
    ids2[6:] = (ids2[6:] + 1) % cfg.vocab
    caches = orc.new_caches(cfg, 1, 16)
    other = orc.model_forward(ids2, np.zeros(10, np.int32),
                              np.arange(10, dtype=np.int32), w, caches, cfg)
    assert np.array_equal(full[:6], other[:6])
    assert not np.array_equal(full[6:], other[6:])
    caches = orc.new_caches(cfg, 1, 16)
    for p in range(10):
        step = orc.model_forward(ids[p:p + 1], np.zeros(1, np.int32),
                                 np.array([p], np.int32), w, caches, cfg)
        assert np.array_equal(step[0], full[p])


# ------------------------------------- decoder composition, float64 --
#
# The pre-norm Llama block (RMSNorm -> QKV -> RoPE -> causal GQA attention ->
# O projection + residual -> RMSNorm of the post-attention residual -> SwiGLU
# FFN + residual) and the model head (untied embedding gather, final RMSNorm,
# LM head) are the reading the oracle takes of the operators the pages name
# (LLM-42 summary, 核心方法: GEMM, attention and normalisation kernels;
# ybb.press section 1: residual and normalisation).  Below they are written a
# second time, independently of ``oracle/``, in float64 numpy with bf16
# rounding (torch's CPU conversion) at the same storage points, plus a closed
# form whose FFN branch is a known function of its normed input.


def _bf(x):
    """float64 -> bf16 -> float64 through torch's CPU conversions."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float64)).to(torch.float32)
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def _w64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()


def _f64_norm(x, w, eps):
    return x / np.sqrt((x * x).mean(axis=1, keepdims=True) + eps) * w


def _f64_block(h, pos, lw, cfg):
    """One block for the rows of ONE request at positions ``pos`` (its
    cache empty before the call), float64 arithmetic."""
    W = {k: _w64(v) for k, v in lw.items()}
    T = h.shape[0]
    Hq, Hkv, D = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    x = _bf(_f64_norm(h, W["attn_norm"], cfg.eps))
    qkv = _bf(x @ W["wqkv"].T)
    q = qkv[:, :Hq * D].reshape(T, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D)
    v = qkv[:, (Hq + Hkv) * D:].reshape(T, Hkv, D)
    half = D // 2
    ang = np.asarray(pos, np.float64)[:, None] * cfg.theta ** (
        -2.0 * np.arange(half) / D)[None, :]
    rot = np.exp(1j * ang)[:, None, :]

    def rope(t):
        z = (t[..., :half] + 1j * t[..., half:]) * rot
        return np.concatenate([z.real, z.imag], axis=-1)

    q, k = _bf(rope(q)), _bf(rope(k))
    out = np.zeros((T, Hq, D))
    for t in range(T):
        vis = np.asarray(pos) <= pos[t]
        for hh in range(Hq):
            g = hh // (Hq // Hkv)
            s = k[vis, g] @ q[t, hh] / math.sqrt(D)
            p = np.exp(s - s.max())
            out[t, hh] = (p / p.sum()) @ v[vis, g]
    h = _bf(h + _bf(out.reshape(T, Hq * D)) @ W["wo"].T)
    x2 = _bf(_f64_norm(h, W["ffn_norm"], cfg.eps))
    g, u = x2 @ W["wg"].T, x2 @ W["wu"].T
    f = _bf(g / (1.0 + np.exp(-g)) * u)
    return _bf(h + f @ W["wd"].T)


def _relerr(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b)
                 / np.linalg.norm(b))


def test_decoder_layer_float64_brute_force(orc):
    """The oracle's block against the float64 restatement: the whole output
    and the residual branch alone (output minus input) agree norm-wise to
    well within what one bf16 rounding step per storage point allows.  A
    block that normalises the layer input instead of the post-attention
    residual for the FFN misses the branch by tens of percent."""
    w, cfg = _tiny_weights()
    rng = np.random.default_rng(31)
    T = 12
    h = orc.bf16r(rng.normal(0, 0.5, size=(T, cfg.hidden)).astype(np.float32))
    pos = np.arange(T, dtype=np.int32)
    for lw in w["layers"]:
        kc, vc = orc.new_caches(cfg, 1, 16)[0]
        got = orc.decoder_layer(h, np.zeros(T, np.int32), pos, lw, kc, vc,
                                cfg)
        ref = _f64_block(h.astype(np.float64), pos, lw, cfg)
        assert _relerr(got, ref) < 2e-3
        assert _relerr(got - h, ref - h) < 1e-2


def test_model_forward_float64_brute_force(orc):
    """Embedding gather, two blocks, final RMSNorm and LM head against the
    float64 restatement: logits within 1e-2 norm-wise, the per-layer hidden
    states within 2e-3.  Dropping the final norm scales the logits by the
    reciprocal RMS of the last hidden state (about 4x here)."""
    w, cfg = _tiny_weights()
    rng = np.random.default_rng(32)
    T = 10
    ids = rng.integers(0, cfg.vocab, size=T)
    pos = np.arange(T, dtype=np.int32)
    hidden = []
    got = orc.model_forward(ids, np.zeros(T, np.int32), pos, w,
                            orc.new_caches(cfg, 1, 16), cfg,
                            hidden_out=hidden)
    h = _w64(w["embed"])[ids]
    assert np.array_equal(hidden[0].astype(np.float64), h)
    for li, lw in enumerate(w["layers"]):
        h = _f64_block(h, pos, lw, cfg)
        assert _relerr(hidden[li + 1], h) < 2e-3
    x = _bf(_f64_norm(h, _w64(w["final_norm"]), cfg.eps))
    ref = x @ _w64(w["lm_head"]).T
    assert _relerr(got, ref) < 1e-2


def test_decoder_layer_ffn_closed_form(orc):
    """A block whose weights make every step a known function, one row at
    position 0 (attention over one key returns that key's value exactly):
      * V rows of wqkv = a permutation P, wo = identity, so the
        post-attention residual is h2 = bf16(h + P n(h)), n = RMSNorm;
      * gate rows (x, -x), up rows (x/4, x/4) and wd = [I I], so the FFN
        returns, per feature, silu(x) x/4 + silu(-x) x/4 = x^2 tanh(x/2) / 4
        of its normed input x = n(h2).
    The block output is therefore bf16(h2 + n(h2)^2 tanh(n(h2)/2) / 4).  The
    FFN reading n(h) instead of n(h2), swapped gate and up (x^2 tanh(x/8)/4),
    V taken from the K rows, or a dropped residual each miss it by far more
    than the bf16 rounding of the intermediate values."""
    cfg = orc.Cfg(n_layers=1)
    H, F = cfg.hidden, cfg.ffn
    assert F == 2 * H and cfg.q_dim == H and cfg.kv_dim == H

    def bits(a):
        t = torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)

    rng = np.random.default_rng(33)
    perm = rng.permutation(H)
    P = np.eye(H)[perm]
    eye = np.eye(H)
    wqkv = np.concatenate([rng.normal(0, 0.02, size=(2 * H, H)), P])
    lw = dict(attn_norm=bits(np.ones(H)), wqkv=bits(wqkv), wo=bits(eye),
              ffn_norm=bits(np.ones(H)), wg=bits(np.concatenate([eye, -eye])),
              wu=bits(np.concatenate([eye, eye]) / 4),
              wd=bits(np.concatenate([eye, eye], axis=1)))
    h = orc.bf16r(rng.normal(0, 1.0, size=(1, H)).astype(np.float32))
    kc, vc = orc.new_caches(cfg, 1, 4)[0]
    got = orc.decoder_layer(h, np.zeros(1, np.int32), np.zeros(1, np.int32),
                            lw, kc, vc, cfg).astype(np.float64)

    def n(x):
        return x / np.sqrt((x * x).mean() + cfg.eps)

    h64 = h.astype(np.float64)
    h2 = _bf(h64 + _bf(n(h64))[:, perm])
    x = n(h2)
    want = h2 + x * x * np.tanh(x / 2) / 4
    # every intermediate is rounded to bf16 once or twice: a few bf16 ulps
    # of the output's magnitude
    tol = 8 * 2.0 ** -8 * np.abs(want).max()
    assert np.abs(got - want).max() < tol
    xn = n(h64)
    for wrong in (h2 + xn * xn * np.tanh(xn / 2) / 4,
                  h2 + x * x * np.tanh(x / 8) / 4,
                  x * x * np.tanh(x / 2) / 4):
        assert np.abs(wrong - want).max() > 4 * tol


def test_model_head_closed_form(orc):
    """A model with no blocks: logits = LM head . bf16(RMSNorm(E[id])).  With
    LM-head row v the unit vector e_(v mod H) times 2^(v // H), logit v is
    2^(v // H) times feature v mod H of the normed embedding row, exactly
    (one nonzero product per sum)."""
    cfg = orc.Cfg(n_layers=0)
    H, V = cfg.hidden, cfg.vocab
    rng = np.random.default_rng(34)
    embed = rand_bf16_bits(rng, (V, H), std=0.02)
    head = np.zeros((V, H), np.float32)
    head[np.arange(V), np.arange(V) % H] = 2.0 ** (np.arange(V) // H)
    t = torch.from_numpy(head).to(torch.bfloat16)
    w = dict(embed=embed, layers=[], final_norm=_bits_ones(H),
             lm_head=t.view(torch.int16).numpy().view(np.uint16))
    ids = rng.integers(0, V, size=6)
    got = orc.model_forward(ids, np.zeros(6, np.int32),
                            np.arange(6, dtype=np.int32), w, [], cfg)
    e = _w64(embed)[ids]
    x = _bf(e / np.sqrt((e * e).mean(axis=1, keepdims=True) + cfg.eps))
    want = x[:, np.arange(V) % H] * 2.0 ** (np.arange(V) // H)
    # x is bf16 on both sides; the normalisation itself differs by at most
    # one bf16 rounding step
    assert np.abs(got - want).max() <= 2.0 ** -7 * np.abs(want).max()
    assert np.array_equal(np.sign(got), np.sign(want))


def _bits_ones(n):
    t = torch.ones(n, dtype=torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_greedy_tokens_identical_at_batch_1_and_32(orc):
    """ybb.press section 8, item 1: batch=1 and batch=32 outputs must be
    token-identical."""
    w, cfg = _tiny_weights(layers=1)
    rng = np.random.default_rng(20)
    prompts = [list(rng.integers(0, cfg.vocab, size=int(n)))
               for n in rng.integers(3, 9, size=32)]
    a = orc.greedy_decode(prompts, 4, w, cfg, batch=1)
    b = orc.greedy_decode(prompts, 4, w, cfg, batch=32)
    assert a == b


# --------------------------------------------------- commit / rollback --

def test_commit_rule_brute_force():
    """Every candidate/verified pair over a 2-letter alphabet for w <= 5:
    the commit length is the longest common prefix, computed another way."""
    import itertools
    import oracle
    for w in range(1, 6):
        for cand in itertools.product((3, 4), repeat=w):
            for ver in itertools.product((3, 4), repeat=w):
                eq = np.cumprod(np.array(cand) == np.array(ver))
                lcp = int(eq.sum())
                j, new_len, fix, keep = oracle.commit_rule(37, cand, ver)
                assert 0 <= j <= w and j == lcp
                assert new_len == 37 + lcp
                assert fix == (ver[lcp] if lcp < w else -1)
                assert keep == math.ceil((37 + lcp) / 16)


def test_commit_equals_first_perturbed_index(orc):
    """Candidates produced by the oracle's own greedy decode with one token
    perturbed: the verify recomputation commits exactly up to it, and the
    fix token is the unperturbed one."""
    w, cfg = _tiny_weights(layers=1)
    rng = np.random.default_rng(21)
    prompt = list(rng.integers(0, cfg.vocab, size=7))
    gen = orc.greedy_decode([prompt], 12, w, cfg)[0]
    for k in (0, 3, 11):
        cand = list(gen)
        cand[k] = (cand[k] + 5) % cfg.vocab
        n_cached = len(prompt) - 1     # committed prompt; its last token pending
        toks, pos = orc.verify_rows(n_cached, prompt[-1], cand)
        caches = orc.new_caches(cfg, 1, 32)
        orc.model_forward(prompt[:-1], np.zeros(n_cached, np.int32),
                          np.arange(n_cached, dtype=np.int32), w, caches, cfg)
        logits = orc.model_forward(toks, np.zeros(len(toks), np.int32),
                                   np.array(pos, np.int32), w, caches, cfg)
        ver = orc.argmax(logits)
        j, new_len, fix, keep = orc.commit_rule(n_cached, cand, ver)
        assert j == k and fix == gen[k] and new_len == n_cached + k


def test_pack_fifo():
    import oracle
    n, starts = oracle.pack_fifo([64, 64, 64, 64, 16])
    assert n == 4 and starts == [0, 64, 128, 192]
    n, starts = oracle.pack_fifo([16] * 20)
    assert n == 16 and starts[-1] == 240
    n, starts = oracle.pack_fifo([40, 50, 60, 70, 80])
    assert n == 4 and sum([40, 50, 60, 70]) <= 256


# ------------------------------------------------- top-k / top-p sampling --

def _rank_order(row):
    """Rank order of a row: larger value first, ties to the lower index,
    NaN as -inf (numpy's stable sort on the negated values)."""
    v = np.where(np.isnan(row), -np.inf, row.astype(np.float64))
    return np.argsort(-v, kind="stable")


def test_sample_top_reductions(orc):
    """top_k = 1 and a nucleus smaller than the largest token's mass are
    greedy; temperature 0 is argmax; K > V keeps every token."""
    rng = np.random.default_rng(31)
    x = rng.normal(size=(40, 300)).astype(np.float32)
    rid = np.arange(40, dtype=np.uint64) * 11
    st = np.arange(40, dtype=np.uint64)
    am = np.argmax(x, 1)
    assert np.array_equal(orc.philox_sample_top(x, rid, st, 0.9, 1, 1.0), am)
    assert np.array_equal(orc.philox_sample_top(x, rid, st, 0.9, 50, 1e-6), am)
    assert np.array_equal(orc.philox_sample_top(x, rid, st, 0.0, 50, 0.5), am)
    # K >= V with top_p = 1: the token's rank-order CDF interval holds u*Z
    ids = orc.philox_sample_top(x[:, :20], rid, st, 1.0, 1000, 1.0)
    assert ids.min() >= 0 and ids.max() < 20


def test_sample_top_ties_and_nan(orc):
    """Equal logits at the cut keep the lower indices; NaN ranks last and
    is never drawn."""
    n = 2000
    row = np.array([1.0, 3.0, 3.0, 3.0, 0.0, np.nan], np.float32)
    lg = np.tile(row, (n, 1))
    rid = np.full(n, 5, np.uint64)
    st = np.arange(n, dtype=np.uint64)
    ids = orc.philox_sample_top(lg, rid, st, 1.0, 2, 1.0)
    assert set(np.unique(ids)) == {1, 2}
    ids = orc.philox_sample_top(lg, rid, st, 1.0, 3, 1.0)
    assert set(np.unique(ids)) == {1, 2, 3}
    ids = orc.philox_sample_top(lg, rid, st, 1.0, 6, 1.0)
    assert 5 not in set(np.unique(ids)) and {0, 4} <= set(np.unique(ids))


def test_sample_top_frequencies(orc):
    """Over many steps the draws follow the kept tokens' renormalised
    probabilities (chi^2 at the 99.9% quantile)."""
    p = np.array([0.05, 0.1, 0.15, 0.2, 0.2, 0.3])
    row = np.log(p).astype(np.float32)
    n = 6000
    lg = np.tile(row, (n, 1))
    rid = np.full(n, 9, np.uint64)
    st = np.arange(n, dtype=np.uint64)
    for k, top_p, kept, q99 in [(4, 1.0, [5, 3, 4, 2], 16.27),
                                (6, 0.6, [5, 3, 4], 13.82)]:
        ids = orc.philox_sample_top(lg, rid, st, 1.0, k, top_p)
        assert set(np.unique(ids)) <= set(kept)
        counts = np.bincount(ids, minlength=6)[kept]
        exp = p[kept] / p[kept].sum() * n
        assert ((counts - exp) ** 2 / exp).sum() < q99


def test_sample_top_within_error_bound(orc):
    """Against float64: the drawn token lies in the top-k set, inside the
    nucleus, and its rank-order CDF interval holds u * Z up to fp32
    rounding of the sums."""
    import oracle
    rng = np.random.default_rng(32)
    T, V, tau = 300, 400, 0.7
    x = (rng.normal(size=(T, V)) * 2).astype(np.float32)
    rid = np.arange(T, dtype=np.uint64) * 7 + 1
    st = np.arange(T, dtype=np.uint64) % 13
    for k, top_p in [(100, 0.8), (400, 0.95), (17, 1.0)]:
        ids = orc.philox_sample_top(x, rid, st, tau, k, top_p)
        near = 0
        for t in range(T):
            order = _rank_order(x[t])[:k]
            j = int(np.nonzero(order == ids[t])[0][0])
            pv = np.exp((x[t][order].astype(np.float64) - x[t][order[0]]) / tau)
            c = np.cumsum(pv)
            n = int(np.nonzero(c >= top_p * c[-1] * (1 - 1e-6))[0][0])
            assert j <= n + 1
            u = oracle.sample_uniform(oracle.sample_seed(int(rid[t]),
                                                          int(st[t])))
            target = u * c[n]
            lo = c[j - 1] if j > 0 else 0.0
            tol = 1e-5 * c[-1]
            assert lo <= target + tol and c[j] >= target - tol, (t, j)
            cut_near = top_p < 1 and (
                abs(c[n] - top_p * c[-1]) < tol or
                (n > 0 and abs(c[n - 1] - top_p * c[-1]) < tol))
            if j > n or abs(lo - target) < tol or cut_near:
                near += 1
        assert near <= T // 50
