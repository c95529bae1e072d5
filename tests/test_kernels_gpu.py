"""Per-kernel GPU tests through the C ABI: RMSNorm with the fused
split-reduction and residual, RoPE + paged KV append, decode and prefill
attention over permuted pages, argmax and Philox sampling.  Each kernel is
checked against the oracle and bitwise against itself across batch
composition, row position, query length and page layout (Vosti abstract;
ybb.press section 4)."""
import math

import numpy as np
import pytest
import torch

from helpers import bits, from_bits, norm_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    from deterministic_invariant_bf16_gb300 import binding, build
    build.build()
    binding.lib()
    return binding


def randn_bf16(shape, seed, std=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(
        torch.bfloat16)


def sync_ok(bi):
    torch.cuda.synchronize()
    assert bi.bi_device_status() == 0


def ulp_diff(a_bits, b_bits):
    return np.abs(a_bits.astype(np.int32) - b_bits.astype(np.int32))


# ------------------------------------------------------------- RMSNorm --

@pytest.mark.parametrize("H", [128, 4096])
def test_rmsnorm_fused_reduce_residual(bi, orc, H):
    T, S = 37, 3
    g = torch.Generator(device="cuda").manual_seed(H)
    parts = torch.randn(S, T, H, generator=g, device="cuda") * 0.3
    h0 = randn_bf16((T, H), 2)
    w = randn_bf16((H,), 3)
    res = h0.clone()
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    bi.bi_rmsnorm(parts, S, None, res, w, T, H, 1e-5, y)
    sync_ok(bi)
    p = parts.cpu().numpy()
    v = (p[0] + p[1]) + p[2]                         # slice order 0, 1, 2
    ref_res = orc.bf16_bits(orc.bf16_value(bits(h0)) + v)
    assert np.array_equal(bits(res), ref_res)       # same fp32 operations
    ref_y = orc.bf16_bits(orc.rmsnorm(orc.bf16_value(ref_res), bits(w), 1e-5))
    d = ulp_diff(bits(y), ref_y)
    assert d.max() <= 1 and (d == 0).mean() > 0.98
    # row invariance: each row alone gives the same bits
    for t in (0, 19, 36):
        r1 = h0[t:t + 1].clone()
        y1 = torch.empty(1, H, dtype=torch.bfloat16, device="cuda")
        p1 = parts[:, t:t + 1].contiguous()
        bi.bi_rmsnorm(p1, S, None, r1, w, 1, H, 1e-5, y1)
        sync_ok(bi)
        assert np.array_equal(bits(y1)[0], bits(y)[t])
        assert np.array_equal(bits(r1)[0], bits(res)[t])
    # plain input (no partials, no residual)
    y2 = torch.empty_like(y)
    bi.bi_rmsnorm(None, 0, h0, None, w, T, H, 1e-5, y2)
    sync_ok(bi)
    ref2 = orc.bf16_bits(orc.rmsnorm(orc.bf16_value(bits(h0)), bits(w), 1e-5))
    assert ulp_diff(bits(y2), ref2).max() <= 1


# ---------------------------------------------------------- RoPE + KV --

def test_rope_and_paged_append(bi, orc):
    T, Hq, Hkv, D, S, theta = 21, 8, 2, 128, 2, 5e5
    QKV = (Hq + 2 * Hkv) * D
    g = torch.Generator(device="cuda").manual_seed(7)
    parts = torch.randn(S, T, QKV, generator=g, device="cuda")
    rng = np.random.default_rng(8)
    pos = rng.integers(0, 3000, size=T).astype(np.int32)
    slots = rng.integers(0, 4, size=T).astype(np.int32)
    slots[3] = -1                                   # a pad row
    max_pages, n_pages = 200, 900
    table = rng.permutation(n_pages)[:4 * max_pages].reshape(4, max_pages)
    table = table.astype(np.int32)
    kp = torch.zeros(n_pages, Hkv, 16, D, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    q = torch.empty(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    bi.bi_rope(parts, S, torch.from_numpy(pos).cuda(),
               torch.from_numpy(slots).cuda(), Hq, Hkv, D, theta, q, kp, vp,
               torch.from_numpy(table).cuda())
    sync_ok(bi)
    p = parts.cpu().numpy()
    qkv = orc.bf16r(p[0] + p[1])
    rq = orc.bf16_bits(orc.rope(qkv[:, :Hq * D].reshape(T, Hq, D), pos, theta))
    rk = orc.bf16_bits(orc.rope(qkv[:, Hq * D:(Hq + Hkv) * D].reshape(
        T, Hkv, D), pos, theta))
    rv = orc.bf16_bits(qkv[:, (Hq + Hkv) * D:].reshape(T, Hkv, D))
    live = slots >= 0
    assert ulp_diff(bits(q)[live], rq[live]).max() <= 1
    assert np.all(bits(q)[~live] == 0)
    kb, vb = bits(kp), bits(vp)
    for t in np.nonzero(live)[0]:
        pg = table[slots[t], pos[t] // 16]
        assert ulp_diff(kb[pg, :, pos[t] % 16], rk[t]).max() <= 1
        assert np.array_equal(vb[pg, :, pos[t] % 16], rv[t])


# ----------------------------------------------------------- attention --

class PagedKV:
    """Random KV contents for R requests, stored in a NaN-filled pool under
    a random page order; the logical caches are kept for the oracle."""

    def __init__(self, lens, Hkv, D, seed, n_pages=None, nan_fill=True):
        rng = np.random.default_rng(seed)
        self.lens = np.asarray(lens)
        self.Hkv, self.D = Hkv, D
        L = int(self.lens.max())
        R = len(lens)
        self.k = orc_bf16(rng.normal(size=(R, L, Hkv, D)))
        self.v = orc_bf16(rng.normal(size=(R, L, Hkv, D)))
        self.max_pages = -(-L // 16) + 1
        need = int(sum(-(-n // 16) for n in lens))
        self.n_pages = n_pages or need + 7
        self.place(rng.permutation(self.n_pages), nan_fill)

    def place(self, perm, nan_fill=True):
        R = len(self.lens)
        table = np.full((R, self.max_pages), -1, np.int32)
        fill = 0x7fc0 if nan_fill else 0
        kp = np.full((self.n_pages, self.Hkv, 16, self.D), fill, np.uint16)
        vp = kp.copy()
        at = 0
        for r, n in enumerate(self.lens):
            for pi in range(-(-n // 16)):
                pg = int(perm[at])
                at += 1
                table[r, pi] = pg
                lo, hi = pi * 16, min(n, pi * 16 + 16)
                kp[pg, :, :hi - lo] = self.k[r, lo:hi].transpose(1, 0, 2)
                vp[pg, :, :hi - lo] = self.v[r, lo:hi].transpose(1, 0, 2)
        self.table = torch.from_numpy(table).cuda()
        self.kp = from_bits(kp)
        self.vp = from_bits(vp)


def orc_bf16(x):
    import oracle
    return oracle.bf16_bits(np.asarray(x, np.float32))


def decode(bi, q, kv, rows, kv_len):
    B, Hq, D = q.shape
    max_kv = int(max(kv_len))
    ws = torch.empty(bi.bi_decode_attn_workspace_size(B, Hq, D, max_kv) // 4,
                     dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    bi.bi_paged_decode_attn(q, kv.kp, kv.vp, kv.table,
                            torch.tensor(rows, dtype=torch.int32).cuda(),
                            torch.tensor(kv_len, dtype=torch.int32).cuda(),
                            max_kv, 1 / math.sqrt(D), out, ws)
    return out


def prefill(bi, q, kv, segs, ws=False, scale=None, split=False):
    """segs: list of (request, first position, n rows); q rows in order.
    ws: run bi_prefill_attn_ws with a workspace (the persistent path);
    split: with the workspace of the split form (verify-sized batches)."""
    cu, sr, pos = [0], [], []
    for r, p0, n in segs:
        cu.append(cu[-1] + n)
        sr.append(r)
        pos += list(range(p0, p0 + n))
    out = torch.empty_like(q)
    args = (q, torch.tensor(cu, dtype=torch.int32).cuda(),
            torch.tensor(sr, dtype=torch.int32).cuda(),
            torch.tensor(pos, dtype=torch.int32).cuda(),
            max(n for _, _, n in segs), max(pos) + 1, kv.kp, kv.vp, kv.table,
            1 / math.sqrt(q.shape[2]) if scale is None else scale, out)
    if ws:
        T, Hq = q.shape[0], q.shape[1]
        nb = bi.bi_prefill_attn_workspace_size(T, len(segs), Hq,
                                               kv.kp.shape[1])
        if split:
            nb = bi.bi_prefill_attn_split_workspace_size(
                T, len(segs), Hq, kv.kp.shape[1], max(pos) + 1)
            assert nb > 0
        w = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
        bi.bi_prefill_attn_ws(*args, w)
    else:
        bi.bi_prefill_attn(*args)
    return out, pos


def attn_ref(orc, q, kv, rows, positions):
    D = q.shape[2]
    return orc.attention(orc.bf16_value(bits(q)), orc.bf16_value(kv.k),
                         orc.bf16_value(kv.v), np.asarray(rows, np.int32),
                         np.asarray(positions, np.int32),
                         np.float32(1 / math.sqrt(D)))


def check_close(got_bits, ref, orc):
    got = orc.bf16_value(got_bits).astype(np.float64)
    T, H, D = ref.shape
    for t in range(T):
        for h in range(H):
            assert norm_rel_err(got[t, h], ref[t, h]) < 1e-2, (t, h)
    assert np.abs(got - ref).max() < 2e-2


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (4, 4, 32)])
def test_decode_attention(bi, orc, Hq, Hkv, D):
    lens = [1, 15, 16, 17, 255, 256, 257, 700, 1500, 40]
    kv = PagedKV(lens, Hkv, D, seed=31)
    q = randn_bf16((len(lens), Hq, D), 32)
    rows = list(range(len(lens)))
    out = decode(bi, q, kv, rows, lens)
    sync_ok(bi)
    ref = attn_ref(orc, q, kv, rows, np.array(lens) - 1)
    check_close(bits(out), ref, orc)
    full = bits(out)
    # each request alone, and the batch in reverse order: same bits
    for b in (0, 6, 8):
        one = decode(bi, q[b:b + 1].contiguous(), kv, [b], [lens[b]])
        sync_ok(bi)
        assert np.array_equal(bits(one)[0], full[b])
    rev = decode(bi, q.flip(0).contiguous(), kv, rows[::-1], lens[::-1])
    sync_ok(bi)
    assert np.array_equal(bits(rev)[::-1], full)
    # another physical page order: same bits
    kv.place(np.random.default_rng(99).permutation(kv.n_pages))
    again = decode(bi, q, kv, rows, lens)
    sync_ok(bi)
    assert np.array_equal(bits(again), full)


@pytest.mark.parametrize("D", [128, 32])
def test_decode_work_list_over_many_rows(bi, orc, D):
    """More rows than the work-list builder has threads (two batches of
    1024), a mix of full and partial chunks: sampled rows against the oracle,
    and the whole batch bitwise equal after a shuffle of its rows (which
    reorders the work list and so changes the CTA that computes each
    chunk)."""
    rng = np.random.default_rng(7)
    lens = rng.integers(1, 200, 1100)
    lens[::97] = 256
    lens[5::89] = 16
    lens[11::101] = 300
    kv = PagedKV(lens, 1, D, seed=71)
    B = len(lens)
    q = randn_bf16((B, 4, D), 72)
    rows = list(range(B))
    out = decode(bi, q, kv, rows, lens)
    sync_ok(bi)
    full = bits(out)
    pick = np.sort(rng.choice(B, 24, replace=False))
    ref = attn_ref(orc, q[torch.from_numpy(pick).cuda()], kv, pick,
                   lens[pick] - 1)
    check_close(full[pick], ref, orc)
    perm = rng.permutation(B)
    shuf = decode(bi, q[torch.from_numpy(perm).cuda()].contiguous(), kv,
                  list(perm), lens[perm])
    sync_ok(bi)
    assert np.array_equal(bits(shuf), full[perm])


def test_decode_whole_rows_match_chunk_items(bi, orc):
    """Batches with at least 8 (row, KV head) items per SM run whole-row
    items merged in registers; smaller ones run (row, chunk) items and a
    separate merge.  Both must give the same bits for a row: a batch of 200
    rows (1600 items) against 40-row sub-batches of it (320 items)."""
    rng = np.random.default_rng(17)
    lens = rng.integers(1, 520, 200)
    lens[::13] = 256
    lens[3::17] = 512
    kv = PagedKV(lens, 8, 128, seed=19)
    q = randn_bf16((200, 32, 128), 20)
    full = bits(decode(bi, q, kv, list(range(200)), lens))
    sync_ok(bi)
    for lo in range(0, 200, 40):
        part = decode(bi, q[lo:lo + 40].contiguous(), kv,
                      list(range(lo, lo + 40)), lens[lo:lo + 40])
        sync_ok(bi)
        assert np.array_equal(bits(part), full[lo:lo + 40])
    pick = np.sort(rng.choice(200, 6, replace=False))
    ref = attn_ref(orc, q[torch.from_numpy(pick).cuda()], kv, pick,
                   lens[pick] - 1)
    check_close(full[pick], ref, orc)


def test_decode_long_contexts_both_forms(bi, orc):
    """Contexts of the long-prompt stress (4100 to 8600 positions: 17 to 34
    chunks merged in order).  A batch of 160 rows (whole-row items, chunks
    merged in registers) holding four long rows among short ones, and each
    long row alone (per-chunk items and the record merge kernel), give the
    same bits; the long rows are within tolerance of the oracle."""
    import types
    long_lens = np.array([4100, 6000, 8192, 8600])
    rng = np.random.default_rng(23)
    short_lens = rng.integers(1, 64, 156)
    A = PagedKV(long_lens, 8, 128, seed=29)
    B = PagedKV(short_lens, 8, 128, seed=31)
    long_rows = [3, 50, 101, 157]
    R = 160
    lens = np.empty(R, np.int64)
    table = np.full((R, A.max_pages), -1, np.int32)
    ta, tb = A.table.cpu().numpy(), B.table.cpu().numpy()
    si = 0
    for r in range(R):
        if r in long_rows:
            j = long_rows.index(r)
            lens[r] = long_lens[j]
            table[r] = ta[j]
        else:
            lens[r] = short_lens[si]
            row = tb[si]
            table[r, :row.shape[0]] = np.where(row >= 0, row + A.n_pages, -1)
            si += 1
    kv = types.SimpleNamespace(kp=torch.cat([A.kp, B.kp]),
                               vp=torch.cat([A.vp, B.vp]),
                               table=torch.from_numpy(table).cuda())
    q = randn_bf16((R, 32, 128), 33)
    full = bits(decode(bi, q, kv, list(range(R)), lens))
    sync_ok(bi)
    # 160 rows x 8 KV heads reach the whole-row form's 8 items per SM
    assert R * 8 >= 8 * torch.cuda.get_device_properties(0).multi_processor_count
    for r in long_rows:
        one = decode(bi, q[r:r + 1].contiguous(), kv, [r], [int(lens[r])])
        sync_ok(bi)
        assert np.array_equal(bits(one)[0], full[r]), r
    ql = q[torch.tensor(long_rows).cuda()].contiguous()
    ref = attn_ref(orc, ql, A, [0, 1, 2, 3], long_lens - 1)
    check_close(full[long_rows], ref, orc)


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (4, 4, 32)])
def test_prefill_matches_decode_bitwise(bi, orc, Hq, Hkv, D):
    """Query-length invariance (Vosti): a position computed inside a window
    of many queries equals the same position decoded on its own."""
    lens = [300, 530, 64, 1030]
    kv = PagedKV(lens, Hkv, D, seed=41)
    segs = [(0, 250, 50), (1, 470, 60), (2, 0, 64), (3, 1000, 17),
            (3, 1017, 13)]
    T = sum(n for _, _, n in segs)
    q = randn_bf16((T, Hq, D), 42)
    out, pos = prefill(bi, q, kv, segs)
    sync_ok(bi)
    rows = sum([[r] * n for r, _, n in segs], [])
    ref = attn_ref(orc, q, kv, rows, pos)
    check_close(bits(out), ref, orc)
    dec = decode(bi, q, kv, rows, [p + 1 for p in pos])
    sync_ok(bi)
    assert np.array_equal(bits(dec), bits(out))
    # segments split differently (chunked prefill): same bits
    segs2 = [(0, 250, 7), (0, 257, 43), (1, 470, 60), (2, 0, 1), (2, 1, 63),
             (3, 1000, 30)]
    out2, pos2 = prefill(bi, q, kv, segs2)
    sync_ok(bi)
    assert pos2 == pos and np.array_equal(bits(out2), bits(out))
    # the persistent path (with a workspace), on both segmentations and with
    # a pad segment: same bits
    for sg in (segs, segs2):
        out3, pos3 = prefill(bi, q, kv, sg, ws=True)
        sync_ok(bi)
        assert pos3 == pos and np.array_equal(bits(out3), bits(out))
    pad = torch.zeros((T + 9, Hq, D), dtype=torch.bfloat16, device="cuda")
    pad[:T] = q
    out4, _ = prefill(bi, pad, kv, segs + [(-1, 0, 9)], ws=True)
    sync_ok(bi)
    assert np.array_equal(bits(out4)[:T], bits(out))
    assert not bits(out4)[T:].any()


def test_prefill_group_path_bitwise(bi, orc):
    """Prompt pieces longer than a verify batch (here 1358 rows) take the
    row-per-thread kernel over 128-row tiles (32 tokens x 4 heads) of a
    segment: its outputs equal, bit for bit, the one-CTA-per-16-row-tile
    prefill and decode of each row alone, over segments whose lengths are
    not multiples of the tile (partial tiles), two pieces of one request, a
    pad segment (zero outputs) and NaN-filled stale pages; sampled rows
    agree with the oracle."""
    Hq, Hkv, D = 32, 8, 128
    lens = [2100, 700, 1600]
    kv = PagedKV(lens, Hkv, D, seed=51)
    segs = [(0, 1300, 700), (1, 100, 533), (2, 1490, 10), (2, 1500, 100),
            (-1, 0, 15)]
    T = sum(n for _, _, n in segs)
    q = randn_bf16((T, Hq, D), 52)
    grp, pos = prefill(bi, q, kv, segs, ws=True)
    sync_ok(bi)
    real = T - 15
    assert not bits(grp)[real:].any()
    one, _ = prefill(bi, q[:real].contiguous(), kv, segs[:-1])
    sync_ok(bi)
    assert np.array_equal(bits(grp)[:real], bits(one))
    rows = sum([[r] * n for r, _, n in segs[:-1]], [])
    dec = decode(bi, q[:real].contiguous(), kv, rows,
                 [p + 1 for p in pos[:real]])
    sync_ok(bi)
    assert np.array_equal(bits(dec), bits(one))
    pick = [0, 31, 32, 699, 700, 1232, 1233, 1242, real - 1]
    ref = attn_ref(orc, q[pick].contiguous(), kv, [rows[i] for i in pick],
                   [pos[i] for i in pick])
    check_close(bits(grp)[pick], ref, orc)


def test_prefill_long_prompt_piece(bi, orc):
    """A 2048-row piece of a long prompt at positions 4096..6143 (the
    long-prompt stress's pieces: up to 24 chunks per row) on the row
    kernel equals decode of each row alone bit for bit on sampled rows, and
    those rows are within tolerance of the oracle."""
    Hq, Hkv, D = 32, 8, 128
    kv = PagedKV([6144], Hkv, D, seed=57)
    segs = [(0, 4096, 2048)]
    q = randn_bf16((2048, Hq, D), 58)
    grp, pos = prefill(bi, q, kv, segs, ws=True)
    sync_ok(bi)
    pick = [0, 1, 31, 32, 127, 128, 1000, 1023, 1024, 2046, 2047]
    dec = decode(bi, q[pick].contiguous(), kv, [0] * len(pick),
                 [pos[i] + 1 for i in pick])
    sync_ok(bi)
    assert np.array_equal(bits(dec), bits(grp)[pick])
    ref = attn_ref(orc, q[pick].contiguous(), kv, [0] * len(pick),
                   [pos[i] for i in pick])
    check_close(bits(grp)[pick], ref, orc)


@pytest.mark.parametrize("Hq,Hkv,scale", [(16, 2, None), (8, 8, None),
                                          (32, 2, None), (16, 8, None),
                                          (8, 2, -0.06)])
def test_prefill_row_tiles_other_groupings(bi, Hq, Hkv, scale):
    """The 128-row tiles hold 128 / G tokens (G = Hq / Hkv query heads per
    KV head: 16, 128, 8 and 64 tokens here); each grouping, and a negative
    scale (the maximum is then taken on the scaled scores), gives the bits
    of the one-CTA-per-16-row-tile kernel."""
    D = 128
    lens = [1100, 900]
    kv = PagedKV(lens, Hkv, D, seed=61)
    segs = [(0, 300, 800), (1, 0, 900)]
    T = sum(n for _, _, n in segs)
    q = randn_bf16((T, Hq, D), 62)
    rows_, _ = prefill(bi, q, kv, segs, ws=True, scale=scale)
    sync_ok(bi)
    one, _ = prefill(bi, q, kv, segs, scale=scale)
    sync_ok(bi)
    assert np.array_equal(bits(rows_), bits(one))
    b = bits(rows_)
    assert not (((b & 0x7f80) == 0x7f80) & ((b & 0x7f) != 0)).any()


def test_prefill_split_form_bitwise(bi, orc):
    """A verify-sized batch (windows of 64, 32 and 16 tokens at contexts
    spanning one to nine 256-position chunks, a pad segment) with the
    workspace of the split form — one work item per (128-row tile, chunk,
    KV head), the chunk records merged in order by the decode merge — gives
    the bits of the in-kernel form, of one CTA per 16-row tile and of each
    row's decode, over NaN-filled stale pages; sampled rows agree with the
    oracle."""
    Hq, Hkv, D = 32, 8, 128
    lens = [2200, 300, 64, 900, 1500]
    kv = PagedKV(lens, Hkv, D, seed=71)
    segs = [(0, 2136, 64), (1, 268, 32), (2, 48, 16), (3, 836, 64),
            (4, 1468, 32), (-1, 0, 16)]
    T = sum(n for _, _, n in segs)
    q = randn_bf16((T, Hq, D), 72)
    spl, pos = prefill(bi, q, kv, segs, ws=True, split=True)
    sync_ok(bi)
    real = T - 16
    assert not bits(spl)[real:].any()
    ink, _ = prefill(bi, q, kv, segs, ws=True)
    sync_ok(bi)
    assert np.array_equal(bits(spl), bits(ink))
    one, _ = prefill(bi, q[:real].contiguous(), kv, segs[:-1])
    sync_ok(bi)
    assert np.array_equal(bits(spl)[:real], bits(one))
    rows = sum([[r] * n for r, _, n in segs[:-1]], [])
    dec = decode(bi, q[:real].contiguous(), kv, rows,
                 [p + 1 for p in pos[:real]])
    sync_ok(bi)
    assert np.array_equal(bits(dec), bits(spl)[:real])
    pick = [0, 63, 64, 95, 96, 111, 112, 175, real - 1]
    ref = attn_ref(orc, q[pick].contiguous(), kv, [rows[i] for i in pick],
                   [pos[i] for i in pick])
    check_close(bits(spl)[pick], ref, orc)


# -------------------------------------------------------------- argmax --

def test_argmax_exact(bi, orc):
    T, V = 40, 128256
    g = torch.Generator(device="cuda").manual_seed(51)
    x = torch.randn(T, V, generator=g, device="cuda")
    x[3, [100, 90000]] = 50.0          # tie: lower index
    x[4, 777] = float("nan")
    x[5, [10, 20]] = float("nan")      # first NaN
    x[6] = 0.0
    x[6, 0] = -0.0
    x[7] = float("-inf")
    x[8, -1] = float("inf")
    ids = torch.empty(T, dtype=torch.int32, device="cuda")
    bi.bi_argmax_logits(x, ids)
    sync_ok(bi)
    assert np.array_equal(ids.cpu().numpy(), orc.argmax(x.cpu().numpy()))
    # rows are independent of the batch they are in
    one = torch.empty(1, dtype=torch.int32, device="cuda")
    bi.bi_argmax_logits(x[17:18].contiguous(), one)
    sync_ok(bi)
    assert one.item() == ids[17].item()
    x2 = torch.randn(9, 513, generator=g, device="cuda")  # V % 4 != 0
    ids2 = torch.empty(9, dtype=torch.int32, device="cuda")
    bi.bi_argmax_logits(x2, ids2)
    sync_ok(bi)
    assert np.array_equal(ids2.cpu().numpy(), orc.argmax(x2.cpu().numpy()))


def test_argmax_short_rows_and_cross_part_ties(bi, orc):
    """A row is split into eight contiguous parts, one per CTA of a
    cluster: rows shorter than the cluster (some parts empty), lengths
    around multiples of 4 and 8, ties and NaNs in different parts, and an
    all -inf row all give the oracle's index."""
    g = torch.Generator(device="cuda").manual_seed(53)
    for V in (1, 2, 3, 4, 5, 7, 8, 9, 31, 32, 33, 4100):
        x = torch.randn(12, V, generator=g, device="cuda")
        x[1] = float("-inf")
        if V >= 2:
            x[2, [0, V - 1]] = 9.0                 # tie: first and last part
            x[3, V - 1] = float("nan")             # a NaN beats any value
            x[4, [V // 2, V - 1]] = float("nan")   # first NaN wins
            x[5] = 1.0                             # all equal: index 0
            x[6, V - 1] = float("inf")
            x[7, 0] = -0.0
            x[7, 1:] = 0.0                         # -0 == +0: index 0
        ids = torch.empty(12, dtype=torch.int32, device="cuda")
        bi.bi_argmax_logits(x, ids)
        sync_ok(bi)
        assert np.array_equal(ids.cpu().numpy(), orc.argmax(x.cpu().numpy())), V
    x = torch.randn(3, 128256, generator=g, device="cuda")
    x[0, [16031, 16032]] = 40.0      # tie across the first part boundary
    x[1, [5000, 120000]] = float("nan")
    x[2, [127000, 130]] = 40.0
    ids = torch.empty(3, dtype=torch.int32, device="cuda")
    bi.bi_argmax_logits(x, ids)
    sync_ok(bi)
    assert ids.cpu().tolist() == [16031, 5000, 130]
    assert np.array_equal(ids.cpu().numpy(), orc.argmax(x.cpu().numpy()))


# -------------------------------------------------------------- Philox --

def _top_boundary_ok(x, rid, st, tau, k, top_p, a, b):
    """Two draws of the same row may differ only where fp32 rounding (of
    exp or the running sums) moves u * Z or the nucleus cut across a
    boundary of the rank-order CDF."""
    import oracle
    v = np.where(np.isnan(x), -np.inf, x.astype(np.float64))
    order = np.argsort(-v, kind="stable")[:k]
    pv = np.exp((v[order] - v[order[0]]) / tau)
    c = np.cumsum(pv)
    cut = top_p * c[-1]
    u = oracle.sample_uniform(oracle.sample_seed(int(rid), int(st)))
    ja = int(np.nonzero(order == a)[0][0])
    jb = int(np.nonzero(order == b)[0][0])
    lo, hi = min(ja, jb), max(ja, jb)
    tol = 1e-4 * c[-1]
    n = int(np.nonzero(c >= cut * (1 - 1e-6))[0][0])
    near_cut = top_p < 1 and abs(c[min(hi, len(c) - 1)] - cut) < tol or \
        abs(c[lo] - cut) < tol
    return near_cut or abs(c[lo] - u * c[n]) < tol


def test_philox_sample_top_against_oracle(bi, orc):
    """Top-k / top-p sampling against the oracle: ids equal except on CDF or
    nucleus boundaries within fp32 rounding (at most 1% of rows); top_k = 1
    is argmax; heavy ties at the cut (the index-ordered path); V not a
    multiple of 4; K > V; the full 128256-token vocabulary at K = 1024 and
    50, and a long row of only six distinct values (ties at the cut on the
    index-ordered path); rows do not depend on the batch."""
    cases = [(1500, 1000, 50, 0.9, False), (1500, 1000, 1024, 0.95, False),
             (1500, 1000, 7, 1.0, False), (800, 1001, 64, 0.8, False),
             (600, 300, 1024, 1.0, False), (800, 512, 40, 0.9, True),
             (16, 128256, 1024, 0.9, False), (16, 128256, 50, 1.0, False),
             (6, 131072, 64, 0.9, True)]
    for ci, (T, V, k, top_p, ties) in enumerate(cases):
        g = torch.Generator(device="cuda").manual_seed(70 + ci)
        if ties:
            x = torch.randint(0, 6, (T, V), generator=g, device="cuda").float()
        else:
            x = torch.randn(T, V, generator=g, device="cuda") * 2
        rid = torch.arange(T, dtype=torch.int64, device="cuda") * 131 + ci
        st = torch.arange(T, dtype=torch.int64, device="cuda") % 29
        ids = torch.empty(T, dtype=torch.int32, device="cuda")
        tau = 0.8
        bi.philox_sample_top(x, rid, st, tau, k, top_p, ids)
        sync_ok(bi)
        got = ids.cpu().numpy()
        xl = x.cpu().numpy()
        rl, sl = rid.cpu().numpy().astype(np.uint64), st.cpu().numpy().astype(np.uint64)
        ref = orc.philox_sample_top(xl, rl, sl, tau, k, top_p)
        mism = np.nonzero(got != ref)[0]
        assert len(mism) <= max(1, T // 100), (ci, len(mism))
        for t in mism:
            assert _top_boundary_ok(xl[t], rl[t], sl[t], tau, min(k, V),
                                    top_p, got[t], ref[t]), (ci, t)
        if ci == 0:
            one = torch.empty(1, dtype=torch.int32, device="cuda")
            bi.philox_sample_top(x[9:10].contiguous(), rid[9:10].contiguous(),
                                 st[9:10].contiguous(), tau, k, top_p, one)
            sync_ok(bi)
            assert one.item() == got[9]
            bi.philox_sample_top(x, rid, st, tau, 1, 1.0, ids)
            sync_ok(bi)
            assert np.array_equal(ids.cpu().numpy(), orc.argmax(xl))
    x = torch.zeros(2, 64, device="cuda")
    ids = torch.empty(2, dtype=torch.int32, device="cuda")
    r = torch.zeros(2, dtype=torch.int64, device="cuda")
    with pytest.raises(bi.BiError, match="UNSUPPORTED"):
        bi.philox_sample_top(x, r, r, 1.0, 1025, 1.0, ids)
    with pytest.raises(bi.BiError, match="INVALID"):
        bi.philox_sample_top(x, r, r, 1.0, 8, 0.0, ids)


def test_philox_sample_against_oracle(bi, orc):
    import oracle
    T, V, tau = 3000, 512, 0.8
    g = torch.Generator(device="cuda").manual_seed(61)
    x = torch.randn(T, V, generator=g, device="cuda") * 2
    rid = torch.arange(T, dtype=torch.int64, device="cuda") * 7919 + 3
    step = torch.arange(T, dtype=torch.int64, device="cuda") % 37
    ids = torch.empty(T, dtype=torch.int32, device="cuda")
    bi.philox_sample(x, rid, step, tau, ids)
    sync_ok(bi)
    got = ids.cpu().numpy()
    xl = x.cpu().numpy()
    ref = orc.philox_sample(xl, rid.cpu().numpy().astype(np.uint64),
                            step.cpu().numpy().astype(np.uint64), tau)
    mism = np.nonzero(got != ref)[0]
    assert len(mism) <= T // 100
    # every disagreement sits on a CDF boundary within fp32 rounding
    for t in mism:
        p = np.exp((xl[t].astype(np.float64) - xl[t].max()) / tau)
        cdf = np.cumsum(p)
        u = oracle.sample_uniform(oracle.sample_seed(int(rid[t]),
                                                      int(step[t])))
        target = u * cdf[-1]
        k = min(got[t], ref[t])
        assert abs(cdf[k] - target) < 1e-4 * cdf[-1]
    # temperature 0 is greedy
    bi.philox_sample(x, rid, step, 0.0, ids)
    sync_ok(bi)
    assert np.array_equal(ids.cpu().numpy(), orc.argmax(xl))
    # rows are independent of the batch
    one = torch.empty(1, dtype=torch.int32, device="cuda")
    bi.philox_sample(x[5:6].contiguous(), rid[5:6].contiguous(),
                     step[5:6].contiguous(), tau, one)
    sync_ok(bi)
    assert one.item() == got[5]


def test_swiglu_standalone_against_oracle(bi, orc):
    """bi_swiglu (the standalone kernel; the model fuses the same formula
    into the gate/up GEMM): out = bf16(silu(g) u) with silu(g) = g / (1 +
    e^-g) in fp32, on a ragged length, against the oracle: at most one bf16
    ulp apart (the fp32 exponential and division of the two sides may round
    differently before the bf16 rounding), and bit-equal on almost every
    element; the limits silu(0) = 0, silu(large) = large, silu(-large) = -0
    hold exactly."""
    n = 1_000_003
    gen = torch.Generator(device="cuda").manual_seed(91)
    g = torch.randn(n, generator=gen, device="cuda") * 4
    u = torch.randn(n, generator=gen, device="cuda") * 2
    special = torch.tensor([0.0, -0.0, 1.0, -1.0, 30.0, -30.0, 88.0, -88.0,
                            100.0, -100.0], device="cuda")
    g[:10] = special
    u[:10] = 1.5
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    bi.bi_swiglu(g, u, out)
    sync_ok(bi)
    got = bits(out).astype(np.int32)
    ref = orc.bf16_bits(orc.swiglu(g.cpu().numpy(), u.cpu().numpy())).astype(
        np.int32)
    assert np.abs(got - ref).max() <= 1
    assert np.mean(got != ref) < 1e-3
    vals = orc.bf16_value(got[:10].astype(np.uint16))
    assert vals[0] == 0 and vals[4] == orc.bf16r(np.float32(45.0))
    assert vals[9] == 0


def test_philox_sample_full_vocabulary(bi, orc):
    """philox_sample at the LM head's 128256-token vocabulary, where each of
    a row's 1024 threads owns about 125 logits: the multi-element slice
    sums, the column-transposed slice reads and the skip of slices whose
    running sum cannot reach the target all run.  Rows like a random-init
    model's logits (N(0, 1.28^2)) and sharper ones (N(0, 4^2)).  Ids must
    equal the oracle's wherever the target u * sum(p) is not within the
    fp32 summation error of a CDF boundary; where they differ, every CDF
    boundary between the two ids is within that error of the target
    (float64 CDF)."""
    import oracle
    V, tau = 128256, 0.7
    for ci, (T, std) in enumerate([(48, 1.28), (48, 4.0)]):
        gen = torch.Generator(device="cuda").manual_seed(95 + ci)
        x = torch.randn(T, V, generator=gen, device="cuda") * std
        rid = torch.arange(T, dtype=torch.int64, device="cuda") * 104729 + ci
        st = torch.arange(T, dtype=torch.int64, device="cuda") * 3 + 1
        ids = torch.empty(T, dtype=torch.int32, device="cuda")
        bi.philox_sample(x, rid, st, tau, ids)
        sync_ok(bi)
        got = ids.cpu().numpy()
        xl = x.cpu().numpy()
        rl = rid.cpu().numpy().astype(np.uint64)
        sl = st.cpu().numpy().astype(np.uint64)
        ref = orc.philox_sample(xl, rl, sl, tau)
        mism = np.nonzero(got != ref)[0]
        assert len(mism) <= T // 4, (ci, len(mism))
        for t in mism:
            row = xl[t].astype(np.float64)
            p = np.exp((row - row.max()) / tau)
            cdf = np.cumsum(p)
            u = oracle.sample_uniform(oracle.sample_seed(int(rl[t]),
                                                          int(sl[t])))
            target = u * cdf[-1]
            lo, hi = sorted((int(got[t]), int(ref[t])))
            # boundaries crossed between the two ids: cdf[lo .. hi-1]
            assert np.all(np.abs(cdf[lo:hi] - target) < 1e-4 * cdf[-1]), \
                (ci, t, lo, hi)
        # a row alone gives its id in the batch
        one = torch.empty(1, dtype=torch.int32, device="cuda")
        bi.philox_sample(x[7:8].contiguous(), rid[7:8].contiguous(),
                         st[7:8].contiguous(), tau, one)
        sync_ok(bi)
        assert one.item() == got[7]
