"""bi_paged_decode_attn_noalloc: the decode-attention entry point for callers
that cannot allocate device memory for a workspace (its scratch is a fixed
array inside the library).  It must give exactly the bits of
bi_paged_decode_attn with a caller workspace, on two calls in a row with
different inputs, and refuse shapes that need more scratch than it has.

This file stands alone (no fixtures from conftest) so that it passes both in
a fresh process and after the rest of the suite; its name makes pytest
collect it last."""
import ctypes
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    from deterministic_invariant_bf16_gb300 import binding, build
    build.build()
    binding.lib()
    return binding


def _paged_case(lens, Hq, Hkv, D, seed):
    """Random K/V in a NaN-filled pool under a random page order, random
    queries, one row per request."""
    rng = np.random.default_rng(seed)
    max_pages = max(-(-n // 16) for n in lens) + 1
    n_pages = sum(-(-n // 16) for n in lens) + 5
    perm = rng.permutation(n_pages)
    table = np.full((len(lens), max_pages), -1, np.int32)
    kp = torch.full((n_pages, Hkv, 16, D), float("nan"), dtype=torch.bfloat16)
    vp = kp.clone()
    at = 0
    for r, n in enumerate(lens):
        for pi in range(-(-n // 16)):
            pg = int(perm[at])
            at += 1
            table[r, pi] = pg
            m = min(16, n - 16 * pi)
            kp[pg, :, :m] = torch.from_numpy(
                rng.standard_normal((Hkv, m, D)).astype(np.float32))
            vp[pg, :, :m] = torch.from_numpy(
                rng.standard_normal((Hkv, m, D)).astype(np.float32))
    q = torch.from_numpy(rng.standard_normal((len(lens), Hq, D)).astype(
        np.float32)).to(torch.bfloat16)
    dev = dict(device="cuda")
    return (q.to(**dev), kp.to(**dev), vp.to(**dev),
            torch.from_numpy(table).to(**dev),
            torch.arange(len(lens), dtype=torch.int32, **dev),
            torch.tensor(lens, dtype=torch.int32, **dev))


def _with_workspace(bi, q, kp, vp, pt, rows, kvl, max_kv, scale):
    B, Hq, D = q.shape
    ws = torch.empty(bi.bi_decode_attn_workspace_size(B, Hq, D, max_kv) // 4,
                     dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    bi.bi_paged_decode_attn(q, kp, vp, pt, rows, kvl, max_kv, scale, out, ws)
    return out


def test_noalloc_matches_workspace_variant_on_two_calls(bi):
    Hq, Hkv, D = 32, 8, 128
    cases = [[1, 17, 256, 257, 900, 2000, 40], [3000, 5, 512, 513]]
    for i, lens in enumerate(cases):
        q, kp, vp, pt, rows, kvl = _paged_case(lens, Hq, Hkv, D, 100 + i)
        max_kv = max(lens)
        scale = 1.0 / math.sqrt(D)
        ref = _with_workspace(bi, q, kp, vp, pt, rows, kvl, max_kv, scale)
        out = torch.empty_like(q)
        bi.bi_paged_decode_attn_noalloc(q, kp, vp, pt, rows, kvl, max_kv,
                                        scale, out)
        torch.cuda.synchronize()
        assert bi.bi_device_status() == 0
        assert not torch.isnan(out.float()).any()
        # the same kernels on the same inputs: bit-identical results
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), i


def test_noalloc_whole_row_items_match_workspace_variant(bi):
    """At 8 or more (row, KV head) items per SM the decode kernel takes
    whole rows and merges their chunks in registers (the form 8B-shape
    batches of 160 rows and more use); with contexts of at most 1024
    positions such a batch fits the fixed scratch.  Same bits as with a
    caller workspace, on two calls in a row."""
    Hq, Hkv, D = 32, 8, 128
    B = 8 * torch.cuda.get_device_properties(0).multi_processor_count // Hkv
    B = max(B, 160)
    for i in range(2):
        rng = np.random.default_rng(300 + i)
        lens = [int(x) for x in rng.integers(1, 1025, size=B)]
        q, kp, vp, pt, rows, kvl = _paged_case(lens, Hq, Hkv, D, 200 + i)
        max_kv = max(lens)
        assert bi.bi_decode_attn_workspace_size(B, Hq, D, max_kv) <= \
            bi.NOALLOC_SCRATCH_BYTES
        scale = 1.0 / math.sqrt(D)
        ref = _with_workspace(bi, q, kp, vp, pt, rows, kvl, max_kv, scale)
        out = torch.empty_like(q)
        bi.bi_paged_decode_attn_noalloc(q, kp, vp, pt, rows, kvl, max_kv,
                                        scale, out)
        torch.cuda.synchronize()
        assert bi.bi_device_status() == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), i


def test_noalloc_rejects_oversized_calls(bi):
    lib = bi.lib()
    # 64 rows of 4096 positions need 64 * 32 * 16 * 528 bytes > 16 MiB
    need = bi.bi_decode_attn_workspace_size(64, 32, 128, 4096)
    assert need > bi.NOALLOC_SCRATCH_BYTES
    p = ctypes.c_void_p(256)
    st = lib.bi_paged_decode_attn_noalloc(p, p, p, p, 256, p, p, 64, 4096, 32,
                                          8, 128, 0.1, p, None)
    assert st == 3  # BI_ERR_WORKSPACE_TOO_SMALL, nothing launched
    assert b"scratch" in lib.bi_last_error()
