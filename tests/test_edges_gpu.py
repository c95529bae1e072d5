"""Edge cases through the C ABI on the GPU: empty inputs, pad rows, contexts
at the page-table limit, bounds violations that the kernels record and skip
(BI_ERR_BOUNDS in the status word, no memory access), and shapes refused on
the host before any launch."""
import math

import numpy as np
import pytest
import torch

from helpers import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bi():
    from deterministic_invariant_bf16_gb300 import binding, build
    build.build()
    binding.lib()
    return binding


def dev(shape, dtype=torch.bfloat16, seed=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda").to(dtype)


def test_empty_inputs_are_no_ops(bi):
    # zero rows of valid buffers: nothing launches, nothing is written
    W = dev((128, 64))
    x = dev((4, 64))[:0]
    out = torch.full((4, 128), 7.0, device="cuda")
    bi.bi_gemm(x, W, out[:0], bi.OUT_F32)
    h = dev((4, 128), seed=2)
    y = torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda")
    bi.bi_rmsnorm(None, 0, h[:0], None, dev((128,)), 0, 128, 1e-5, y[:0])
    ids = torch.full((4,), -3, dtype=torch.int32, device="cuda")
    bi.bi_argmax_logits(torch.zeros(4, 512, device="cuda")[:0], ids[:0])
    torch.cuda.synchronize()
    assert bi.bi_device_status() == 0
    assert torch.all(out == 7.0) and torch.count_nonzero(y) == 0
    assert torch.all(ids == -3)


def test_host_refuses_bad_shapes(bi):
    W = dev((100, 64))   # N not a multiple of 8
    x = dev((4, 64))
    out = torch.empty(4, 100, dtype=torch.float32, device="cuda")
    with pytest.raises(bi.BiError) as e:
        bi.bi_gemm(x, W, out, bi.OUT_F32)
    assert e.value.status == 1
    W = dev((128, 60))   # K not a multiple of 8
    with pytest.raises(bi.BiError):
        bi.bi_gemm(dev((4, 60)), W, out, bi.OUT_F32)
    # SwiGLU with more than one K slice needs the second-stage workspace
    K = 4096
    wgu = dev((256, K), seed=3)
    xs = dev((3, K), seed=4)
    sw = torch.empty(3, 128, dtype=torch.bfloat16, device="cuda")
    assert bi.bi_gemm_splits(256, K) > 1
    with pytest.raises(bi.BiError) as e:
        bi.bi_gemm(xs, wgu, sw, bi.OUT_SWIGLU)
    assert e.value.status == 3
    ws = torch.empty(bi.bi_gemm_workspace_size(3, 256, K) // 4,
                     dtype=torch.float32, device="cuda")
    bi.bi_gemm(xs, wgu, sw, bi.OUT_SWIGLU, ws)
    torch.cuda.synchronize()
    assert bi.bi_device_status() == 0


def _pool(lens, Hkv=8, D=128, seed=1):
    rng = np.random.default_rng(seed)
    max_pages = max(-(-n // 16) for n in lens)
    n_pages = sum(-(-n // 16) for n in lens)
    perm = rng.permutation(n_pages).astype(np.int32)
    table = np.full((len(lens), max_pages), -1, np.int32)
    at = 0
    for r, n in enumerate(lens):
        k = -(-n // 16)
        table[r, :k] = perm[at:at + k]
        at += k
    kp = dev((n_pages, Hkv, 16, D), seed=seed)
    vp = dev((n_pages, Hkv, 16, D), seed=seed + 1)
    return kp, vp, table, max_pages


def _decode(bi, q, kp, vp, table, rows, lens, max_kv):
    B, Hq, D = q.shape
    ws = torch.empty(bi.bi_decode_attn_workspace_size(B, Hq, D, max_kv) // 4,
                     dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    bi.bi_paged_decode_attn(q, kp, vp, torch.from_numpy(table).cuda(),
                            torch.tensor(rows, dtype=torch.int32).cuda(),
                            torch.tensor(lens, dtype=torch.int32).cuda(),
                            max_kv, 1 / math.sqrt(D), out, ws)
    torch.cuda.synchronize()
    return out


def test_pad_rows_and_context_at_the_page_table_limit(bi):
    lens = [48, 320, 1024]           # the last fills its page-table row
    kp, vp, table, max_pages = _pool(lens)
    assert 16 * max_pages == 1024
    q = dev((4, 32, 128), seed=9)
    rows = [0, -1, 1, 2]             # row 1 is a pad row
    out = _decode(bi, q, kp, vp, table, rows, [48, 1, 320, 1024], 1024)
    assert bi.bi_device_status() == 0
    assert torch.count_nonzero(out[1]) == 0
    # the pad row does not disturb its neighbours
    alone = _decode(bi, q[[0, 2, 3]].contiguous(), kp, vp, table, [0, 1, 2],
                    [48, 320, 1024], 1024)
    assert np.array_equal(bits(out[[0, 2, 3]]), bits(alone))


def test_unmapped_visible_page_is_recorded_not_read(bi):
    lens = [100, 200]
    kp, vp, table, _ = _pool(lens)
    table[1, 3] = -1                 # a visible position without a page
    q = dev((2, 32, 128), seed=11)
    _decode(bi, q, kp, vp, table, [0, 1], lens, 200)
    assert bi.bi_device_status() == 5   # BI_ERR_BOUNDS
    assert bi.bi_device_status() == 0   # read-and-clear


def test_bad_token_id_is_recorded(bi):
    E = dev((512, 128))
    tok = torch.tensor([3, 600, 7], dtype=torch.int32, device="cuda")
    h = torch.empty(3, 128, dtype=torch.bfloat16, device="cuda")
    bi.bi_embed(tok, E, h)
    torch.cuda.synchronize()
    assert bi.bi_device_status() == 5
    assert torch.count_nonzero(h[1]) == 0
    assert torch.equal(h[0], E[3]) and torch.equal(h[2], E[7])


def test_bounded_wait_runs_out_and_the_library_recovers(bi):
    """A device wait that nothing completes gives up after its limit (here
    5 ms, the same wait loop the kernels run with 2 s), records
    BI_ERR_TIMEOUT in the status word and lets its kernel return; the
    context stays usable and the next ordinary call gives the same bits as
    before."""
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn(64, 512, generator=g, device="cuda").to(torch.bfloat16)
    w = torch.randn(384, 512, generator=g, device="cuda").to(torch.bfloat16)
    S = bi.bi_gemm_splits(384, 512)
    before = torch.empty(S, 64, 384, dtype=torch.float32, device="cuda")
    bi.bi_gemm(x, w, before, bi.OUT_PARTIALS)
    torch.cuda.synchronize()
    assert bi.bi_device_status() == 0
    done = torch.zeros(1, dtype=torch.int32, device="cuda")
    bi.bi_test_wait_timeout(5_000_000, done)
    torch.cuda.synchronize()
    assert done.item() == 2
    assert bi.bi_device_status() == 6      # BI_ERR_TIMEOUT, read and cleared
    assert bi.bi_device_status() == 0
    after = torch.empty_like(before)
    bi.bi_gemm(x, w, after, bi.OUT_PARTIALS)
    torch.cuda.synchronize()
    assert bi.bi_device_status() == 0
    assert torch.equal(before.view(torch.int32), after.view(torch.int32))
    with pytest.raises(bi.BiError, match="INVALID"):
        bi.bi_test_wait_timeout(10**9, done)
