"""The C ABI library loads on a machine without a GPU, exports every entry
point include/bi.h declares, and rejects bad arguments before launching."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bi():
    from deterministic_invariant_bf16_gb300 import build, binding
    build.build()
    return binding


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            if not m.group(0).lstrip().startswith(("typedef", "#")):
                names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(bi):
    names = declared_functions()
    assert {"bi_gemm", "bi_rmsnorm", "bi_rope", "bi_swiglu",
            "bi_paged_decode_attn", "bi_prefill_attn", "bi_argmax_logits",
            "verify_commit_rollback", "philox_sample"} <= names
    lib = ctypes.CDLL(bi.LIB_PATH)
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding wraps each of them under the same name
    assert names <= set(bi.SIGNATURES)


def test_split_counts_depend_only_on_weight_shape(bi):
    # 8B shapes: QKV, O, gate/up (interleaved), down, LM head
    s = {(n, k): bi.bi_gemm_splits(n, k) for n, k in
         [(6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336),
          (128256, 4096), (384, 128), (512, 128)]}
    assert s[(28672, 4096)] == 1 and s[(128256, 4096)] == 1
    assert s[(512, 128)] == 1
    assert all(1 <= v <= 8 for v in s.values())
    assert bi.bi_gemm_workspace_size(1, 4096, 4096) == \
        s[(4096, 4096)] * 4096 * 4 * (s[(4096, 4096)] > 1)


def test_bad_arguments_fail_before_launch(bi):
    lib = bi.lib()
    # K not a multiple of 8
    assert lib.bi_gemm(ctypes.c_void_p(16), 4, 7, ctypes.c_void_p(16), 8,
                       ctypes.c_void_p(16), 1, None, 0, None) == 1
    # null pointers
    assert lib.bi_gemm(None, 4, 64, None, 8, None, 1, None, 0, None) == 1
    assert b"null" in lib.bi_last_error()
    # unsupported head dim
    assert lib.bi_paged_decode_attn(
        ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
        ctypes.c_void_p(16), 4, ctypes.c_void_p(16), ctypes.c_void_p(16),
        1, 16, 4, 4, 64, 0.1, ctypes.c_void_p(16), ctypes.c_void_p(16),
        1 << 20, None) == 2
    # sampling: a row of 2^30 logits, a negative temperature, top_k > 1024
    f = ctypes.c_void_p(16)
    assert lib.philox_sample(f, 1, 1 << 30, f, f, ctypes.c_float(1.0), f,
                             None) == 1
    assert lib.philox_sample(f, 1, 64, f, f, ctypes.c_float(-1.0), f,
                             None) == 1
    assert b"temperature" in lib.bi_last_error()
    assert lib.philox_sample_top(f, 1, 64, f, f, ctypes.c_float(1.0), 1025,
                                 ctypes.c_float(0.9), f, None) == 2
    # verify needs a model
    assert lib.verify_commit_rollback(None, 1, *([None] * 5), None, None,
                                      None, None, None, 0, None, None, None,
                                      None) == 1
    cfg = bi.ModelCfg(n_layers=1, hidden=128, n_heads=4, n_kv_heads=4,
                      head_dim=64, ffn=256, vocab=512, eps=1e-5, theta=1e4,
                      max_tokens=8, max_kv_len=64, max_pages=4, n_pages=8)
    assert bi.bi_model_workspace_size(cfg) == 0   # head_dim 64 unsupported
    cfg.head_dim = 32
    assert bi.bi_model_workspace_size(cfg) > 0


def test_decode_workspace_formula(bi):
    # chunk partials (m, l, pad, o[D]) per (row, head, chunk), the per-row
    # chunk prefix (B + 1 ints) and the (row, chunk) work list (8 bytes per
    # entry), each rounded up to 256 bytes
    def up(n):
        return (n + 255) // 256 * 256
    assert bi.bi_decode_attn_workspace_size(3, 32, 128, 257) == \
        up(3 * 32 * 2 * 132 * 4) + up(4 * 4) + up(3 * 2 * 8)
    assert bi.bi_decode_attn_workspace_size(1, 4, 32, 16) == \
        up(1 * 4 * 1 * 36 * 4) + up(2 * 4) + up(1 * 1 * 8)


def test_verify_refuses_bad_plans_before_launch(bi):
    """The host entry point checks the FIFO plan before it uploads anything:
    two taken windows naming one request (both would write that request's
    KV and cut its page-table row), an empty window, a window past the
    model's longest context.  No GPU is touched: the model handle holds
    placeholder addresses that nothing dereferences."""
    lib = bi.lib()
    cfg = bi.ModelCfg(n_layers=1, hidden=128, n_heads=4, n_kv_heads=4,
                      head_dim=32, ffn=256, vocab=512, eps=1e-5, theta=1e4,
                      max_tokens=256, max_kv_len=64, max_pages=4, n_pages=8)
    nbytes = bi.bi_model_workspace_size(cfg)
    assert nbytes > 0
    fake = ctypes.c_void_p(1 << 20)
    arr = (ctypes.c_void_p * 1)(1 << 20)
    pp = ctypes.cast(arr, bi.PP)
    w = bi.ModelWeights(embed=1 << 20, final_norm=1 << 20, lm_head=1 << 20,
                        attn_norm=pp, wqkv=pp, wo=pp, ffn_norm=pp, wgu=pp,
                        wd=pp, k_pool=pp, v_pool=pp)
    handle = ctypes.c_void_p()
    assert lib.bi_model_create(ctypes.byref(cfg), ctypes.byref(w), fake,
                               nbytes, ctypes.byref(handle)) == 0
    try:
        I32 = ctypes.c_int32

        def call(req, kv, last, wl, cands):
            R = len(req)
            a = [(I32 * max(1, len(x)))(*x) for x in (req, kv, last, wl,
                                                      cands)]
            out = [(I32 * 8)() for _ in range(2)]
            freed = (I32 * 8)()
            nf, tk = I32(0), I32(0)
            return lib.verify_commit_rollback(
                handle, R, *a, fake, fake, out[0], out[1], freed, 8,
                ctypes.byref(nf), ctypes.byref(tk), fake, None)

        st = call([3, 3], [10, 12], [1, 2], [4, 4], [0] * 8)
        assert st == 1 and b"both name request 3" in lib.bi_last_error()
        st = call([3, 4], [10, 12], [1, 2], [4, 0], [0] * 4)
        assert st == 1 and b"length 0" in lib.bi_last_error()
        st = call([3], [62], [1], [4], [0] * 4)
        assert st == 1 and b"max_kv_len" in lib.bi_last_error()
        # the device variant needs every pointer
        assert lib.verify_commit_rollback_device(
            handle, *([None] * 11), 0, None, None, None, None) == 1
    finally:
        lib.bi_model_destroy(handle)
