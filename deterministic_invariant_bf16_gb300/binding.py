"""ctypes binding of ``libbi.so``: one Python function per C entry point,
same name, argument marshalling only.

Tensor arguments are torch tensors on the GPU (their ``data_ptr()`` is
passed); host arrays are numpy arrays.  Every non-zero status raises
``BiError`` with the library's message.  The library is required: there is
no fallback of any kind, and a missing ``libbi.so`` is an ImportError-like
failure at first use.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbi.so")

BI_OK = 0
STATUS_NAMES = {0: "BI_OK", 1: "BI_ERR_INVALID_ARG", 2: "BI_ERR_UNSUPPORTED",
                3: "BI_ERR_WORKSPACE_TOO_SMALL", 4: "BI_ERR_CUDA",
                5: "BI_ERR_BOUNDS", 6: "BI_ERR_TIMEOUT"}

OUT_PARTIALS, OUT_F32, OUT_BF16, OUT_SWIGLU = 0, 1, 2, 3
VERIFY_ROWS = 256


class BiError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


class ModelCfg(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("eps", ctypes.c_float),
                ("theta", ctypes.c_double), ("max_tokens", ctypes.c_int),
                ("max_kv_len", ctypes.c_int), ("max_pages", ctypes.c_int),
                ("n_pages", ctypes.c_int)]


PP = ctypes.POINTER(ctypes.c_void_p)


class ModelWeights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p), ("attn_norm", PP),
                ("wqkv", PP), ("wo", PP), ("ffn_norm", PP), ("wgu", PP),
                ("wd", PP), ("k_pool", PP), ("v_pool", PP)]


_lib = None

V, I, L, F, D, Z = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                    ctypes.c_float, ctypes.c_double, ctypes.c_size_t)
I32P = ctypes.POINTER(ctypes.c_int32)

SIGNATURES = {
    "bi_last_error": ([], ctypes.c_char_p),
    "bi_device_status": ([I32P, V], I),
    "bi_gemm_splits": ([I, I], I),
    "bi_gemm_tile_n": ([I, I], I),
    "bi_gemm_workspace_size": ([I, I, I], Z),
    "bi_gemm": ([V, I, I, V, I, V, I, V, Z, V], I),
    "bi_pack_gate_up": ([V, V, I, I, V, V], I),
    "bi_rmsnorm": ([V, I, V, V, V, I, I, F, V, V], I),
    "bi_embed": ([V, I, V, I, I, V, V], I),
    "bi_rope": ([V, I, V, V, I, I, I, I, D, V, V, V, V, I, I, V], I),
    "bi_swiglu": ([V, V, L, V, V], I),
    "bi_decode_attn_workspace_size": ([I, I, I, I], Z),
    "bi_paged_decode_attn": ([V, V, V, V, I, V, V, I, I, I, I, I, F, V, V, Z,
                              V], I),
    "bi_paged_decode_attn_noalloc": ([V, V, V, V, I, V, V, I, I, I, I, I, F,
                                      V, V], I),
    "bi_prefill_attn": ([V, V, V, I, I, V, I, I, V, V, V, I, I, I, I, F, V,
                         V], I),
    "bi_prefill_attn_workspace_size": ([I, I, I, I], Z),
    "bi_prefill_attn_split_workspace_size": ([I, I, I, I, I], Z),
    "bi_prefill_attn_ws": ([V, V, V, I, I, V, I, I, V, V, V, I, I, I, I, F, V,
                            V, Z, V], I),
    "bi_argmax_logits": ([V, I, I, V, V], I),
    "philox_sample": ([V, I, I, V, V, F, V, V], I),
    "philox_sample_top": ([V, I, I, V, V, F, I, F, V, V], I),
    "bi_model_workspace_size": ([ctypes.POINTER(ModelCfg)], Z),
    "bi_model_create": ([ctypes.POINTER(ModelCfg),
                         ctypes.POINTER(ModelWeights), V, Z,
                         ctypes.POINTER(V)], I),
    "bi_model_destroy": ([V], None),
    "bi_model_forward": ([V, I, V, V, V, I, V, V, I, I, V, V, V, V], I),
    "bi_model_profile": ([V, I], I),
    "bi_model_profile_read": ([V, ctypes.POINTER(ctypes.c_double),
                               ctypes.POINTER(ctypes.c_int64)], I),
    "verify_commit_rollback": ([V, I, I32P, I32P, I32P, I32P, I32P, V, V,
                                I32P, I32P, I32P, I, I32P, I32P, V, V], I),
    "verify_commit_rollback_device": ([V, V, V, V, V, V, V, V, V, V, V, V,
                                       I, V, V, V, V], I),
    "bi_model_hidden": ([V, ctypes.POINTER(V)], I),
    "bi_test_wait_timeout": ([L, V, V], I),
}


def lib():
    """Open ``libbi.so`` (built by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                "libbi.so is not built (run deterministic_invariant_bf16_gb300"
                "/build.py); there is no fallback path")
        h = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(h, name)
            fn.argtypes = args
            fn.restype = res
        _lib = h
    return _lib


def _check(status):
    if status != BI_OK:
        msg = lib().bi_last_error()
        raise BiError(status, msg.decode() if msg else "")


def _p(t):
    """Device pointer of a tensor (or None)."""
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(I32P)


# ------------------------------------------------------------- queries --

def bi_gemm_splits(N, K):
    return lib().bi_gemm_splits(N, K)


def bi_gemm_tile_n(N, K):
    return lib().bi_gemm_tile_n(N, K)


def bi_gemm_workspace_size(M, N, K):
    return lib().bi_gemm_workspace_size(M, N, K)


def bi_decode_attn_workspace_size(B, Hq, D, max_kv_len):
    return lib().bi_decode_attn_workspace_size(B, Hq, D, max_kv_len)


def bi_device_status(stream=None):
    out = ctypes.c_int32(0)
    _check(lib().bi_device_status(ctypes.byref(out), _stream(stream)))
    return out.value


# ---------------------------------------------------------- operators --

def bi_gemm(x, W, out, out_kind, ws=None, stream=None):
    M, K = x.shape
    N = W.shape[0]
    _check(lib().bi_gemm(_p(x), M, K, _p(W), N, _p(out), out_kind, _p(ws),
                         0 if ws is None else ws.numel() * ws.element_size(),
                         _stream(stream)))


def bi_pack_gate_up(wg, wu, wgu, stream=None):
    F, K = wg.shape
    _check(lib().bi_pack_gate_up(_p(wg), _p(wu), F, K, _p(wgu),
                                 _stream(stream)))


def bi_rmsnorm(partials, S, x, residual, w, T, H, eps, y, stream=None):
    _check(lib().bi_rmsnorm(_p(partials), S, _p(x), _p(residual), _p(w), T, H,
                            eps, _p(y), _stream(stream)))


def bi_embed(tokens, E, h, stream=None):
    V_, H = E.shape
    _check(lib().bi_embed(_p(tokens), tokens.numel(), _p(E), V_, H, _p(h),
                          _stream(stream)))


def bi_rope(qkv, S, pos, row_req, Hq, Hkv, D_, theta, q_out, k_pool, v_pool,
            page_table, stream=None):
    T = pos.numel()
    _check(lib().bi_rope(_p(qkv), S, _p(pos), _p(row_req), T, Hq, Hkv, D_,
                         theta, _p(q_out), _p(k_pool), _p(v_pool),
                         _p(page_table), page_table.shape[1], k_pool.shape[0],
                         _stream(stream)))


def bi_swiglu(g, u, out, stream=None):
    _check(lib().bi_swiglu(_p(g), _p(u), g.numel(), _p(out), _stream(stream)))


def bi_paged_decode_attn(q, k_pool, v_pool, page_table, row_req, kv_len,
                         max_kv_len, scale, out, ws, stream=None):
    B, Hq, D_ = q.shape
    Hkv = k_pool.shape[1]
    _check(lib().bi_paged_decode_attn(
        _p(q), _p(k_pool), _p(v_pool), _p(page_table), page_table.shape[1],
        _p(row_req), _p(kv_len), B, max_kv_len, Hq, Hkv, D_, scale, _p(out),
        _p(ws), ws.numel() * ws.element_size(), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def bi_paged_decode_attn_noalloc(q, k_pool, v_pool, page_table, row_req,
                                 kv_len, max_kv_len, scale, out, stream=None):
    """bi_paged_decode_attn without a workspace argument, for callers that
    cannot allocate device memory: its scratch is a fixed array inside the
    library (NOALLOC_SCRATCH_BYTES per GPU).  Calls that would need more
    scratch raise BiError (BI_ERR_WORKSPACE_TOO_SMALL); calls that overlap
    on the GPU share the array and must be ordered on one stream."""
    B, Hq, D_ = q.shape
    Hkv = k_pool.shape[1]
    _check(lib().bi_paged_decode_attn_noalloc(
        _p(q), _p(k_pool), _p(v_pool), _p(page_table), page_table.shape[1],
        _p(row_req), _p(kv_len), B, max_kv_len, Hq, Hkv, D_, scale, _p(out),
        _stream(stream)))


def bi_prefill_attn(q, cu_q, seg_req, pos, max_q, max_kv_len, k_pool, v_pool,
                    page_table, scale, out, stream=None):
    T, Hq, D_ = q.shape
    R = seg_req.numel()
    Hkv = k_pool.shape[1]
    _check(lib().bi_prefill_attn(
        _p(q), _p(cu_q), _p(seg_req), R, T, _p(pos), max_q, max_kv_len,
        _p(k_pool), _p(v_pool), _p(page_table), page_table.shape[1], Hq, Hkv,
        D_, scale, _p(out), _stream(stream)))


def bi_prefill_attn_workspace_size(T, R, Hq, Hkv):
    return lib().bi_prefill_attn_workspace_size(T, R, Hq, Hkv)


def bi_prefill_attn_split_workspace_size(T, R, Hq, Hkv, max_kv_len):
    return lib().bi_prefill_attn_split_workspace_size(T, R, Hq, Hkv,
                                                      max_kv_len)


def bi_prefill_attn_ws(q, cu_q, seg_req, pos, max_q, max_kv_len, k_pool,
                       v_pool, page_table, scale, out, ws, stream=None):
    T, Hq, D_ = q.shape
    R = seg_req.numel()
    Hkv = k_pool.shape[1]
    _check(lib().bi_prefill_attn_ws(
        _p(q), _p(cu_q), _p(seg_req), R, T, _p(pos), max_q, max_kv_len,
        _p(k_pool), _p(v_pool), _p(page_table), page_table.shape[1], Hq, Hkv,
        D_, scale, _p(out), _p(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def bi_argmax_logits(logits, ids, stream=None):
    T, V_ = logits.shape
    _check(lib().bi_argmax_logits(_p(logits), T, V_, _p(ids),
                                  _stream(stream)))


def philox_sample(logits, request_id, step, temperature, ids, stream=None):
    T, V_ = logits.shape
    _check(lib().philox_sample(_p(logits), T, V_, _p(request_id), _p(step),
                               temperature, _p(ids), _stream(stream)))


def philox_sample_top(logits, request_id, step, temperature, top_k, top_p,
                      ids, stream=None):
    T, V_ = logits.shape
    _check(lib().philox_sample_top(_p(logits), T, V_, _p(request_id),
                                   _p(step), temperature, top_k, top_p,
                                   _p(ids), _stream(stream)))


# -------------------------------------------------------------- model --

def bi_model_workspace_size(cfg: ModelCfg):
    return lib().bi_model_workspace_size(ctypes.byref(cfg))


def bi_model_create(cfg: ModelCfg, weights: ModelWeights, ws):
    handle = ctypes.c_void_p()
    _check(lib().bi_model_create(ctypes.byref(cfg), ctypes.byref(weights),
                                 _p(ws), ws.numel() * ws.element_size(),
                                 ctypes.byref(handle)))
    return handle


def bi_model_destroy(handle):
    lib().bi_model_destroy(handle)


def bi_model_forward(handle, tokens, pos, row_req, cu_q, seg_req, max_q,
                     max_kv_len, page_table, logits, ids, stream=None):
    T = tokens.numel()
    R = 0 if seg_req is None else seg_req.numel()
    _check(lib().bi_model_forward(handle, T, _p(tokens), _p(pos), _p(row_req),
                                  R, _p(cu_q), _p(seg_req), max_q, max_kv_len,
                                  _p(page_table), _p(logits), _p(ids),
                                  _stream(stream)))


PROF_CLASSES = ["attn", "attn_merge", "gemm_qkv", "gemm_o", "gemm_gate_up",
                "gemm_down", "lm_head", "norm", "rope", "other",
                "attn_prefill"]


def bi_model_profile(handle, enable):
    _check(lib().bi_model_profile(handle, 1 if enable else 0))


def bi_model_profile_read(handle):
    """Returns {class name: (milliseconds, launches)}."""
    n = len(PROF_CLASSES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _check(lib().bi_model_profile_read(handle, ms, cnt))
    return {name: (ms[i], cnt[i]) for i, name in enumerate(PROF_CLASSES)}


def verify_commit_rollback(handle, req, kv_len_host, last_token, win_len,
                           candidates, page_table, kv_len, logits,
                           freed_cap=4096, stream=None):
    """Returns (taken, commit_len, fix_token, freed_pages) as numpy arrays."""
    R = len(req)
    a_req, p_req = _i32(req)
    a_kv, p_kv = _i32(kv_len_host)
    a_last, p_last = _i32(last_token)
    a_w, p_w = _i32(win_len)
    a_c, p_c = _i32(candidates)
    commit = np.zeros(R, np.int32)
    fix = np.zeros(R, np.int32)
    freed = np.zeros(max(freed_cap, 1), np.int32)
    n_freed = ctypes.c_int32(0)
    taken = ctypes.c_int32(0)
    _check(lib().verify_commit_rollback(
        handle, R, p_req, p_kv, p_last, p_w, p_c, _p(page_table), _p(kv_len),
        commit.ctypes.data_as(I32P), fix.ctypes.data_as(I32P),
        freed.ctypes.data_as(I32P), freed_cap, ctypes.byref(n_freed),
        ctypes.byref(taken), _p(logits), _stream(stream)))
    n = taken.value
    return n, commit[:n], fix[:n], freed[:n_freed.value]


class VerifyBuffers:
    """Device buffers of one verify_commit_rollback_device call: the plan
    (window count, per-window request / KV length / last token / length,
    candidates) and the results (commit length, fix token, freed pages and
    their count, windows taken).  ``load`` fills the plan from host lists
    (a caller that captures the call refills these buffers between
    replays); ``read`` returns the results as numpy arrays."""

    def __init__(self, freed_cap, device="cuda"):
        import torch
        n = VERIFY_ROWS
        i32 = dict(dtype=torch.int32, device=device)
        # plan: [0] = R, then req, kv_len, last token, window length (n
        # each) and n candidates
        self.plan = torch.zeros(8 + 5 * n, **i32)
        self.n_windows = self.plan[0:1]
        self.req = self.plan[8:8 + n]
        self.win_kv_len = self.plan[8 + n:8 + 2 * n]
        self.last_token = self.plan[8 + 2 * n:8 + 3 * n]
        self.win_len = self.plan[8 + 3 * n:8 + 4 * n]
        self.candidates = self.plan[8 + 4 * n:8 + 5 * n]
        # results: [0] = taken, [1] = n_freed, commit, fix, freed pages
        self.freed_cap = int(freed_cap)
        self.out = torch.zeros(8 + 2 * n + max(self.freed_cap, 1), **i32)
        self.taken = self.out[0:1]
        self.n_freed = self.out[1:2]
        self.commit_len = self.out[8:8 + n]
        self.fix_token = self.out[8 + n:8 + 2 * n]
        self.freed = self.out[8 + 2 * n:]

    @staticmethod
    def host_plan(req, kv_len, last_token, windows):
        """The plan as one int32 array in the layout of ``plan`` (windows
        past the fixed batch's capacity are dropped from the candidates,
        as the packing never reads them)."""
        n = VERIFY_ROWS
        a = np.zeros(8 + 5 * n, np.int32)
        R = len(req)
        if not 1 <= R < n:
            raise ValueError("1 <= number of windows < %d" % n)
        a[0] = R
        a[8:8 + R] = req
        a[8 + n:8 + n + R] = kv_len
        a[8 + 2 * n:8 + 2 * n + R] = last_token
        a[8 + 3 * n:8 + 3 * n + R] = [len(w) for w in windows]
        cands = np.concatenate([np.asarray(w, np.int32) for w in windows])
        cands = cands[:n]
        a[8 + 4 * n:8 + 4 * n + len(cands)] = cands
        return a

    def load(self, req, kv_len, last_token, windows):
        import torch
        self.plan.copy_(torch.from_numpy(
            self.host_plan(req, kv_len, last_token, windows)))

    def read(self):
        """(taken, commit_len, fix_token, freed_pages) as numpy arrays."""
        o = self.out.cpu().numpy()
        n, nf = int(o[0]), int(o[1])
        m = VERIFY_ROWS
        return (n, o[8:8 + n].copy(), o[8 + m:8 + m + n].copy(),
                o[8 + 2 * m:8 + 2 * m + min(nf, self.freed_cap)].copy())


def verify_commit_rollback_device(handle, bufs: VerifyBuffers, page_table,
                                  kv_len, logits, stream=None):
    """Enqueues the device-side verification on ``bufs`` (no host sync)."""
    b = bufs
    _check(lib().verify_commit_rollback_device(
        handle, _p(b.n_windows), _p(b.req), _p(b.win_kv_len),
        _p(b.last_token), _p(b.win_len), _p(b.candidates), _p(page_table),
        _p(kv_len), _p(b.commit_len), _p(b.fix_token), _p(b.freed),
        b.freed_cap, _p(b.n_freed), _p(b.taken), _p(logits),
        _stream(stream)))


def bi_model_hidden(handle, T, hidden):
    """The residual stream of the last forward of T rows (a bf16 [T][hidden]
    tensor viewing the model's workspace)."""
    import torch
    ptr = ctypes.c_void_p()
    _check(lib().bi_model_hidden(handle, ctypes.byref(ptr)))
    return _view_bf16(ptr.value, T, hidden)


def _view_bf16(addr, rows, cols):
    """A torch bf16 [rows][cols] tensor over device memory at ``addr`` (not
    owned; valid while the memory is)."""
    import torch

    class _Mem:
        __cuda_array_interface__ = {
            "shape": (rows, cols), "typestr": "<i2", "version": 3,
            "data": (addr, False), "strides": None}
    return torch.as_tensor(_Mem(), device="cuda").view(torch.bfloat16)


def bi_test_wait_timeout(limit_ns, done, stream=None):
    _check(lib().bi_test_wait_timeout(int(limit_ns), _p(done),
                                      _stream(stream)))
