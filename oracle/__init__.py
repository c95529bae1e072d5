"""Oracle: a plain, slow CPU statement of the batch-invariant decoder and of
the LLM-42 commit/rollback rule.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the GPU library and never imports it; the two meet only through the
seeded inputs that the tests hand to both.

Arithmetic lives in ``oracle.c`` (sequential fp32 sums, one per output,
separately rounded multiplies and adds).  This module composes those
operations into the decoder exactly in the order a pre-norm Llama block runs,
and states the integer rules (packing, commit, rollback) in plain Python.

Sources (the three web pages on deterministic LLM inference):
  * "LLM-42: Enabling Determinism in LLM Inference with Verified Speculation"
    (ai-infra-wiki summary of the SOSP'26 paper), section "核心方法" (core
    method, paper sections 4.1-4.3 and Fig. 8): candidate window, fixed-shape
    verification, commit of the matching prefix, rollback at the first
    mismatch, grouped 256-token verification.
  * ybb.press, "LLM 推理确定性工程深度实战", sections 2.1 (non-associativity),
    4 (batch-invariant kernels), 6 item 3 (Philox per (request_id, step)).
  * Vosti abstract (arxivdaily 2609.38981): bitwise-identical logits across
    batch composition, query length and paged KV layout.

Where the pages leave a step open the reading taken is stated beside it.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against values the pages print, closed forms, float64 brute force, invariants
or numpy/torch library routines.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
        i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
        u64p = np.ctypeslib.ndpointer(np.uint64, flags="C_CONTIGUOUS")
        I, L, F, D = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        sig = {
            "orc_f32_to_bf16": [f32p, L, u16p],
            "orc_bf16_to_f32": [u16p, L, f32p],
            "orc_nonassoc_demo": [F, F, F, ctypes.POINTER(F), ctypes.POINTER(F)],
            "orc_gemm_bf16": [u16p, I, I, u16p, I, f32p],
            "orc_rmsnorm": [f32p, I, I, u16p, F, f32p],
            "orc_rope": [f32p, I, I, I, i32p, D],
            "orc_attention": [f32p, I, I, I, I, f32p, f32p, I, i32p, i32p, F,
                              f32p, f32p],
            "orc_swiglu": [f32p, f32p, L, f32p],
            "orc_argmax": [f32p, I, I, i32p],
            "orc_philox4x64_10": [u64p, u64p, u64p],
            "orc_sample_seed": [ctypes.c_uint64, ctypes.c_uint64],
            "orc_sample_uniform": [ctypes.c_uint64],
            "orc_philox_sample": [f32p, I, I, u64p, u64p, F, f32p, i32p],
            "orc_philox_sample_top": [f32p, I, I, u64p, u64p, F, I, F, i32p,
                                      f32p, i32p],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = None
        lib.orc_sample_seed.restype = ctypes.c_uint64
        lib.orc_sample_uniform.restype = ctypes.c_float
        _LIB = lib
    return _LIB


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _u16(a):
    a = np.asarray(a)
    assert a.dtype == np.uint16, "bf16 values travel as uint16 bit patterns"
    return np.ascontiguousarray(a)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


# ----------------------------------------------------------------- bf16 --

def bf16_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (ybb.press 2.1)."""
    x = _f32(x)
    out = np.empty(x.shape, np.uint16)
    _lib().orc_f32_to_bf16(x.reshape(-1), x.size, out.reshape(-1))
    return out


def bf16_value(bits) -> np.ndarray:
    """bf16 bit patterns -> the fp32 numbers they denote (exact)."""
    bits = _u16(bits)
    out = np.empty(bits.shape, np.float32)
    _lib().orc_bf16_to_f32(bits.reshape(-1), bits.size, out.reshape(-1))
    return out


def bf16r(x) -> np.ndarray:
    """Round fp32 values to bf16 and return them as fp32 (a storage point)."""
    return bf16_value(bf16_bits(x))


def nonassoc_demo(a=1e8, b=-1e8, c=1.0):
    """fp32 (a+b)+c and a+(b+c) (ybb.press 2.1): 1.0 and 0.0 for the page's
    values."""
    left, right = ctypes.c_float(), ctypes.c_float()
    _lib().orc_nonassoc_demo(a, b, c, ctypes.byref(left), ctypes.byref(right))
    return left.value, right.value


# ------------------------------------------------------------ operators --

def gemm(x_bits, w_bits) -> np.ndarray:
    """y = x W^T in fp32, W stored [N, K]; each output a sequential k-sum
    (ybb.press 2.2 and 4: the GEMM K-loop is the reduction at stake)."""
    x_bits, w_bits = _u16(x_bits), _u16(w_bits)
    M, K = x_bits.shape
    N, K2 = w_bits.shape
    assert K == K2
    y = np.empty((M, N), np.float32)
    if M and N:
        _lib().orc_gemm_bf16(x_bits, M, K, w_bits, N, y)
    return y


def rmsnorm(x, w_bits, eps) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w per row, fp32."""
    x = _f32(x)
    T, H = x.shape
    y = np.empty_like(x)
    if T:
        _lib().orc_rmsnorm(x, T, H, _u16(w_bits), eps, y)
    return y


def rope(x, pos, theta) -> np.ndarray:
    """Half-split rotary embedding of x [T, nh, D] at absolute positions
    [reading: pairs (i, i + D/2), angle pos * theta^(-2i/D), no frequency
    scaling]."""
    x = _f32(x).copy()
    T, nh, D = x.shape
    if T:
        _lib().orc_rope(x, T, nh, D, _i32(pos), float(theta))
    return x


def attention(q, kc, vc, row_req, row_pos, scale) -> np.ndarray:
    """Causal GQA attention of rows at absolute positions over per-request
    caches in logical order (Vosti: the result may depend only on the logical
    token prefix, never on the paged layout)."""
    q = _f32(q)
    T, Hq, D = q.shape
    kc, vc = _f32(kc), _f32(vc)
    R, L, Hkv, D2 = kc.shape
    assert D == D2 and vc.shape == kc.shape and Hq % Hkv == 0
    out = np.empty_like(q)
    if T:
        scratch = np.empty((T * Hq, max(L, 1)), np.float32)
        _lib().orc_attention(q, T, Hq, Hkv, D, kc, vc, L, _i32(row_req),
                             _i32(row_pos), scale, scratch, out)
    return out


def swiglu(g, u) -> np.ndarray:
    """silu(g) * u, silu(g) = g / (1 + e^-g)."""
    g, u = _f32(g), _f32(u)
    assert g.shape == u.shape
    out = np.empty_like(g)
    _lib().orc_swiglu(g.reshape(-1), u.reshape(-1), g.size, out.reshape(-1))
    return out


def argmax(x) -> np.ndarray:
    """First index of the row maximum; NaN is maximal, first NaN wins."""
    x = _f32(x)
    T, V = x.shape
    ids = np.empty(T, np.int32)
    if T:
        _lib().orc_argmax(x, T, V, ids)
    return ids


# --------------------------------------------------------------- Philox --

def philox4x64_10(counter, key) -> np.ndarray:
    """Raw Philox4x64-10 block for a 4-word counter and a 2-word key."""
    ctr = np.ascontiguousarray(counter, dtype=np.uint64)
    k = np.ascontiguousarray(key, dtype=np.uint64)
    out = np.empty(4, np.uint64)
    _lib().orc_philox4x64_10(ctr, k, out)
    return out


def sample_seed(request_id: int, step: int) -> int:
    """(request_id * 1000003 + step) mod 2^64 (ybb.press section 6, item 3)."""
    return int(_lib().orc_sample_seed(request_id, step))


def sample_uniform(seed: int) -> float:
    """u = top 24 bits of Philox4x64-10(counter 0, key (seed, 0)) word 0,
    times 2^-24 [reading: the page's torch.Generator seeding names no keyed
    API; a keyed Philox4x64-10 is the counter-based generator it describes]."""
    return float(_lib().orc_sample_uniform(seed))


def philox_sample(logits, request_id, step, tau) -> np.ndarray:
    """Inverse-CDF temperature sampling with the per-request uniform."""
    logits = _f32(logits)
    T, V = logits.shape
    rid = np.ascontiguousarray(request_id, dtype=np.uint64)
    st = np.ascontiguousarray(step, dtype=np.uint64)
    ids = np.empty(T, np.int32)
    scratch = np.empty((T, V), np.float32)
    if T:
        _lib().orc_philox_sample(logits, T, V, rid, st, float(tau), scratch,
                                 ids)
    return ids


def philox_sample_top(logits, request_id, step, tau, top_k, top_p):
    """Temperature sampling within the top_k highest-ranked tokens (larger
    logit first, ties to the lower index, NaN as -inf) and their nucleus of
    mass top_p, inverse CDF in rank order with the request's Philox
    uniform."""
    logits = _f32(logits)
    T, V = logits.shape
    rid = np.ascontiguousarray(request_id, dtype=np.uint64)
    st = np.ascontiguousarray(step, dtype=np.uint64)
    ids = np.empty(T, np.int32)
    if T:
        _lib().orc_philox_sample_top(logits, T, V, rid, st, float(tau),
                                     int(top_k), float(top_p),
                                     np.empty(V, np.int32),
                                     np.empty(V, np.float32), ids)
    return ids


# -------------------------------------------------------------- decoder --

@dataclass(frozen=True)
class Cfg:
    """Decoder shape.  Defaults are the tiny random-init decoder."""
    n_layers: int = 2
    hidden: int = 128
    n_heads: int = 4
    n_kv_heads: int = 4
    head_dim: int = 32
    ffn: int = 256
    vocab: int = 512
    eps: float = 1e-5
    theta: float = 1e4

    @property
    def q_dim(self):
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self):
        return self.n_kv_heads * self.head_dim


def decoder_layer(h, row_req, row_pos, lw, kc, vc, cfg: Cfg) -> np.ndarray:
    """One pre-norm Llama block over rows at absolute positions.

    h is [T, H] (bf16-valued fp32); lw holds the layer's bf16 weights as
    uint16: attn_norm [H], wqkv [(Hq+2Hkv)D, H] (rows: q heads, k heads,
    v heads), wo [H, Hq D], ffn_norm [H], wg [F, H], wu [F, H], wd [H, F].
    kc, vc [R, L, Hkv, D] are the per-request caches, written here at
    (row_req, row_pos) before any row reads them.  Values are rounded to bf16
    where the method stores them (normed activations, q/k/v, the KV cache,
    the attention output, the SwiGLU output, the residual stream) [reading:
    the storage points of the GPU path; the tolerance would accept fp32]."""
    T = h.shape[0]
    Hq, Hkv, D = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    x = bf16_bits(rmsnorm(h, lw["attn_norm"], cfg.eps))
    qkv = bf16r(gemm(x, lw["wqkv"]))
    q = qkv[:, :Hq * D].reshape(T, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D)
    v = qkv[:, (Hq + Hkv) * D:].reshape(T, Hkv, D)
    q = bf16r(rope(q, row_pos, cfg.theta))
    k = bf16r(rope(k, row_pos, cfg.theta))
    kc[row_req, row_pos] = k
    vc[row_req, row_pos] = v
    scale = np.float32(1.0 / math.sqrt(D))
    a = bf16_bits(attention(q, kc, vc, row_req, row_pos, scale)
                  .reshape(T, Hq * D))
    h = bf16r(h + gemm(a, lw["wo"]))
    x2 = bf16_bits(rmsnorm(h, lw["ffn_norm"], cfg.eps))
    f = bf16_bits(swiglu(gemm(x2, lw["wg"]), gemm(x2, lw["wu"])))
    h = bf16r(h + gemm(f, lw["wd"]))
    return h


def new_caches(cfg: Cfg, n_requests: int, max_len: int):
    """Per-layer logical KV caches [R, L, Hkv, D] (fp32 holding bf16 values)."""
    shape = (n_requests, max_len, cfg.n_kv_heads, cfg.head_dim)
    return [(np.zeros(shape, np.float32), np.zeros(shape, np.float32))
            for _ in range(cfg.n_layers)]


def model_forward(ids, row_req, row_pos, weights, caches, cfg: Cfg,
                  hidden_out=None) -> np.ndarray:
    """Untied embedding gather, the layer stack, final RMSNorm and the LM head
    with fp32 logits [reading: fp32 logits leave fewer argmax ties].  Returns
    logits [T, V]; if ``hidden_out`` is a list, the input of every layer and
    the final hidden state are appended to it."""
    ids = np.asarray(ids, np.int64)
    h = bf16_value(weights["embed"][ids])
    for li, lw in enumerate(weights["layers"]):
        if hidden_out is not None:
            hidden_out.append(h.copy())
        kc, vc = caches[li]
        h = decoder_layer(h, row_req, row_pos, lw, kc, vc, cfg)
    if hidden_out is not None:
        hidden_out.append(h.copy())
    x = bf16_bits(rmsnorm(h, weights["final_norm"], cfg.eps))
    return gemm(x, weights["lm_head"])


def greedy_decode(prompts, n_new, weights, cfg: Cfg, batch=None):
    """Greedy decoding: prefill each prompt, then repeatedly take the argmax
    and feed it back (ybb.press section 8, item 1: outputs at batch=1 and at
    batch=32 must be token-identical).  ``batch`` groups requests into one
    forward call per step (rows of several requests side by side); None means
    all requests together.  Returns a list of token lists."""
    R = len(prompts)
    max_len = max(len(p) for p in prompts) + n_new + 1
    caches = new_caches(cfg, R, max_len)
    batch = batch or R
    outs = [[] for _ in range(R)]
    for lo in range(0, R, batch):
        reqs = list(range(lo, min(R, lo + batch)))
        ids, rr, rp = [], [], []
        for r in reqs:
            ids += list(prompts[r])
            rr += [r] * len(prompts[r])
            rp += list(range(len(prompts[r])))
        logits = model_forward(ids, np.array(rr), np.array(rp), weights,
                               caches, cfg)
        last = np.cumsum([len(prompts[r]) for r in reqs]) - 1
        nxt = argmax(logits[last])
        for r, t in zip(reqs, nxt):
            outs[r].append(int(t))
        for step in range(1, n_new):
            ids = [outs[r][-1] for r in reqs]
            rp = [len(prompts[r]) + step - 1 for r in reqs]
            logits = model_forward(ids, np.array(reqs), np.array(rp), weights,
                                   caches, cfg)
            for r, t in zip(reqs, argmax(logits)):
                outs[r].append(int(t))
    return outs


# ------------------------------------------------- LLM-42 verification --

def pack_fifo(window_lens, capacity=256):
    """Grouped verification batch (LLM-42 section 4.3): take windows in FIFO
    order while their total stays within the fixed verify shape.  Returns the
    number of windows taken and, per taken window, its first row."""
    taken, starts, used = 0, [], 0
    for w in window_lens:
        if used + w > capacity:
            break
        starts.append(used)
        used += w
        taken += 1
    return taken, starts


def verify_rows(kv_len, last_token, candidates):
    """Rows a window contributes to the verify batch: row i sits at absolute
    position kv_len + i; its input is the last committed token for i = 0 and
    candidate c[i-1] after that; its argmax is compared with c[i]
    [reading: the cache holds every committed token but the last one]."""
    w = len(candidates)
    toks = [int(last_token)] + [int(c) for c in candidates[:w - 1]]
    return toks, [kv_len + i for i in range(w)]


def commit_rule(kv_len, candidates, verified, page_size=16):
    """LLM-42 commit/rollback (section 4.2, Fig. 8): commit the prefix of
    candidates that the fixed-shape recomputation reproduces, stop at the
    first mismatch j, drop every later candidate and roll the KV back to the
    committed prefix.  Returns (j, new kv_len, fix token or -1, pages kept)."""
    w = len(candidates)
    j = w
    for i in range(w):
        if int(verified[i]) != int(candidates[i]):
            j = i
            break
    new_len = kv_len + j
    fix = int(verified[j]) if j < w else -1
    keep = -(-new_len // page_size)
    return j, new_len, fix, keep
