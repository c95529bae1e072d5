"""The non-invariant fast path LLM-42 pairs with verification.

LLM-42 ("LLM-42: Enabling Determinism in LLM Inference with Verified
Speculation", section 核心方法) decodes every request on the engine's
ordinary fast kernels and recomputes only the deterministic requests'
tokens on a fixed-shape invariant path.  Here the fast path is the same
decoder with every GEMM through cuBLAS (torch.mm: the library heuristics
pick tiles and split-K from the batch shape, so results depend on the batch;
ybb.press section 2.2) and the library's RMSNorm, RoPE + KV append and paged
attention around them.  It writes its K and V into the engine's pools; a
verification overwrites the window positions with invariant values before
any of them is committed.

This is a comparator of the invariant path, not part of it: the GEMMs are
plain library GEMMs (gate and up as one [2F, H] weight, fp32 output
straight from cuBLAS where torch offers it), the rest are libbi's kernels.
"""
from __future__ import annotations

import math

import torch

from . import binding as bi


def _mm_f32_supported(dev) -> bool:
    try:
        a = torch.zeros(16, 16, dtype=torch.bfloat16, device=dev)
        torch.mm(a, a, out_dtype=torch.float32)
        return True
    except (TypeError, RuntimeError):
        return False


class FastPath:
    """Greedy decode of one row per request on the non-invariant path, over
    an Engine's weights, KV pools and page table."""

    def __init__(self, eng, max_batch: int):
        s = eng.shape
        self.eng, self.s = eng, s
        dev = eng.device
        self.dev = dev
        W = eng.w
        self.wgu = [torch.cat([lw["wg"], lw["wu"]]) for lw in W["layers"]]
        self.f32 = _mm_f32_supported(dev)
        B, H, D = max_batch, s.hidden, s.head_dim
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.x = torch.empty(B, H, **bf)
        self.h = torch.empty(B, H, **bf)
        self.q = torch.empty(B, s.n_heads, D, **bf)
        self.a = torch.empty(B, s.n_heads, D, **bf)
        self.kvl = torch.empty(B, dtype=torch.int32, device=dev)
        self.ws = torch.empty(bi.bi_decode_attn_workspace_size(
            B, s.n_heads, D, eng.max_kv_len) // 4 + 64, dtype=torch.float32,
            device=dev)
        self.scale = 1.0 / math.sqrt(D)

    def _mm(self, x, w):
        """x w^T with an fp32 result (the library's norm and RoPE read fp32)."""
        if self.f32:
            return torch.mm(x, w.t(), out_dtype=torch.float32)
        return torch.mm(x, w.t()).float()

    def decode(self, tokens, pos, slots, ids, max_kv_len):
        """tokens, pos, slots: device int32 [B]; ids: int32 [B] receives
        the greedy tokens.  Returns the fp32 logits [B][V].  Pages must
        cover every position."""
        s, eng = self.s, self.eng
        B = tokens.numel()
        H, F, D = s.hidden, s.ffn, s.head_dim
        x, h = self.x[:B], self.h[:B]
        q, a = self.q[:B], self.a[:B]
        kvl = self.kvl[:B]
        W = eng.w
        bi.bi_embed(tokens, W["embed"], h)
        torch.add(pos, 1, out=kvl)
        d = None
        for l, lw in enumerate(W["layers"]):
            bi.bi_rmsnorm(d, 0 if d is None else 1, None, h, lw["attn_norm"],
                          B, H, s.eps, x)
            qkv = self._mm(x, lw["wqkv"])
            bi.bi_rope(qkv, 1, pos, slots, s.n_heads, s.n_kv_heads, D,
                       s.theta, q, eng.k_pool[l], eng.v_pool[l],
                       eng.page_table)
            bi.bi_paged_decode_attn(q, eng.k_pool[l], eng.v_pool[l],
                                    eng.page_table, slots, kvl, max_kv_len,
                                    self.scale, a, self.ws)
            o = self._mm(a.view(B, -1), lw["wo"])
            bi.bi_rmsnorm(o, 1, None, h, lw["ffn_norm"], B, H, s.eps, x)
            gu = torch.mm(x, self.wgu[l].t())
            f = torch.nn.functional.silu(gu[:, :F]) * gu[:, F:]
            d = self._mm(f, lw["wd"])
        bi.bi_rmsnorm(d, 1, None, h, W["final_norm"], B, H, s.eps, x)
        logits = self._mm(x, W["lm_head"])
        bi.bi_argmax_logits(logits, ids)
        return logits
