"""A thin caller of the C ABI for whole-model work: owns the device buffers
(weights, paged KV pools, page table, workspace) through torch, and calls
bi_model_forward / verify_commit_rollback.  No arithmetic happens here;
every step of the forward pass runs in libbi's kernels.

Page management is host bookkeeping: pages are handed out from a shuffled
free list, so a request's logical pages land in random physical order
(the layout the kernels must be invariant to; Vosti abstract).
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import binding as bi
from .synth import PAGE_SIZE, ModelShape


class PageAllocator:
    """Free list of physical page ids, drawn in a seeded random order, with
    a reference count per page in use: a page shared by several requests'
    page tables (a common prefix) returns to the free list when the last
    of them gives it back."""

    def __init__(self, n_pages: int, seed: int = 0):
        self.free = list(np.random.default_rng(seed).permutation(n_pages))
        self.refs = {}

    def take(self, n: int):
        if n > len(self.free):
            raise RuntimeError("KV pool exhausted (%d pages asked, %d free)"
                               % (n, len(self.free)))
        out, self.free = self.free[:n], self.free[n:]
        out = [int(p) for p in out]
        for p in out:
            self.refs[p] = 1
        return out

    def share(self, pages):
        for p in pages:
            p = int(p)
            if p not in self.refs:
                raise RuntimeError("page %d is not in use" % p)
            self.refs[p] += 1

    def give_back(self, pages):
        for p in pages:
            p = int(p)
            n = self.refs.get(p, 0)
            if n <= 0:
                raise RuntimeError("page %d given back but not in use" % p)
            if n == 1:
                del self.refs[p]
                self.free.append(p)
            else:
                self.refs[p] = n - 1


class PrefixIndex:
    """Token-keyed index of cached KV prefixes in whole pages.

    KV is bound to its logical prefix: with batch- and query-length-
    invariant kernels the K and V of positions [0, 16 k) depend only on the
    tokens there, not on the request, batch or step that computed them
    (Vosti abstract: cached KV tied to its logical token prefix, a paged
    prefix-sharing KV cache).  So a new request whose first 16 k tokens
    equal a cached request's may point its page table at that request's
    first k pages.  Only full pages are shared; the position after a shared
    prefix always starts a page of the new request's own."""

    def __init__(self):
        self.by_prefix = {}   # tokens of a whole-page prefix -> [slots]

    def add(self, slot: int, tokens):
        """Record the whole-page prefixes of `tokens` (the slot's committed
        KV) as available from `slot`."""
        t = tuple(int(x) for x in tokens)
        for k in range(1, len(t) // PAGE_SIZE + 1):
            owners = self.by_prefix.setdefault(t[:k * PAGE_SIZE], [])
            if slot not in owners:
                owners.append(slot)

    def drop(self, slot: int):
        """Forget `slot` (before its pages are released)."""
        for key in list(self.by_prefix):
            owners = self.by_prefix[key]
            if slot in owners:
                owners.remove(slot)
                if not owners:
                    del self.by_prefix[key]

    def lookup(self, tokens):
        """(slot, n_positions) of the longest cached whole-page prefix of
        `tokens` (its earliest recorded owner), or (None, 0)."""
        t = tuple(int(x) for x in tokens)
        for k in range(len(t) // PAGE_SIZE, 0, -1):
            owners = self.by_prefix.get(t[:k * PAGE_SIZE])
            if owners:
                return owners[0], k * PAGE_SIZE
        return None, 0


class Engine:
    def __init__(self, shape: ModelShape, weights: dict, *, max_tokens: int,
                 max_kv_len: int, n_slots: int, n_pages: int,
                 page_seed: int = 0, device="cuda"):
        self.shape = shape
        self.device = device
        self.max_tokens = max_tokens
        self.max_kv_len = max_kv_len
        self.max_pages = -(-max_kv_len // PAGE_SIZE)
        self.n_pages = n_pages
        s = shape
        self.w = weights
        self.wgu = []
        for lw in weights["layers"]:
            wgu = torch.empty(2 * s.ffn, s.hidden, dtype=torch.bfloat16,
                              device=device)
            bi.bi_pack_gate_up(lw["wg"], lw["wu"], wgu)
            self.wgu.append(wgu)
        L = len(weights["layers"])
        pool_shape = (n_pages, s.n_kv_heads, PAGE_SIZE, s.head_dim)
        self.k_pool = [torch.zeros(pool_shape, dtype=torch.bfloat16,
                                   device=device) for _ in range(L)]
        self.v_pool = [torch.zeros(pool_shape, dtype=torch.bfloat16,
                                   device=device) for _ in range(L)]
        self.page_table = torch.full((n_slots, self.max_pages), -1,
                                     dtype=torch.int32, device=device)
        self.kv_len = torch.zeros(n_slots, dtype=torch.int32, device=device)
        self.host_table = np.full((n_slots, self.max_pages), -1, np.int32)
        self.alloc = PageAllocator(n_pages, page_seed)
        self.cfg = bi.ModelCfg(
            n_layers=L, hidden=s.hidden, n_heads=s.n_heads,
            n_kv_heads=s.n_kv_heads, head_dim=s.head_dim, ffn=s.ffn,
            vocab=s.vocab, eps=s.eps, theta=s.theta, max_tokens=max_tokens,
            max_kv_len=max_kv_len, max_pages=self.max_pages, n_pages=n_pages)
        nbytes = bi.bi_model_workspace_size(self.cfg)
        if nbytes == 0:
            raise bi.BiError(1, "unsupported model configuration")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)

        def ptrs(ts):
            arr = (ctypes.c_void_p * L)(*[t.data_ptr() for t in ts])
            return ctypes.cast(arr, bi.PP), arr

        lays = weights["layers"]
        self._keep = []
        fields = {}
        for name, ts in [("attn_norm", [l["attn_norm"] for l in lays]),
                         ("wqkv", [l["wqkv"] for l in lays]),
                         ("wo", [l["wo"] for l in lays]),
                         ("ffn_norm", [l["ffn_norm"] for l in lays]),
                         ("wgu", self.wgu),
                         ("wd", [l["wd"] for l in lays]),
                         ("k_pool", self.k_pool), ("v_pool", self.v_pool)]:
            p, arr = ptrs(ts)
            self._keep.append(arr)
            fields[name] = p
        self.wstruct = bi.ModelWeights(
            embed=weights["embed"].data_ptr(),
            final_norm=weights["final_norm"].data_ptr(),
            lm_head=weights["lm_head"].data_ptr(), **fields)
        self.handle = bi.bi_model_create(self.cfg, self.wstruct, self.ws)

    def close(self):
        if self.handle is not None:
            bi.bi_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ pages --

    def reserve(self, slot: int, n_positions: int):
        """Make sure page-table row `slot` covers positions [0, n)."""
        need = -(-n_positions // PAGE_SIZE)
        row = self.host_table[slot]
        have = int((row >= 0).sum())
        if need > have:
            row[have:need] = self.alloc.take(need - have)
            self.page_table[slot, have:need] = torch.from_numpy(
                row[have:need].copy()).to(self.device)

    def set_pages(self, slot: int, pages):
        """Place explicit physical pages into a slot (layout tests)."""
        pages = np.asarray(pages, np.int32)
        self.host_table[slot, :] = -1
        self.host_table[slot, :len(pages)] = pages
        self.page_table[slot] = torch.from_numpy(self.host_table[slot].copy()
                                                 ).to(self.device)

    def share_prefix(self, src: int, dst: int, n_positions: int) -> int:
        """Point the first n_positions // 16 page-table entries of the empty
        slot `dst` at the pages holding positions [0, 16 k) of slot `src`
        (whose KV there must be committed and computed from the same
        tokens).  Returns 16 k, the first position `dst` must compute
        itself; its later pages are its own (reserve)."""
        k = n_positions // PAGE_SIZE
        src_row, dst_row = self.host_table[src], self.host_table[dst]
        if (dst_row >= 0).any():
            raise RuntimeError("slot %d is not empty" % dst)
        pages = src_row[:k]
        if (pages < 0).any():
            raise RuntimeError("slot %d has no pages for positions [0, %d)"
                               % (src, k * PAGE_SIZE))
        self.alloc.share(pages)
        dst_row[:k] = pages
        self.page_table[dst, :k] = torch.from_numpy(pages.copy()).to(
            self.device)
        return k * PAGE_SIZE

    def release(self, slot: int):
        row = self.host_table[slot]
        self.alloc.give_back(row[row >= 0])
        row[:] = -1
        self.page_table[slot] = -1

    def drop_pages(self, slot: int, pages):
        """Host bookkeeping after verify freed pages of a slot."""
        row = self.host_table[slot]
        row[np.isin(row, np.asarray(pages))] = -1
        self.alloc.give_back(pages)

    # ---------------------------------------------------------- forward --

    def _i32(self, a):
        return torch.as_tensor(np.asarray(a, np.int32)).to(self.device)

    def decode(self, tokens, positions, slots, logits=None, ids=None,
               max_kv_len=None, stream=None):
        """One row per request: token at absolute position, slot = page-table
        row.  Pages must already cover every position."""
        T = len(tokens)
        tok = tokens if torch.is_tensor(tokens) else self._i32(tokens)
        pos = positions if torch.is_tensor(positions) else self._i32(positions)
        rr = slots if torch.is_tensor(slots) else self._i32(slots)
        if logits is None:
            logits = torch.empty(T, self.shape.vocab, dtype=torch.float32,
                                 device=self.device)
        if max_kv_len is None:
            max_kv_len = int(pos.max().item()) + 1
        bi.bi_model_forward(self.handle, tok, pos, rr, None, None, 0,
                            max_kv_len, self.page_table, logits, ids, stream)
        return logits

    def capture(self, fn, warm=True):
        """Record the library calls that `fn()` makes as one CUDA graph
        and return it (`torch.cuda.CUDAGraph`; `.replay()` issues them
        again).  fn runs once first on a side stream (unless warm is
        False: everything fn touches already exists), then once under
        capture.  Every tensor fn passes must stay alive and be refilled in
        place between replays (tokens, positions, ids ...); fn must not
        read results on the host, so verify_commit_rollback, which does,
        stays outside.  A decode iteration captured this way launches the
        same kernels with the same arguments, so its results are those of
        the eager calls bit for bit."""
        dev = torch.device(self.device)
        torch.cuda.synchronize(dev)
        if warm:
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                fn()
            torch.cuda.current_stream(dev).wait_stream(side)
            torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        torch.cuda.synchronize(dev)
        return graph

    def prefill(self, segments, logits=None, ids=None, stream=None):
        """segments: list of (slot, tokens, first_position).  Rows of a
        segment take consecutive positions."""
        toks, pos, rr, cu, sr = [], [], [], [0], []
        max_q = 1
        max_kv = 1
        for slot, t, p0 in segments:
            n = len(t)
            toks += list(t)
            pos += list(range(p0, p0 + n))
            rr += [slot] * n
            cu.append(cu[-1] + n)
            sr.append(slot)
            max_q = max(max_q, n)
            max_kv = max(max_kv, p0 + n)
        T = len(toks)
        if logits is None:
            logits = torch.empty(T, self.shape.vocab, dtype=torch.float32,
                                 device=self.device)
        bi.bi_model_forward(self.handle, self._i32(toks), self._i32(pos),
                            self._i32(rr), self._i32(cu), self._i32(sr),
                            max_q, max_kv, self.page_table, logits, ids,
                            stream)
        return logits

    def verify(self, slots, kv_lens, last_tokens, windows, logits=None,
               stream=None):
        """LLM-42 grouped verification of candidate windows; returns
        (taken, commit_len, fix_token, freed_pages) and updates the page
        table and kv_len rows on the device."""
        if logits is None:
            logits = torch.empty(bi.VERIFY_ROWS, self.shape.vocab,
                                 dtype=torch.float32, device=self.device)
        cands = np.concatenate([np.asarray(w, np.int32) for w in windows])
        taken, commit, fix, freed = bi.verify_commit_rollback(
            self.handle, slots, kv_lens, last_tokens,
            [len(w) for w in windows], cands, self.page_table, self.kv_len,
            logits, freed_cap=self.max_pages * bi.VERIFY_ROWS, stream=stream)
        self.mirror_cut(slots, kv_lens, taken, commit)
        return taken, commit, fix, freed

    def verify_buffers(self):
        """Device plan and result buffers for verify_device."""
        return bi.VerifyBuffers(self.max_pages * bi.VERIFY_ROWS, self.device)

    def verify_device(self, bufs, logits, stream=None):
        """verify_commit_rollback_device on a plan already in ``bufs``: no
        host synchronisation, so a caller may capture it (Engine.capture).
        The page table and kv_len are cut on the device; once the results
        are read (``bufs.read()``), ``mirror_cut`` brings the host page
        bookkeeping in line."""
        bi.verify_commit_rollback_device(self.handle, bufs, self.page_table,
                                         self.kv_len, logits, stream)

    def mirror_cut(self, slots, kv_lens, taken, commit):
        """Mirror a verify's page-table cut in the host bookkeeping: pages
        at or past ceil((kv_len + commit) / 16) go back to the allocator."""
        for r in range(taken):
            keep = -(-(int(kv_lens[r]) + int(commit[r])) // PAGE_SIZE)
            row = self.host_table[slots[r]]
            gone = row[keep:][row[keep:] >= 0]
            row[keep:] = -1
            self.alloc.give_back(gone)

    def hidden(self, T):
        """The residual stream after the last forward of T rows: bf16
        [T][hidden], the last layer's output before the final RMSNorm
        (a view of the workspace, valid until the next forward)."""
        return bi.bi_model_hidden(self.handle, T, self.shape.hidden)


def to_device(weights: dict, device="cuda") -> dict:
    return dict(embed=weights["embed"].to(device),
                final_norm=weights["final_norm"].to(device),
                lm_head=weights["lm_head"].to(device),
                layers=[{k: v.to(device) for k, v in lw.items()}
                        for lw in weights["layers"]])
