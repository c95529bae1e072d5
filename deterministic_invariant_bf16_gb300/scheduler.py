"""Selective determinism with verified speculation (LLM-42).

"LLM-42: Enabling Determinism in LLM Inference with Verified Speculation"
(section 核心方法; paper sections 4.1-4.3, Fig. 8): every request decodes
on the fast, non-invariant path; only requests flagged deterministic have
their tokens treated as candidates, which a fixed-shape invariant
recomputation verifies in groups: windows of several requests packed
first-in first-out into one 256-row batch.  Each verified request commits
the prefix of its window that the recomputation reproduces; at the first
mismatch the rest is dropped and the KV cache is cut back to the committed
prefix (verify_commit_rollback).

Host bookkeeping only: the fast path (FastPath), the invariant prefill and
the verification (Engine) run in the library's kernels and in cuBLAS.

Per request the committed tokens are kept, and the cache holds all but the
last of them.  A flagged request's fast-path tokens accumulate as
candidates after its committed tokens (their K and V in the cache from the
fast path); at `window` candidates (or when the request's output budget is
reached) its window joins the next verify batch.  After a rollback at
candidate j the verifier's own token at j -- the invariant path's next
token -- becomes the first candidate of the next window, and the request
spends one fast-path step recomputing the K and V of its last committed
position (the cut dropped them) before it continues from that token.  So a
flagged request's output is exactly the invariant greedy output, whatever
the fast path produces; an unflagged request keeps the fast path's tokens.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import binding as bi


@dataclass
class Request:
    slot: int
    tokens: list              # committed tokens: prompt, then outputs
    n_prompt: int
    max_new: int
    deterministic: bool
    cand: list = field(default_factory=list)   # unverified candidates
    repair: bool = False      # next fast step recomputes the last position
    fix: int = -1             # the verifier's token after a rollback

    @property
    def n_out(self):
        return len(self.tokens) - self.n_prompt

    @property
    def done(self):
        return self.n_out >= self.max_new


class SelectiveScheduler:
    """Mixed deterministic and ordinary traffic over one Engine.

    engine: the invariant Engine (prefill, verification, pages);
    fast: a FastPath over the same engine;
    window: candidates per verify window (at most 256);
    perturb: optional callable (request, token) -> token applied to a
    flagged request's fast-path tokens (forces mismatches in tests and
    benchmarks)."""

    def __init__(self, engine, fast, window=32, perturb=None):
        assert 1 <= window <= bi.VERIFY_ROWS
        self.eng, self.fast = engine, fast
        self.window = window
        self.perturb = perturb
        self.reqs = []
        self.verify_log = []   # per verify call: (slots, kv, last, windows,
        #                        commit, fix, verify logits on the host)
        self.keep_logits = False
        self.stats = dict(verify_calls=0, windows=0, rollbacks=0,
                          committed=0, recomputed=0, fast_steps=0)
        dev = engine.device
        self.vlogits = torch.empty(bi.VERIFY_ROWS, engine.shape.vocab,
                                   dtype=torch.float32, device=dev)

    # ------------------------------------------------------------ intake --

    def add(self, slot, prompt, deterministic, max_new):
        """Prefill the prompt on the invariant path (LLM-42 keeps prefill
        deterministic) and commit its greedy next token."""
        prompt = [int(t) for t in prompt]
        eng = self.eng
        eng.reserve(slot, len(prompt) + 1)
        lg = eng.prefill([(slot, prompt, 0)])
        ids = torch.empty(1, dtype=torch.int32, device=eng.device)
        bi.bi_argmax_logits(lg[-1:].contiguous(), ids)
        r = Request(slot=slot, tokens=prompt + [int(ids.item())],
                    n_prompt=len(prompt), max_new=max_new,
                    deterministic=bool(deterministic))
        self.reqs.append(r)
        return r

    def adopt(self, slot, history, deterministic, max_new):
        """Take over a request whose cache already holds every token of
        `history` but the last (pages reserved), e.g. one caught in the
        middle of its output; `max_new` more tokens are produced."""
        r = Request(slot=slot, tokens=[int(t) for t in history],
                    n_prompt=len(history), max_new=max_new,
                    deterministic=bool(deterministic))
        self.reqs.append(r)
        return r

    # -------------------------------------------------------------- steps --

    def _fast_rows(self):
        """(request, input token, position) of this step's fast-path rows."""
        rows = []
        for r in self.reqs:
            if r.done:
                continue
            if r.deterministic:
                if r.repair:
                    rows.append((r, r.tokens[-1], len(r.tokens) - 1))
                    continue
                if r.n_out + len(r.cand) >= r.max_new:
                    continue   # waiting for verification
                if len(r.cand) >= self.window:
                    continue
                last = r.cand[-1] if r.cand else r.tokens[-1]
                rows.append((r, last, len(r.tokens) - 1 + len(r.cand)))
            else:
                rows.append((r, r.tokens[-1], len(r.tokens) - 1))
        return rows

    def step(self):
        """One fast-path decode iteration of every request that can take
        one, then the verification of every full window.  Returns False
        when every request is done."""
        rows = self._fast_rows()
        eng = self.eng
        if rows:
            for r, _, p in rows:
                eng.reserve(r.slot, p + 2)
            dev = eng.device
            tok = torch.tensor([t for _, t, _ in rows], dtype=torch.int32,
                               device=dev)
            pos = torch.tensor([p for _, _, p in rows], dtype=torch.int32,
                               device=dev)
            slots = torch.tensor([r.slot for r, _, _ in rows],
                                 dtype=torch.int32, device=dev)
            ids = torch.empty(len(rows), dtype=torch.int32, device=dev)
            self.fast.decode(tok, pos, slots, ids,
                             max(p for _, _, p in rows) + 1)
            out = ids.cpu().numpy()
            self.stats["fast_steps"] += 1
            for (r, _, _), t in zip(rows, out):
                t = int(t)
                if not r.deterministic:
                    r.tokens.append(t)
                elif r.repair:
                    # the committed last position's K and V are back; the
                    # verifier's token is the next candidate
                    r.repair = False
                    r.cand = [r.fix]
                else:
                    r.cand.append(self.perturb(r, t) if self.perturb else t)
        self._verify_ready(force=not rows)
        return not all(r.done for r in self.reqs)

    def run(self, max_steps=100000):
        for _ in range(max_steps):
            if not self.step():
                return
        raise RuntimeError("scheduler did not finish")

    # ------------------------------------------------------ verification --

    def _verify_ready(self, force=False):
        ready = [r for r in self.reqs
                 if r.deterministic and not r.done and r.cand and not r.repair
                 and (len(r.cand) >= self.window or
                      r.n_out + len(r.cand) >= r.max_new or force)]
        while ready:
            batch, used = [], 0
            for r in ready:
                if used + len(r.cand) > bi.VERIFY_ROWS:
                    break
                batch.append(r)
                used += len(r.cand)
            ready = ready[len(batch):]
            self._verify(batch)

    def _verify(self, batch):
        eng = self.eng
        slots = [r.slot for r in batch]
        kv = [len(r.tokens) - 1 for r in batch]
        last = [r.tokens[-1] for r in batch]
        wins = [list(r.cand) for r in batch]
        taken, commit, fix, _ = eng.verify(slots, kv, last, wins,
                                           logits=self.vlogits)
        assert taken == len(batch)
        if self.keep_logits:
            self.verify_log.append((slots, kv, last, wins, commit.copy(),
                                    fix.copy(), self.vlogits.cpu().numpy()))
        st = self.stats
        st["verify_calls"] += 1
        for r, j, f, w in zip(batch, commit, fix, wins):
            j = int(j)
            st["windows"] += 1
            st["committed"] += j
            r.tokens += w[:j]
            r.cand = []
            if j < len(w):
                st["rollbacks"] += 1
                st["recomputed"] += len(w) - j
                if not r.done:
                    r.repair, r.fix = True, int(f)
            r.tokens = r.tokens[:r.n_prompt + r.max_new]

    def outputs(self):
        return {r.slot: r.tokens[r.n_prompt:] for r in self.reqs}
