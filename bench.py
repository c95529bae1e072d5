#!/usr/bin/env python3
"""Benchmark: batch-invariant decode tokens/s of a Llama-3.1-8B-shaped bf16
decoder on one GB300, with the roofline fraction of the dominant kernel.

Workload (LLM-42 grouped verification on the full 32-layer model; "LLM-42:
Enabling Determinism in LLM Inference with Verified Speculation", sections
4.3 and 5.1): 256 requests with ShareGPT-like lengths (prompts lognormal
median 256 clipped 4..2048, outputs lognormal median 200 clipped 16..1024;
each request is caught at a uniform point of its output), 10% of them flagged
deterministic.  Random-init weights N(0, 0.02); the KV cache of the already
processed tokens is N(0, 1) bf16 in randomly ordered 16-token pages.

One step = 10 invariant decode iterations of all 256 requests (greedy for
flagged requests, Philox temperature sampling keyed by (request, step) for
the rest) followed by one fixed 256-row grouped verification of 8 flagged
requests' 32-token candidate windows with commit and rollback.  Ten
iterations per verify is the ratio 10% deterministic traffic implies
(26 flagged requests x 10 tokens ~ one 256-row verify batch).  The metric
counts decoded tokens: 10 x 256 per step.

Run with no flags for one GPU.  Under torchrun (N > 1) every rank runs an
independent replica (the path has no exchange step) and the line reports the
aggregate over ranks with max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batch-invariant decode tok/s (8B-shape bf16) + % of tensor/HBM roofline"
UNIT = "tok/s"
WORKLOAD = "llm42-grouped-verify-8b-decode"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=256)
    ap.add_argument("--iters", type=int, default=10)
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--no-comparator", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--report", action="store_true",
                    help="instead of the step benchmark: decode tok/s over "
                         "batch sizes 1..256 and invariant prefill tok/s on "
                         "a sample of long prompts (one JSON line)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the decode iterations one call at a time "
                         "instead of replaying them as one CUDA graph")
    return ap.parse_args()


# ----------------------------------------------------------------- workload --

def make_workload(batch, iters, seed=1003):
    from deterministic_invariant_bf16_gb300 import synth
    rng = np.random.default_rng(seed)
    prompts = synth.lognormal_lengths(batch, 256, 1.0, 4, 2048, rng)
    outputs = synth.lognormal_lengths(batch, 200, 1.0, 16, 1024, rng)
    progress = rng.uniform(0.0, 1.0, size=batch)
    ctx = (prompts + np.floor(progress * outputs)).astype(np.int64)
    n_flag = max(1, int(round(0.10 * batch)))
    n_ver = min(8, n_flag)
    window = 256 // n_ver
    return dict(batch=batch, iters=iters, ctx=ctx, prompts=prompts,
                outputs=outputs, n_flag=n_flag, n_ver=n_ver, window=window,
                headroom=iters + window + 2,
                first_tokens=synth.token_ids(batch, synth.LLAMA8B.vocab, rng),
                rng=rng)


# ------------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clock and throttle-reason samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1])]
        mx = [num(r[2]) for r in rows if num(r[2])]
        power = [num(r[3]) for r in rows if num(r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------ helpers --

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"],
                    bf16_sus=p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


def src_hash(name):
    path = os.path.join(ROOT, "deterministic_invariant_bf16_gb300", "csrc",
                        name)
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def recorded_traffic(kernel_class):
    """Per-launch DRAM bytes from the committed ncu summary for this kernel
    class, or None when missing or when the kernel source has changed since
    the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(kernel_class)
    if not rec or rec.get("source_sha") != src_hash(rec["source"]):
        return None
    return rec.get("bytes_per_launch")


def aggregate(ms_local, tokens_per_step_per_rank, world, dist=None,
              device="cpu"):
    """Replicas: every rank decodes its own requests; the step time is the
    slowest rank's and the throughput counts every rank's tokens."""
    ms = float(ms_local)
    if world > 1 and dist is not None:
        import torch
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, tokens_per_step_per_rank * world / (ms / 1000.0)


# --------------------------------------------------------------- our arm ----

class Bench:
    def __init__(self, args, device, weights=None):
        import torch
        from deterministic_invariant_bf16_gb300 import binding as bi
        from deterministic_invariant_bf16_gb300 import engine, synth
        self.torch, self.bi = torch, bi
        self.args = args
        self.dev = device
        self.shape = synth.LLAMA8B
        wl = make_workload(args.batch, args.iters)
        self.wl = wl
        B, it = wl["batch"], wl["iters"]
        ctx = wl["ctx"]
        max_kv = int(ctx.max()) + wl["headroom"]
        need = int(sum(-(-(int(c) + wl["headroom"]) // 16) for c in ctx))
        self.weights = weights if weights is not None else \
            synth.make_weights(self.shape, 4, device, n_layers=args.layers)
        self.eng = engine.Engine(self.shape, self.weights, max_tokens=256,
                                 max_kv_len=max_kv, n_slots=B,
                                 n_pages=need + 64, page_seed=5)
        for r in range(B):
            self.eng.reserve(r, int(ctx[r]) + wl["headroom"])
        g = torch.Generator(device=device).manual_seed(6)
        for kp, vp in zip(self.eng.k_pool, self.eng.v_pool):
            kp.normal_(generator=g)
            vp.normal_(generator=g)
        i32 = dict(dtype=torch.int32, device=device)
        self.slots = torch.arange(B, **i32)
        self.tok0 = torch.from_numpy(wl["first_tokens"]).to(device)
        self.pos = torch.stack([torch.from_numpy(ctx + i).to(device).int()
                                for i in range(it)])
        self.maxkv = [int(ctx.max()) + i + 1 for i in range(it)]
        self.ids = torch.empty(it, B, **i32)
        self.logits = torch.empty(B, self.shape.vocab, dtype=torch.float32,
                                  device=device)
        self.vlogits = torch.empty(bi.VERIFY_ROWS, self.shape.vocab,
                                   dtype=torch.float32, device=device)
        self.rid = torch.arange(B, dtype=torch.int64, device=device) + 1000
        self.stepv = torch.stack([torch.from_numpy(ctx + i).to(device)
                                  for i in range(it)]).long()
        self.tau = 0.7
        self.n_flag = wl["n_flag"]
        self._make_candidates()

    def decode_iters(self, n=None):
        bi, eng = self.bi, self.eng
        F = self.n_flag
        for i in range(n or self.wl["iters"]):
            src = self.tok0 if i == 0 else self.ids[i - 1]
            eng.decode(src, self.pos[i], self.slots, logits=self.logits,
                       max_kv_len=self.maxkv[i])
            ids = self.ids[i]
            bi.bi_argmax_logits(self.logits[:F], ids[:F])
            bi.philox_sample(self.logits[F:], self.rid[F:],
                             self.stepv[i % len(self.stepv)][F:], self.tau,
                             ids[F:])

    def _make_candidates(self):
        """Candidate windows of the verified requests: their own invariant
        greedy continuation (32 decode iterations run once here), with each
        candidate perturbed with probability 0.003 to force mismatches."""
        wl = self.wl
        nv, w = wl["n_ver"], wl["window"]
        ctx = wl["ctx"]
        keep_pos, keep_maxkv = self.pos, self.maxkv
        self.pos = self.torch.stack([self.torch.from_numpy(ctx + i).to(
            self.dev).int() for i in range(w)])
        self.maxkv = [int(ctx.max()) + i + 1 for i in range(w)]
        keep_ids = self.ids
        self.ids = self.torch.empty(w, wl["batch"], dtype=self.torch.int32,
                                    device=self.dev)
        self.decode_iters(w)
        cand = self.ids[:, :nv].T.cpu().numpy().copy()
        self.pos, self.maxkv, self.ids = keep_pos, keep_maxkv, keep_ids
        rng = wl["rng"]
        flip = rng.uniform(size=cand.shape) < 0.003
        V = self.shape.vocab
        cand[flip] = (cand[flip] + 1 + rng.integers(0, V - 1, size=flip.sum())) % V
        self.cand = [list(map(int, c)) for c in cand]
        self.v_slots = list(range(nv))
        self.v_kv = [int(c) for c in ctx[:nv]]
        self.v_last = [int(t) for t in wl["first_tokens"][:nv]]
        self.commits = []

    def verify(self):
        wl = self.wl
        taken, commit, fix, freed = self.eng.verify(
            self.v_slots, self.v_kv, self.v_last, self.cand,
            logits=self.vlogits)
        self.commits.append((taken, commit.copy(), fix.copy()))
        for r in self.v_slots:  # pages for the next step's positions
            self.eng.reserve(r, int(wl["ctx"][r]) + wl["headroom"])

    def capture(self):
        """Capture one step's decode iterations (the library's calls, same
        buffers and arguments) as a CUDA graph through Engine.capture; the
        verify part syncs with the host and stays eager."""
        self.graph = self.eng.capture(self.decode_iters)

    def step(self, graph=False):
        if graph and getattr(self, "graph", None) is not None:
            self.graph.replay()
        else:
            self.decode_iters()
        self.verify()


def algorithmic_bytes(b, cls, launches_per_step):
    """Algorithmic bytes per launch of a kernel class in one step (HBM
    traffic an ideal kernel must move)."""
    wl, S = b.wl, b.shape
    B, it = wl["batch"], wl["iters"]
    H, F, D = S.hidden, S.ffn, S.head_dim
    Hq, Hkv = S.n_heads, S.n_kv_heads
    QKV = S.qkv_dim
    ctx = wl["ctx"]
    bi = b.bi
    if cls == "attn":
        # decode attention (chunks merged in registers): K and V of every
        # visible position, the queries in and the outputs out
        kv = sum(float((ctx + i + 1).sum()) for i in range(it)) / it
        return kv * Hkv * D * 2 * 2 + 2 * B * Hq * D * 2
    if cls == "attn_merge":
        chunks = sum(float(np.ceil((ctx + i + 1) / 256).sum())
                     for i in range(it)) / it
        return chunks * Hq * (D + 4) * 4 + B * Hq * D * 2
    # Algorithmic bytes count each tensor the step must read or write once:
    # a GEMM reads its weight and input and writes its fp32 (or bf16)
    # result; split-K slices are an implementation choice and not counted.
    if cls == "rope":
        # the fp32 q/k/v row in, q out, k and v appended to the cache
        return B * QKV * 4.0 + B * QKV * 2.0
    if cls == "norm":
        # per forward: the first attention norm reads the embedded rows; each
        # later norm reads the fp32 projection output, updates the residual
        # and writes y
        Lr = b.args.layers
        per_fwd = (B * H * 4.0 + 2 * Lr * (B * H * 4.0 + 3 * B * H * 2.0))
        return per_fwd / (2 * Lr + 1)
    gemms = {"gemm_qkv": (QKV, H), "gemm_o": (H, Hq * D),
             "gemm_gate_up": (2 * F, H), "gemm_down": (H, F),
             "lm_head": (S.vocab, H)}
    if cls in gemms:
        N, K = gemms[cls]
        out = B * N // 2 * 2 if cls == "gemm_gate_up" else B * N * 4
        return 2.0 * N * K + 2.0 * B * K + out
    return None


def gemm_flops(b, cls):
    S = b.shape
    B = b.wl["batch"]
    dims = {"gemm_qkv": (S.qkv_dim, S.hidden), "gemm_o": (S.hidden, S.q_dim),
            "gemm_gate_up": (2 * S.ffn, S.hidden),
            "gemm_down": (S.hidden, S.ffn), "lm_head": (S.vocab, S.hidden)}
    if cls not in dims:
        return None
    N, K = dims[cls]
    return 2.0 * B * N * K


def verify_stats(b, ms):
    """The step's grouped verification: windows, rollbacks (windows cut
    before their end), candidates recomputed (those after the first
    mismatch) and the committed output rate of the step (decoded tokens of
    the unverified rows plus the committed tokens of the verified ones)."""
    wl = b.wl
    w = wl["window"]
    commit = [int(x) for x in b.commits[-1][1]]
    committed = sum(commit)
    recomputed = sum(w - j for j in commit)
    out_tokens = (wl["batch"] - wl["n_ver"]) * wl["iters"] + committed
    return {"windows": len(commit), "window": w,
            "rollbacks": sum(1 for j in commit if j < w),
            "committed": committed, "recomputed": recomputed,
            "recompute_fraction": recomputed / float(len(commit) * w),
            "committed_tok_s": out_tokens / (ms / 1000.0)}


def run_report(args):
    """Decode tok/s over batch sizes (the same step workload at each B,
    decode iterations replayed as a CUDA graph, no verify) and invariant
    prefill tok/s on long prompts (8 requests, prompts U[4096, 8192], each
    prefilled in 2048-token pieces).  Synthetic inputs, random weights."""
    import copy
    import torch
    from deterministic_invariant_bf16_gb300 import binding as bi
    from deterministic_invariant_bf16_gb300 import build, engine, synth
    build.build()
    bi.lib()
    dev = "cuda:0"
    torch.cuda.set_device(0)
    shape = synth.LLAMA8B
    W = synth.make_weights(shape, 4, dev, n_layers=args.layers)
    rep = {"decode_tok_s": {}, "layers": args.layers}
    for B in (1, 8, 32, 64, 128, 256):
        a = copy.copy(args)
        a.batch = B
        b = Bench(a, dev, weights=W)
        b.capture()
        for _ in range(3):
            b.graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            b.graph.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        rep["decode_tok_s"][str(B)] = B * b.wl["iters"] / (ms / 1000.0)
        del b
        torch.cuda.empty_cache()
    # LLM-42 with the cuBLAS path as the fast path (B = 256)
    a = copy.copy(args)
    a.batch = 256
    b = Bench(a, dev, weights=W)
    rep["llm42_fast_path"] = fast_path_report(b)
    del b
    torch.cuda.empty_cache()
    # prefill
    rng = np.random.default_rng(1005)
    R, piece = 8, 2048
    prompts = rng.integers(4096, 8193, size=R)
    max_kv = int(prompts.max()) + 16
    need = int(sum(-(-int(p) // 16) for p in prompts)) + 64
    eng = engine.Engine(shape, W, max_tokens=piece, max_kv_len=max_kv,
                        n_slots=R, n_pages=need, page_seed=7)
    for r in range(R):
        eng.reserve(r, int(prompts[r]))
    toks = [synth.token_ids(int(p), shape.vocab, rng) for p in prompts]
    logits = torch.empty(piece, shape.vocab, dtype=torch.float32, device=dev)

    def prefill_all():
        for r in range(R):
            for p0 in range(0, int(prompts[r]), piece):
                t = toks[r][p0:p0 + piece]
                eng.prefill([(r, t, p0)], logits=logits[:len(t)])

    prefill_all()  # warm-up
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    prefill_all()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    rep["prefill"] = {"tok_s": float(prompts.sum()) / (ms / 1000.0),
                      "requests": R, "tokens": int(prompts.sum()),
                      "piece": piece, "ms": ms}
    del eng, logits
    torch.cuda.empty_cache()
    rep["prefix_sharing"] = prefix_report(torch, bi, engine, synth, shape, W,
                                          dev, piece)
    rep["gemm_sweep"] = gemm_sweep(torch, bi, dev)
    rep["device_status"] = bi.bi_device_status()
    # the oracle's own timings (CPU baseline) beside the GPU numbers
    rep["cpu_baseline_configs"] = oracle_configs()
    print(json.dumps({"report": rep, "workload": WORKLOAD,
                      "data": "synthetic (random-init weights, random KV)"}),
          flush=True)


def prefix_report(torch, bi, engine, synth, shape, W, dev, piece):
    """8 prompts = one common 4096-token prefix + 256 tokens of their own,
    prefilled (a) each from scratch and (b) with the prefix computed once
    and its 256 pages shared (Engine.share_prefix); the last-row logits of
    every prompt must be bitwise equal between (a) and (b)."""
    rng = np.random.default_rng(1006)
    R, P, U = 8, 4096, 256
    common = synth.token_ids(P, shape.vocab, rng)
    toks = [np.concatenate([common, synth.token_ids(U, shape.vocab, rng)])
            for _ in range(R)]
    per = (P + U) // 16
    eng = engine.Engine(shape, W, max_tokens=piece, max_kv_len=P + U + 16,
                        n_slots=2 * R, n_pages=R * per + per +
                        (R - 1) * (U // 16) + 32, page_seed=9)
    logits = torch.empty(piece, shape.vocab, dtype=torch.float32, device=dev)
    last = torch.empty(2, R, shape.vocab, dtype=torch.float32, device=dev)
    for r in range(R + 1):
        eng.reserve(r, P + U)

    def fill(slot, t, p0, out):
        for q in range(p0, P + U, piece):
            c = t[q:q + piece]
            eng.prefill([(slot, c, q)], logits=logits[:len(c)])
        out.copy_(logits[len(c) - 1])

    def scratch():
        for r in range(R):
            fill(r, toks[r], 0, last[0, r])

    def shared():
        fill(R, toks[0], 0, last[1, 0])
        for r in range(1, R):
            start = eng.share_prefix(R, R + r, P)
            eng.reserve(R + r, P + U)
            fill(R + r, toks[r], start, last[1, r])

    scratch()  # warm-up
    out = {"requests": R, "prefix": P, "own": U, "piece": piece}
    for name, fn in (("scratch", scratch), ("shared", shared)):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        out[name + "_ms"] = ms
        out[name + "_prompt_tok_s"] = R * (P + U) / (ms / 1000.0)
    out["bitwise_equal"] = bool(torch.equal(last[0].view(torch.int32),
                                            last[1].view(torch.int32)))
    return out


def gemm_sweep(torch, bi, dev):
    """bi_gemm at the GEMM sweep's shapes: M = 1 .. 256 against a 4096 x 4096
    weight, and at M = 256 the literal 14336 x 14336, the FFN shapes and the
    LM head.  Split partials out (as the model uses it), weights cycled over
    copies larger than L2, 20 launches per CUDA graph."""
    import math
    x = (torch.randn(256, 14336, device=dev) * 0.5).bfloat16()
    out = torch.empty(8 * 256 * 128256, dtype=torch.float32, device=dev)
    res = {}
    cases = [(m, 4096, 4096) for m in (1, 2, 4, 8, 16, 32, 64, 128, 256)] + \
        [(256, 14336, 14336), (256, 14336, 4096), (256, 4096, 14336),
         (256, 128256, 4096)]
    Ws, key = None, None
    for M, N, K in cases:
        if key != (N, K):
            Ws = None
            torch.cuda.empty_cache()
            n = max(2, math.ceil(400e6 / (N * K * 2)))
            Ws = [(torch.randn(N, K, device=dev) * 0.02).bfloat16()
                  for _ in range(n)]
            key = (N, K)
        xm = x[:M, :K].contiguous()

        def run():
            for i in range(20):
                bi.bi_gemm(xm, Ws[i % len(Ws)], out, bi.OUT_PARTIALS)

        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            run()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / 60 * 1e3
        wbytes = 2.0 * N * K + 2.0 * M * K + 4.0 * M * N
        res["%dx%dx%d" % (M, N, K)] = {
            "us": us, "GBps": wbytes / us / 1e3,
            "TFLOPs": 2.0 * M * N * K / us / 1e6,
            "splits": bi.bi_gemm_splits(N, K)}
    del Ws
    torch.cuda.empty_cache()
    return res


def oracle_configs():
    """The oracle as it stands on the host cores, beside the GPU numbers:
    the 4096 x 4096 GEMM at M = 1, 8, 256; one 8B-shape decoder layer for
    B = 1, 8, 32 decode rows (contexts from the step workload's
    distribution); the tiny decoder's greedy run (8 requests, 16-token
    prompts, 16 new tokens)."""
    import oracle
    from deterministic_invariant_bf16_gb300 import synth
    rng = np.random.default_rng(11)
    cores = len(os.sched_getaffinity(0))
    out = {"cores": cores, "kind": "oracle", "gemm_4096": {}, "layer_8b": {}}
    w = oracle.bf16_bits(rng.normal(0, 0.02, (4096, 4096)).astype(np.float32))
    for M in (1, 8, 256):
        x = oracle.bf16_bits(rng.normal(0, 1, (M, 4096)).astype(np.float32))
        t0 = time.perf_counter()
        oracle.gemm(x, w)
        t = time.perf_counter() - t0
        out["gemm_4096"][str(M)] = {"s": t, "GFLOPs": 2 * M * 4096 * 4096 / t / 1e9}
    S = synth.LLAMA8B
    cfg = oracle.Cfg(n_layers=1, hidden=S.hidden, n_heads=S.n_heads,
                     n_kv_heads=S.n_kv_heads, head_dim=S.head_dim, ffn=S.ffn,
                     vocab=256, eps=S.eps, theta=S.theta)
    lw = oracle_weights()["layer"]
    for B in (1, 8, 32):
        L = synth.lognormal_lengths(B, 512, 1.0, 16, 4096, rng)
        Lm = int(L.max())
        kc = oracle.bf16r(rng.standard_normal((B, Lm, S.n_kv_heads, S.head_dim),
                                              np.float32))
        vc = oracle.bf16r(rng.standard_normal(kc.shape, np.float32))
        h = oracle.bf16r(rng.standard_normal((B, S.hidden), np.float32))
        t0 = time.perf_counter()
        oracle.decoder_layer(h, np.arange(B, dtype=np.int32),
                             (L - 1).astype(np.int32), lw, kc, vc, cfg)
        t = time.perf_counter() - t0
        out["layer_8b"][str(B)] = {"s": t, "rows_per_s": B / t}
    tiny = synth.TINY
    import torch
    tw = synth.make_weights(tiny, 0, "cpu")

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    ow = dict(embed=u16(tw["embed"]), final_norm=u16(tw["final_norm"]),
              lm_head=u16(tw["lm_head"]),
              layers=[{k: u16(v) for k, v in lw_.items()}
                      for lw_ in tw["layers"]])
    prompts = [synth.token_ids(16, tiny.vocab, rng) for _ in range(8)]
    t0 = time.perf_counter()
    oracle.greedy_decode(prompts, 16, ow, oracle.Cfg())
    t = time.perf_counter() - t0
    out["tiny_greedy"] = {"s": t, "tok_s": 8 * 16 / t}
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = "cuda:%d" % local
    from deterministic_invariant_bf16_gb300 import binding as bi
    from deterministic_invariant_bf16_gb300 import build
    build.build()
    bi.lib()
    b = Bench(args, dev)
    B, it = b.wl["batch"], b.wl["iters"]
    tokens_per_step = B * it

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        b.step()
    torch.cuda.synchronize()
    use_graph = not args.no_graph
    if use_graph:
        b.capture()
        b.step(graph=True)
        torch.cuda.synchronize()
    # ---- device-resident timed region (inputs are in HBM: weights 16 GB,
    # KV ~20 GB, far beyond the 129 MB L2, so no flush is needed)
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    e0.record(stream)
    for _ in range(args.steps):
        b.step(graph=use_graph)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    # ---- the same steps again with every kernel launch of the forward
    # bracketed by CUDA events on its stream (per-kernel time for the
    # roofline); kept out of the headline region above.
    bi.bi_model_profile(b.eng.handle, True)
    ep0 = torch.cuda.Event(enable_timing=True)
    ep1 = torch.cuda.Event(enable_timing=True)
    ep0.record(stream)
    for _ in range(args.steps):
        b.step()
    ep1.record(stream)
    torch.cuda.synchronize()
    ms_profiled = ep0.elapsed_time(ep1) / args.steps
    prof = bi.bi_model_profile_read(b.eng.handle)
    bi.bi_model_profile(b.eng.handle, False)
    status = bi.bi_device_status()
    ms, value = aggregate(ms, tokens_per_step, world,
                          dist if world > 1 else None, dev)

    # ---- end to end through the public API with host buffers: every step
    # uploads its inputs from pinned host memory into the buffers the
    # decode graph (Engine.capture) reads, replays it, runs the verify
    # group, and reads back the tokens.
    h_in_tok = b.tok0.cpu().pin_memory()
    h_in_pos = b.pos.cpu().pin_memory()
    h_in_step = b.stepv.cpu().pin_memory()
    h_out = torch.empty(it, B, dtype=torch.int32).pin_memory()
    bytes_in = (h_in_tok.numel() * 4 + h_in_pos.numel() * 4 +
                h_in_step.numel() * 8)
    bytes_out = h_out.numel() * 4
    barrier()
    torch.cuda.synchronize()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.steps):
        b.tok0.copy_(h_in_tok, non_blocking=True)
        b.pos.copy_(h_in_pos, non_blocking=True)
        b.stepv.copy_(h_in_step, non_blocking=True)
        b.step(graph=use_graph)
        h_out.copy_(b.ids, non_blocking=True)
        stream.synchronize()
    e3.record(stream)
    torch.cuda.synchronize()
    ms_e2e, v_e2e = aggregate(e2.elapsed_time(e3) / args.steps,
                              tokens_per_step, world,
                              dist if world > 1 else None, dev)
    e2e = {"value": v_e2e, "unit": UNIT,
           "h2d_bytes_per_step": bytes_in,
           "d2h_bytes_per_step": bytes_out + 3 * 4 * b.wl["n_ver"]}

    # ---- roofline of the dominant kernel (largest share of device time)
    pk = peaks()
    shares = {k: v[0] for k, v in prof.items()
              if v[1] > 0 and algorithmic_bytes(b, k, v[1]) is not None}
    dom = max(shares, key=shares.get)
    n_launch = prof[dom][1]
    avg_ms = prof[dom][0] / n_launch
    flops = gemm_flops(b, dom)
    ab = algorithmic_bytes(b, dom, n_launch / args.steps)
    hbm_time = ab / (pk["hbm"] * 1e9) if ab else 0.0
    ten_time = flops / (pk["bf16_sus"] * 1e12) if flops else 0.0
    if flops and ten_time > hbm_time:
        ach = flops / (avg_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": pk["bf16_sus"],
                "unit": "TFLOP/s", "frac": ach / pk["bf16_sus"]}
    else:
        ach = ab / (avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm"],
                "unit": "GB/s", "frac": ach / pk["hbm"]}
    roof["traffic"] = recorded_traffic(dom)
    roof["kernel"] = dom
    roof["peak_source"] = pk["source"]
    roof["algorithmic_bytes_per_launch"] = ab
    roof["avg_launch_ms"] = avg_ms
    total_ms = sum(v[0] for v in prof.values())
    kernels = {}
    for k, (kms, cnt) in prof.items():
        if cnt == 0:
            continue
        entry = {"ms_per_step": kms / args.steps, "launches_per_step":
                 cnt / args.steps, "share": kms / total_ms}
        abk = algorithmic_bytes(b, k, cnt / args.steps)
        if abk:
            entry["GBps"] = abk / (kms / cnt / 1e3) / 1e9
            entry["hbm_frac"] = entry["GBps"] / pk["hbm"]
        fl = gemm_flops(b, k)
        if fl:
            entry["TFLOPs"] = fl / (kms / cnt / 1e3) / 1e12
        kernels[k] = entry

    launches = sum(v[1] for v in prof.values()) / args.steps
    # kernels the profile does not bracket: per decode iteration the
    # kv-length setup, the greedy argmax and the Philox sampler; per verify
    # the commit kernel.  Every bracketed class is one kernel per launch.
    launches += 3 * it + 1
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (random-init weights, random KV)",
        "config": {"workload": WORKLOAD, "model": "llama-3.1-8b-shape",
                   "layers": args.layers, "batch": B,
                   "decode_iters_per_step": it,
                   "verify_rows_per_step": 256,
                   "verify_windows": "%d x %d" % (b.wl["n_ver"],
                                                  b.wl["window"]),
                   "deterministic_fraction": b.wl["n_flag"] / B,
                   "mean_context": float(b.wl["ctx"].mean()),
                   "l2": "inputs larger than L2 (weights + KV >> 129 MB)",
                   "parallelism": "replicas" if world > 1 else "single",
                   "decode_launch": "cuda_graph" if use_graph else "eager",
                   "e2e_launch": "cuda_graph" if use_graph else "eager"},
        "e2e": e2e,
        "gpu_launches": int(round(launches * args.steps)),
        "roofline": roof,
        "kernels": kernels,
        "profiled_ms_per_step": ms_profiled,
        "clocks": clk,
        "device_status": status,
        "verify_commits": [int(x) for x in b.commits[-1][1]],
        "verify": verify_stats(b, ms),
    }
    if rank == 0 and not args.no_comparator:
        line["comparator"] = run_comparator(b, args)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, b.wl, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------- comparator --

def cublas_forward(b):
    """Decode forward of the bench's requests with every GEMM through
    torch.matmul (cuBLAS heuristics: not batch-invariant), the library's
    norm / RoPE / attention around them; returns fwd(tok, pos, maxkv) ->
    fp32 logits [B, V]."""
    import torch
    bi = b.bi
    eng = b.eng
    S = b.shape
    B = b.wl["batch"]
    H, F, D, Hq, Hkv = S.hidden, S.ffn, S.head_dim, S.n_heads, S.n_kv_heads
    dev = b.dev
    x = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
    h = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
    q = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    a = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    kvl = torch.empty(B, dtype=torch.int32, device=dev)
    ws = torch.empty(bi.bi_decode_attn_workspace_size(
        B, Hq, D, eng.max_kv_len) // 4, dtype=torch.float32, device=dev)
    W = b.weights
    scale = 1.0 / math.sqrt(D)

    def fwd(tok, pos, maxkv):
        torch.index_select(W["embed"], 0, tok, out=h)
        kvl.copy_(pos + 1)
        d = None
        for l, lw in enumerate(W["layers"]):
            if d is None:
                bi.bi_rmsnorm(None, 0, None, h, lw["attn_norm"], B, H, S.eps, x)
            else:
                bi.bi_rmsnorm(d, 1, None, h, lw["attn_norm"], B, H, S.eps, x)
            qkv = torch.matmul(x, lw["wqkv"].T).float()
            bi.bi_rope(qkv, 1, pos, b.slots, Hq, Hkv, D, S.theta, q,
                       eng.k_pool[l], eng.v_pool[l], eng.page_table)
            bi.bi_paged_decode_attn(q, eng.k_pool[l], eng.v_pool[l],
                                    eng.page_table, b.slots, kvl, maxkv, scale,
                                    a, ws)
            o = torch.matmul(a.view(B, Hq * D), lw["wo"].T).float()
            bi.bi_rmsnorm(o, 1, None, h, lw["ffn_norm"], B, H, S.eps, x)
            g = torch.matmul(x, lw["wg"].T)
            u = torch.matmul(x, lw["wu"].T)
            f = torch.nn.functional.silu(g) * u
            d = torch.matmul(f, lw["wd"].T).float()
        bi.bi_rmsnorm(d, 1, None, h, W["final_norm"], B, H, S.eps, x)
        return torch.matmul(x, W["lm_head"].T).float()

    return fwd


def run_comparator(b, args):
    """The same decode iterations with every GEMM through torch.matmul
    (cuBLAS default heuristics), the library's norm / RoPE / attention /
    argmax around them, against the invariant path's decode iterations alone.
    Run with the default bf16 reduced-precision setting and with it off
    (ybb.press section 5)."""
    import torch
    bi = b.bi
    B, it = b.wl["batch"], b.wl["iters"]
    fwd = cublas_forward(b)

    def run_cmp():
        cur = b.tok0.clone()
        for i in range(it):
            lg = fwd(cur, b.pos[i], b.maxkv[i])
            ids = b.ids[i]
            bi.bi_argmax_logits(lg, ids)
            cur = ids

    def timed(fn, reps):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    reps = max(2, min(args.steps, 4))
    ours_ms = timed(b.decode_iters, reps)
    out = {"what": "same decode iterations, GEMMs via torch.matmul (cuBLAS)",
           "invariant_decode_tok_s": B * it / (ours_ms / 1e3)}
    flag = torch.backends.cuda.matmul.allow_bf16_reduced_precision_reduction
    for name, val in (("cublas_default", flag), ("cublas_no_reduced_bf16", False)):
        torch.backends.cuda.matmul.allow_bf16_reduced_precision_reduction = val
        cms = timed(run_cmp, reps)
        out[name + "_tok_s"] = B * it / (cms / 1e3)
    torch.backends.cuda.matmul.allow_bf16_reduced_precision_reduction = flag
    out["invariant_over_default"] = (out["invariant_decode_tok_s"] /
                                     out["cublas_default_tok_s"])
    return out


def fast_path_report(b, fractions=(0.02, 0.10, 0.50, 1.0)):
    """LLM-42 with a real non-deterministic fast path (LLM-42 page, core
    method: decode everything on the fast path, verify the deterministic
    requests' windows with the invariant path, commit up to the first
    mismatch).  Per deterministic fraction d, one round: 32 greedy decode
    iterations of all B requests on the cuBLAS path, then the first
    round(d * B) requests' 32-token windows verified in groups of 8 (256
    rows) by verify_commit_rollback.  Committed tokens: 32 per unverified
    request, commit length (+1 for the verifier's own token after a
    mismatch) per verified one.  Against: 32 invariant decode iterations of
    all B requests."""
    import torch
    eng, wl = b.eng, b.wl
    B, w = wl["batch"], 32
    ctx = wl["ctx"]
    dev = b.dev
    fwd = cublas_forward(b)
    pos = [torch.from_numpy(ctx + i).to(dev).int() for i in range(w)]
    maxkv = [int(ctx.max()) + i + 1 for i in range(w)]
    ids = torch.empty(w, B, dtype=torch.int32, device=dev)
    logits = torch.empty(B, b.shape.vocab, dtype=torch.float32, device=dev)

    def fast():
        cur = b.tok0
        for i in range(w):
            lg = fwd(cur, pos[i], maxkv[i])
            b.bi.bi_argmax_logits(lg, ids[i])
            cur = ids[i]

    def invariant():
        cur = b.tok0
        for i in range(w):
            eng.decode(cur, pos[i], b.slots, logits=logits, ids=ids[i],
                       max_kv_len=maxkv[i])
            cur = ids[i]

    def rearm(slots):
        for r in slots:
            eng.reserve(r, int(ctx[r]) + wl["headroom"])

    def timed(fn):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        out = fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1), out

    fast()
    invariant()
    inv_ms, _ = timed(invariant)
    out = {"window": w, "batch": B,
           "invariant_only_tok_s": B * w / (inv_ms / 1e3), "fractions": {}}
    last = b.tok0.cpu().numpy()
    for d in fractions:
        n_f = max(1, int(round(d * B)))

        def llm42():
            fast()
            cand = ids[:, :n_f].T.cpu().numpy()
            res = []
            for g in range(0, n_f, 8):
                sl = list(range(g, min(n_f, g + 8)))
                res.append(eng.verify(sl, ctx[sl], last[sl],
                                      [list(map(int, cand[r])) for r in sl]))
            return res

        ms, res = timed(llm42)
        commit = np.concatenate([r[1] for r in res])
        rolled = int((commit < w).sum())
        committed = (B - n_f) * w + int(commit.sum()) + rolled
        out["fractions"][str(d)] = {
            "verified": n_f, "ms": ms,
            "committed_tok_s": committed / (ms / 1e3),
            "windows_rolled_back": rolled,
            "mean_commit": float(commit.mean()),
            "recomputed": int((w - commit - 1)[commit < w].sum())}
        rearm(range(n_f))
    return out


# -------------------------------------------------------------- CPU oracle --

_ORACLE_W = {}


def oracle_weights():
    """One random 8B-shape layer, the final norm, the LM head and embedding
    rows, generated once on the host (bf16 bit patterns)."""
    if not _ORACLE_W:
        import torch
        from deterministic_invariant_bf16_gb300 import synth
        S = synth.LLAMA8B

        def u16(t):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)

        w = synth.make_weights(synth.ModelShape(
            n_layers=1, hidden=S.hidden, n_heads=S.n_heads,
            n_kv_heads=S.n_kv_heads, head_dim=S.head_dim, ffn=S.ffn,
            vocab=256, eps=S.eps, theta=S.theta), 7, "cpu")
        _ORACLE_W["layer"] = {k: u16(v) for k, v in w["layers"][0].items()}
        _ORACLE_W["final_norm"] = u16(w["final_norm"])
        _ORACLE_W["embed"] = u16(w["embed"])
        _ORACLE_W["lm_head"] = u16(synth.normal_bf16((S.vocab, S.hidden),
                                                     0.02, 9, "cpu"))
    return _ORACLE_W


def oracle_sample(wl, seconds, n_layers=32, max_requests=16):
    """Time the oracle on a bounded sample of the workload: one decode token
    for each of a few requests through the full layer stack and LM head.
    One random layer's weights serve every layer (the oracle's cost does not
    depend on the values); each request's cache holds random bf16 values."""
    import oracle
    from deterministic_invariant_bf16_gb300 import synth
    S = synth.LLAMA8B
    cfg = oracle.Cfg(n_layers=n_layers, hidden=S.hidden, n_heads=S.n_heads,
                     n_kv_heads=S.n_kv_heads, head_dim=S.head_dim, ffn=S.ffn,
                     vocab=S.vocab, eps=S.eps, theta=S.theta)
    W = oracle_weights()
    lw, lm, fnorm, emb = W["layer"], W["lm_head"], W["final_norm"], W["embed"]
    rng = np.random.default_rng(8)
    ctx = wl["ctx"]
    # requests spread over the context distribution (the median alone when
    # only one is asked for)
    srt = np.argsort(ctx)
    if max_requests == 1:
        order = srt[[len(ctx) // 2]]
    else:
        order = srt[np.linspace(0, len(ctx) - 1, max_requests).astype(int)]
    done, t_compute = 0, 0.0
    for r in order:
        L = int(ctx[r])
        h = oracle.bf16_value(emb[[int(wl["first_tokens"][r]) % emb.shape[0]]])
        for _ in range(n_layers):
            kc = oracle.bf16r(rng.standard_normal((1, L + 1, S.n_kv_heads,
                                                   S.head_dim), np.float32))
            vc = oracle.bf16r(rng.standard_normal(kc.shape, np.float32))
            t0 = time.perf_counter()
            h = oracle.decoder_layer(h, np.zeros(1, np.int32),
                                     np.array([L], np.int32), lw, kc, vc, cfg)
            t_compute += time.perf_counter() - t0
        t0 = time.perf_counter()
        x = oracle.bf16_bits(oracle.rmsnorm(h, fnorm, cfg.eps))
        logits = oracle.gemm(x, lm)
        oracle.argmax(logits)
        t_compute += time.perf_counter() - t0
        done += 1
        if t_compute >= seconds:
            break
    return done, t_compute


def cpu_baseline(args, wl, seconds):
    done, t = oracle_sample(wl, seconds, n_layers=args.layers)
    cores = len(os.sched_getaffinity(0))
    return {"value": done / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "threads": int(os.environ.get("OMP_NUM_THREADS", cores)),
            "sample": "%d decode tokens (one per request, contexts spread over "
                      "the workload), %d layers + LM head, %.1f s of oracle "
                      "compute" % (done, args.layers, t)}


def run_reference(args):
    """The oracle arm: the CPU oracle, as it stands, on the host cores; each
    step is one decode token of one request through the full model."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = make_workload(args.batch, args.iters)
    from oracle import build as obuild
    obuild.build()
    for _ in range(args.warmup):
        oracle_sample(wl, 0.0, n_layers=args.layers, max_requests=1)
    t_tot, n_tot = 0.0, 0
    for _ in range(args.steps):
        n, t = oracle_sample(wl, 0.0, n_layers=args.layers, max_requests=1)
        t_tot += t
        n_tot += n
    value = n_tot / t_tot
    cores = len(os.sched_getaffinity(0))
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * t_tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "model": "llama-3.1-8b-shape",
                       "layers": args.layers, "batch": args.batch},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores,
                             "kind": "oracle",
                             "sample": "one decode token of one request per "
                                       "step, full layer stack + LM head"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.report:
        run_report(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
