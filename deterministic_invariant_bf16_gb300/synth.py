"""Seeded synthetic inputs: random-init weights, token ids, request lengths
and paged-KV layouts.

This module only draws numbers; it holds none of the method's arithmetic.
Both the GPU path and the CPU oracle are fed from it by the tests and the
benchmark, so the two sides always see bit-identical inputs.

Workload shapes follow the deterministic-inference pages: Llama-3.1-8B-shaped
decoders (LLM-42 summary, section "实验与结果": SGLang with
Llama-3.1-8B-Instruct), ShareGPT-like and ArXiv-like length mixes (LLM-42,
section 5.1, Table 2), and PagedAttention pages (ybb.press executive summary;
Vosti abstract).  The public datasets themselves are not used: seeded
lognormal and uniform length draws stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class ModelShape:
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    eps: float
    theta: float

    @property
    def q_dim(self):
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self):
        return self.n_kv_heads * self.head_dim

    @property
    def qkv_dim(self):
        return self.q_dim + 2 * self.kv_dim


# Tiny random-init decoder: 2 layers, hidden 128, 4 heads of 32, FFN 256,
# vocab 512, RoPE theta 1e4.
TINY = ModelShape(n_layers=2, hidden=128, n_heads=4, n_kv_heads=4, head_dim=32,
                  ffn=256, vocab=512, eps=1e-5, theta=1e4)

# Llama-3.1-8B shape: hidden 4096, 32 query / 8 KV heads of 128, FFN 14336,
# vocab 128256, RoPE theta 5e5, 32 layers.
LLAMA8B = ModelShape(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=8,
                     head_dim=128, ffn=14336, vocab=128256, eps=1e-5,
                     theta=5e5)

PAGE_SIZE = 16


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32 with a seeded torch generator, stored bf16."""
    g = generator(seed, device)
    x = torch.randn(tuple(shape), generator=g, device=device,
                    dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def make_weights(shape: ModelShape, seed: int, device="cpu", std=0.02,
                 n_layers=None) -> dict:
    """Random-init decoder weights (bf16): N(0, std^2) matrices, RMSNorm
    weights one [reading: the usual RMSNorm init].  Matrices are [out, in]:
    wqkv rows are q heads, then k heads, then v heads; wg and wu are the gate
    and up projections, wd the down projection; the embedding is untied from
    the LM head."""
    L = shape.n_layers if n_layers is None else n_layers
    H, F, V = shape.hidden, shape.ffn, shape.vocab
    s = seed * 1000

    def mat(rows, cols, k):
        return normal_bf16((rows, cols), std, s + k, device)

    ones = torch.ones(H, dtype=torch.bfloat16, device=device)
    layers = []
    for li in range(L):
        b = 10 + 10 * li
        layers.append(dict(
            attn_norm=ones.clone(),
            wqkv=mat(shape.qkv_dim, H, b + 0),
            wo=mat(H, shape.q_dim, b + 1),
            ffn_norm=ones.clone(),
            wg=mat(F, H, b + 2),
            wu=mat(F, H, b + 3),
            wd=mat(H, F, b + 4),
        ))
    return dict(embed=mat(V, H, 1), layers=layers, final_norm=ones.clone(),
                lm_head=mat(V, H, 2))


def token_ids(n: int, vocab: int, rng: np.random.Generator) -> np.ndarray:
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def lognormal_lengths(n: int, median: float, sigma: float, lo: int, hi: int,
                      rng: np.random.Generator) -> np.ndarray:
    """clip(round(exp(N(ln median, sigma))), lo, hi)."""
    x = np.exp(rng.normal(np.log(median), sigma, size=n))
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


def uniform_lengths(n: int, lo: int, hi: int, rng: np.random.Generator):
    return rng.integers(lo, hi + 1, size=n).astype(np.int64)


def paged_layout(capacities, page_size: int, rng: np.random.Generator,
                 extra_pages: int = 0):
    """Assign physical pages to requests in a random order.

    capacities[r] is the number of token slots request r must hold.  Returns
    (page_table int32 [R, max_pages] with -1 for unused entries, number of
    physical pages in the pool).  Pages are a random permutation of the pool,
    so logical neighbours are never physical neighbours."""
    caps = np.asarray(capacities, np.int64)
    need = -(-caps // page_size)
    max_pages = int(max(1, need.max(initial=1)))
    total = int(need.sum()) + extra_pages
    perm = rng.permutation(total).astype(np.int32)
    table = np.full((len(caps), max_pages), -1, np.int32)
    at = 0
    for r, n in enumerate(need):
        table[r, :n] = perm[at:at + n]
        at += n
    return table, total
