"""Seeded synthetic inputs for packed multi-document attention.

This module is shared by the oracle tests and the CUDA path. It only draws
random numbers and lays documents end to end; it holds none of the method's
arithmetic (no masks, no position IDs, no rotations, no softmax).

Packing convention: token 0 is the anchor; document k (k = 1..K) occupies
tokens [cu_doclens[k-1], cu_doclens[k]), so cu_doclens[0] == 1 and
cu_doclens[K] == T. The last document is truncated so the documents fill
exactly T - 1 tokens after the anchor.

Workload shapes follow the long-context training setup of "When Precision
Meets Position: BFloat16 Breaks Down RoPE in Long-Context Training"
(architecture page, section "Long-Context Training Protocol": LLaMA-2-7B,
32 heads of dimension 128, 64K/128K packed sequences, RoPE bases 5e6 / 5e5),
with synthetic Gaussian activations standing in for the SlimPajama packings.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "doc_lengths", "pack", "gaussian_bf16",
    "workload_cu_doclens", "make_qkv",
]


def doc_lengths(kind: str, total: int, rng: np.random.Generator, **p) -> list[int]:
    """Draw document lengths until they cover ``total`` tokens.

    kind == "fixed":      p["lengths"] used as given (then truncated/padded by pack()).
    kind == "loguniform": floor(exp(U(ln lo, ln hi))).
    kind == "lognormal":  round(exp(ln median + sigma * N(0,1))) clipped to [lo, hi].
    """
    if kind == "fixed":
        return [int(x) for x in p["lengths"]]
    out: list[int] = []
    covered = 0
    while covered < total:
        if kind == "loguniform":
            lo, hi = p["lo"], p["hi"]
            n = int(math.floor(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
        elif kind == "lognormal":
            med, sig, lo, hi = p["median"], p["sigma"], p["lo"], p["hi"]
            n = int(round(math.exp(math.log(med) + sig * rng.standard_normal())))
            n = min(max(n, lo), hi)
        else:
            raise ValueError(f"unknown length distribution {kind!r}")
        out.append(n)
        covered += n
    return out


def pack(lengths: list[int], total_tokens: int) -> np.ndarray:
    """Lay documents after the anchor token; truncate the last one to fit.

    Returns int32 cu_doclens of size K + 1 with cu[0] = 1 and cu[K] = T.
    A list that does not reach T is extended by one final document.
    """
    if total_tokens < 2:
        raise ValueError("a packing needs the anchor plus at least one token")
    cu = [1]
    for n in lengths:
        if n <= 0:
            raise ValueError("document lengths must be positive")
        nxt = min(cu[-1] + n, total_tokens)
        cu.append(nxt)
        if nxt == total_tokens:
            break
    if cu[-1] < total_tokens:
        cu.append(total_tokens)
    return np.asarray(cu, dtype=np.int32)


def gaussian_bf16(shape, seed: int, device="cpu"):
    """N(0,1) samples rounded to bf16, drawn by torch's seeded generator on ``device``."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


@dataclass(frozen=True)
class Workload:
    name: str
    total_tokens: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    rope_base: float
    lengths: str                 # distribution kind for doc_lengths()
    length_params: dict = field(default_factory=dict)
    seed: int = 0


WORKLOADS = {
    # anchor + 4 documents of lengths 31/64/96/64, one head of dimension 64
    "tiny_256": Workload("tiny_256", 256, 1, 1, 64, 1e4, "fixed",
                         {"lengths": [31, 64, 96, 64]}),
    # LLaMA-2-7B-shaped layer, 8K packing, log-uniform 128..4096
    "llama7b_8k": Workload("llama7b_8k", 8192, 32, 32, 128, 1e4, "loguniform",
                           {"lo": 128, "hi": 4096}),
    # long-context training shape, 64K packing, log-normal median 1500
    "llama7b_64k": Workload("llama7b_64k", 65536, 32, 32, 128, 5e6, "lognormal",
                            {"median": 1500, "sigma": 1.0, "lo": 64, "hi": 65535}),
    # grouped-query 128K packing, 32 query heads / 8 kv heads, median 3000
    "gqa_128k": Workload("gqa_128k", 131072, 32, 8, 128, 5e5, "lognormal",
                         {"median": 3000, "sigma": 1.0, "lo": 64, "hi": 131071}),
    # 64K length-mix sweep points (median 512 / 4096 / one single document)
    "sweep_64k_m512": Workload("sweep_64k_m512", 65536, 32, 32, 128, 5e6, "lognormal",
                               {"median": 512, "sigma": 1.0, "lo": 64, "hi": 65535}),
    "sweep_64k_m4096": Workload("sweep_64k_m4096", 65536, 32, 32, 128, 5e6, "lognormal",
                                {"median": 4096, "sigma": 1.0, "lo": 64, "hi": 65535}),
    "sweep_64k_single": Workload("sweep_64k_single", 65536, 32, 32, 128, 5e6, "fixed",
                                 {"lengths": [65535]}),
}


def workload_cu_doclens(w: Workload) -> np.ndarray:
    rng = np.random.default_rng(w.seed)
    return pack(doc_lengths(w.lengths, w.total_tokens - 1, rng, **w.length_params),
                w.total_tokens)


def make_qkv(w: Workload, device="cpu", with_grad_out: bool = True, seed_offset: int = 0):
    """Q [T,Hq,d], K/V [T,Hkv,d] and dO [T,Hq,d] as bf16 N(0,1), each with its own seed."""
    T, Hq, Hkv, d = w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    s = 1000 * (w.seed + seed_offset)
    q = gaussian_bf16((T, Hq, d), s + 1, device)
    k = gaussian_bf16((T, Hkv, d), s + 2, device)
    v = gaussian_bf16((T, Hkv, d), s + 3, device)
    do = gaussian_bf16((T, Hq, d), s + 4, device) if with_grad_out else None
    return q, k, v, do


def interleaved_chunks(lengths, chunks_per_doc: int, rng) -> np.ndarray:
    """doc_of_token [1 + sum(lengths)] for documents split into chunks and
    interleaved at random, each document's chunks kept in order (the
    "interleaved chunks" data layout): 0 for the anchor token, document k
    (1-based) for its tokens. Split points are uniform; the merge picks the
    next chunk from a random document with chunks left, weighted by how many
    it has left."""
    pieces = []
    for k, n in enumerate(lengths, start=1):
        c = min(chunks_per_doc, n)
        cuts = np.sort(rng.choice(np.arange(1, n), size=c - 1, replace=False)) if c > 1 else np.array([], int)
        sizes = np.diff(np.concatenate([[0], cuts, [n]]))
        pieces.append([(k, int(sz)) for sz in sizes])
    out = [0]
    left = [len(p) for p in pieces]
    nxt = [0] * len(pieces)
    while sum(left):
        w = np.asarray(left, dtype=np.float64)
        d = int(rng.choice(len(pieces), p=w / w.sum()))
        k, sz = pieces[d][nxt[d]]
        out.extend([k] * sz)
        nxt[d] += 1
        left[d] -= 1
    return np.asarray(out, dtype=np.int32)
