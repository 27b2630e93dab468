"""One packing sharded across ranks (one process per GPU): documents and kv
heads are split by aa_shard_plan, every rank runs its pieces as ordinary
packings through the library's kernels, and the ranks exchange only the
anchor token's data.

Why this is exact ("When Precision Meets Position", architecture page, §3.4
"AnchorAttention: The Shared Anchor Design", "Mask construction"): a token
sees the anchor (token 0) and the earlier tokens of its own document, nothing
else. So a document's outputs and gradients depend only on its own tokens and
the anchor, and each kv head only on its own heads. A rank's pieces with the
same kv-head range form one local packing [anchor, its documents...] with the
documents' own (reset or continuous) positions; the anchor's k_0 / v_0 are
broadcast from the rank that holds them, and dk_0 / dv_0, which sum over
every query row of every document, are all-reduced (fp32) across the ranks.
The anchor row itself (which sees only itself) is computed once, by rank 0,
in a two-token packing whose second token is inert (zero q, k, v and dO).

The pages run this step over 8 GPUs with DeepSpeed-Ulysses (§3.4
"AnchorContext: Implementation Infrastructure"); this module is the
document/head split with the two one-token collectives instead.

Tensors here are global-layout torch tensors [T, H, D] (and LSE [Hq, T]);
`compute(spec, q, k, v, dout)` runs one local packing and returns
(o, lse, dq, dk, dv) for it. `kernel_compute` is the library's version
(aa_fwd + aa_bwd); tests may pass another.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .binding import POS_CONTINUOUS, POS_RESET, Plan, shard_plan


@dataclass
class LocalPacking:
    """One packing a rank runs: token 0 is the anchor, then whole documents.

    tokens: global token index of each local token (tokens[0] == 0).
    kv_heads: [g0, g1) kv heads; q_heads: the matching query heads.
    cu_doclens: local document boundaries (cu[0] == 1). Positions are reset
    per document (each starts at 1), so they match the whole packing's.
    anchor_row: True for the two-token packing that owns the anchor row.
    """
    tokens: np.ndarray
    kv_heads: tuple
    q_heads: tuple
    cu_doclens: np.ndarray
    anchor_row: bool = False


def local_packings(cu_doclens, num_q_heads, num_kv_heads, num_shards, rank):
    """The packings rank `rank` runs (its pieces grouped by kv-head range, plus
    the anchor row's packing on rank 0) and the full piece list."""
    cu = np.asarray(cu_doclens, dtype=np.int64)
    group = num_q_heads // num_kv_heads
    pieces, cost = shard_plan(cu, num_kv_heads, group, num_shards)
    by_range = {}
    for shard, doc, g0, g1, _ in pieces:
        if shard == rank:
            by_range.setdefault((g0, g1), []).append(doc)
    out = []
    for (g0, g1), docs in sorted(by_range.items()):
        docs = sorted(docs)
        toks = [np.zeros(1, dtype=np.int64)] + [np.arange(cu[d - 1], cu[d]) for d in docs]
        lens = [int(cu[d] - cu[d - 1]) for d in docs]
        lcu = np.concatenate([[1], 1 + np.cumsum(lens)]).astype(np.int32)
        out.append(LocalPacking(np.concatenate(toks), (g0, g1), (g0 * group, g1 * group), lcu))
    if rank == 0:
        out.append(LocalPacking(np.array([0, -1]), (0, num_kv_heads), (0, num_q_heads),
                                np.array([1, 2], dtype=np.int32), anchor_row=True))
    return out, pieces, cost


def gather(x, spec, heads):
    """Rows spec.tokens, heads [h0, h1) of a global [T, H, D] tensor; the
    anchor row's packing gets an inert (zero) second token."""
    import torch
    h0, h1 = heads
    idx = torch.as_tensor(np.maximum(spec.tokens, 0), device=x.device)
    y = x.index_select(0, idx)[:, h0:h1].contiguous()
    if spec.anchor_row:
        y[1].zero_()
    return y


def broadcast_anchor_kv(k, v, src=0, group=None):
    """Forward's exchange: every rank gets the anchor's k_0 / v_0 [Hkv, D]
    from `src` (the rank whose sequence shard holds token 0)."""
    import torch.distributed as dist
    for t in (k, v):
        row = t[0].contiguous()
        dist.broadcast(row, src=src, group=group)
        t[0].copy_(row)


def allreduce_anchor_grads(dk0, dv0, group=None):
    """Backward's exchange: dk_0 / dv_0 [Hkv, D] (fp32) summed over ranks."""
    import torch.distributed as dist
    dist.all_reduce(dk0, group=group)
    dist.all_reduce(dv0, group=group)


def kernel_compute(base, mask_mode, pos_mode=POS_RESET):
    """compute() through the library: aa_fwd + aa_bwd on one local packing."""
    if pos_mode == POS_CONTINUOUS:
        raise NotImplementedError("sharded packings use reset positions (every document starts at 1)")

    def run(spec, q, k, v, dout):
        T, Hq, D = q.shape
        with Plan(spec.cu_doclens, T, Hq, k.shape[1], D, base, mask_mode, pos_mode) as p:
            o, lse = p.fwd(q, k, v)
            dq, dk, dv = p.bwd(q, k, v, o, lse, dout)
            p.check_device_error()
        return o, lse, dq, dk, dv
    return run


def run_local(q, k, v, dout, cu_doclens, rank, world, compute):
    """Rank `rank`'s share of the step without any exchange: global-shaped
    (o, lse, dq, dk, dv) holding its rows and heads (zero elsewhere, row 0 of
    dk / dv left zero) and its partial anchor gradients (dk0, dv0) [Hkv, D]."""
    import torch
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    specs, _, _ = local_packings(cu_doclens, Hq, Hkv, world, rank)
    # fp32 for LSE and the anchor sums (fp64 when the inputs are fp64)
    acc = torch.float64 if q.dtype == torch.float64 else torch.float32
    o = torch.zeros_like(q)
    lse = torch.zeros(Hq, T, dtype=acc, device=q.device)
    dq, dk, dv = torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)
    dk0 = torch.zeros(Hkv, D, dtype=acc, device=q.device)
    dv0 = torch.zeros_like(dk0)
    for spec in specs:
        hq, hk = spec.q_heads, spec.kv_heads
        lq, lk, lv, ldo = gather(q, spec, hq), gather(k, spec, hk), gather(v, spec, hk), gather(dout, spec, hq)
        if not spec.anchor_row:
            ldo[0].zero_()   # the anchor row's own gradient is counted once, by the anchor packing
        lo, llse, ldq, ldk, ldv = compute(spec, lq, lk, lv, ldo)
        rows = torch.as_tensor(spec.tokens[1:], device=q.device)
        if spec.anchor_row:
            o[0, hq[0]:hq[1]] = lo[0]
            lse[hq[0]:hq[1], 0] = llse[:, 0].to(acc)
            dq[0, hq[0]:hq[1]] = ldq[0]
        else:
            o[rows, hq[0]:hq[1]] = lo[1:]
            lse[hq[0]:hq[1], rows] = llse[:, 1:].to(acc)
            dq[rows, hq[0]:hq[1]] = ldq[1:]
            dk[rows, hk[0]:hk[1]] = ldk[1:]
            dv[rows, hk[0]:hk[1]] = ldv[1:]
        dk0[hk[0]:hk[1]] += ldk[0].to(acc)
        dv0[hk[0]:hk[1]] += ldv[0].to(acc)
    return (o, lse, dq, dk, dv), (dk0, dv0)


def sharded_step(q, k, v, dout, cu_doclens, rank, world, compute, group=None):
    """One forward + backward of the whole packing on `world` ranks.

    q, k, v, dout: global tensors ([T, Hq, D], [T, Hkv, D]); only token 0's
    k / v must be valid on rank 0 (they are broadcast), each rank reads the
    rows of its own pieces. Returns global-shaped (o, lse, dq, dk, dv) holding
    this rank's rows and heads (zero elsewhere) with dk[0] / dv[0] already
    summed over every rank.
    """
    if world > 1:
        broadcast_anchor_kv(k, v, group=group)
    (o, lse, dq, dk, dv), (dk0, dv0) = run_local(q, k, v, dout, cu_doclens, rank, world, compute)
    if world > 1:
        allreduce_anchor_grads(dk0, dv0, group=group)
    dk[0] = dk0.to(dk.dtype)
    dv[0] = dv0.to(dv.dtype)
    return o, lse, dq, dk, dv
