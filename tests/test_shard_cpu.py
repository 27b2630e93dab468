"""Sharding one packing across ranks (aa_shard_plan and shard.py), on CPU.

"When Precision Meets Position", architecture page, §3.4 "AnchorAttention:
The Shared Anchor Design", "Mask construction": a token sees the anchor and
the earlier tokens of its own document only, so documents (and kv heads) can
be dealt to different ranks, with the anchor replicated; the pages run the
step over 8 GPUs (§3.4 "AnchorContext: Implementation Infrastructure").

The planner is checked on the host (every (document, kv head) in exactly one
piece, LPT balance, the split rule). The sharded step runs as two gloo ranks
with the fp64 oracle standing in for the per-packing kernels, and the
reassembled O, LSE, dq, dk, dv and the all-reduced anchor gradients must equal
the oracle on the whole packing.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from aa_synth import WORKLOADS, workload_cu_doclens

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def aa():
    import __graft_entry__
    __graft_entry__.build()
    import packed_sequence_rope_gb300 as pkg
    return pkg


def _pairs(cu, d):
    n = int(cu[d] - cu[d - 1])
    return n * (n + 1) // 2 + n


@pytest.mark.parametrize("name, Hq, Hkv", [("llama7b_64k", 32, 32), ("gqa_128k", 32, 8), ("llama7b_8k", 32, 32)])
@pytest.mark.parametrize("W", [1, 2, 3, 8])
def test_shard_plan_covers_and_balances(aa, name, Hq, Hkv, W):
    cu = workload_cu_doclens(WORKLOADS[name])
    group = Hq // Hkv
    pieces, cost = aa.shard_plan(cu, Hkv, group, W)
    K = len(cu) - 1
    seen = np.zeros((K + 1, Hkv), dtype=np.int64)
    for shard, doc, g0, g1, c in pieces:
        assert 0 <= shard < W and 1 <= doc <= K and 0 <= g0 < g1 <= Hkv
        assert c == _pairs(cu, doc) * (g1 - g0) * group
        seen[doc, g0:g1] += 1
    assert (seen[1:] == 1).all()                            # each (document, kv head) exactly once
    total = sum(_pairs(cu, d) for d in range(1, K + 1)) * Hq
    assert cost.sum() == total
    share = total / W
    biggest = max(p[4] for p in pieces)
    assert cost.max() <= share + biggest                    # LPT: no shard above the mean by more than one piece
    for d in range(1, K + 1):                               # only documents above one share are cut, into ceil(cost/share) ranges
        parts = sum(1 for p in pieces if p[1] == d)
        want = min(Hkv, max(1, int(np.ceil(_pairs(cu, d) * Hq / share - 1e-9))))
        assert parts == want
    assert [(p[0], p[2], p[1]) for p in pieces] == sorted((p[0], p[2], p[1]) for p in pieces)


def test_shard_plan_balance_at_8_ranks(aa):
    # the 64K packing over 8 ranks: within 1 % of an even split
    cu = workload_cu_doclens(WORKLOADS["llama7b_64k"])
    _, cost = aa.shard_plan(cu, 32, 1, 8)
    assert cost.max() / cost.mean() < 1.01


def test_shard_plan_rejects_bad_input(aa):
    with pytest.raises(aa.AAError, match="cu_doclens"):
        aa.shard_plan([0, 10], 2, 1, 2)
    with pytest.raises(aa.AAError, match="increase"):
        aa.shard_plan([1, 10, 10], 2, 1, 2)
    with pytest.raises(aa.AAError, match=">= 1"):
        aa.shard_plan([1, 10], 2, 1, 0)


# ------------------------------------------------------------------ two gloo ranks
CU = [1, 301, 341, 401, 501]      # one document above a rank's share: cut by kv head
T, HQ, HKV, D, BASE = 501, 4, 2, 16, 1e4


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs():
    import torch
    g = torch.Generator().manual_seed(5)
    mk = lambda h: torch.randn(T, h, D, generator=g, dtype=torch.float64)
    return mk(HQ), mk(HKV), mk(HKV), mk(HQ)


def _oracle_compute(spec, q, k, v, dout):
    import torch
    import oracle as orc
    Tl, hq, _ = q.shape
    prob = orc.Problem(spec.cu_doclens, Tl, hq, k.shape[1], D, BASE, orc.MASK_ANCHOR, orc.POS_RESET)
    O, L = orc.forward(prob, q, k, v)
    dq, dk, dv = orc.backward(prob, q, k, v, dout)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    return t(O), t(L), t(dq), t(dk), t(dv)


def _worker(rank, world, port, out):
    import sys
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from packed_sequence_rope_gb300 import shard
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v, do = _inputs()
    if rank != 0:                  # only the rank holding token 0 has the anchor's k, v
        k[0].zero_()
        v[0].zero_()
    res = list(shard.sharded_step(q, k, v, do, CU, rank, world, _oracle_compute))
    anchor = (res[3][0].clone(), res[4][0].clone())
    if rank != 0:                  # dk_0 / dv_0 are already summed on every rank
        res[3][0].zero_()
        res[4][0].zero_()
    for t in res:
        dist.all_reduce(t)
    if rank == 0:
        out.put([t.numpy() for t in res] + [a.numpy() for a in anchor])
    else:
        out.put([a.numpy() for a in anchor])
    dist.destroy_process_group()


def test_sharded_step_equals_the_whole_packing_gloo_world2(aa):
    import oracle as orc
    from packed_sequence_rope_gb300 import shard
    specs0, pieces, _ = shard.local_packings(CU, HQ, HKV, 2, 0)
    specs1, _, _ = shard.local_packings(CU, HQ, HKV, 2, 1)
    assert any(p[3] - p[2] < HKV for p in pieces)            # the long document is cut by kv head
    assert specs0[-1].anchor_row and not any(s.anchor_row for s in specs1)
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = [out.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    full = next(g for g in got if len(g) == 7)
    other = next(g for g in got if len(g) == 2)
    o, lse, dq, dk, dv, dk0, dv0 = full
    q, k, v, do = _inputs()
    prob = orc.Problem(CU, T, HQ, HKV, D, BASE)
    O, L = orc.forward(prob, q, k, v)
    gq, gk, gv = orc.backward(prob, q, k, v, do)
    for nm, a, b in (("O", o, O), ("LSE", lse, L), ("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
        assert np.allclose(a, b, rtol=1e-10, atol=1e-12), nm
    # both ranks hold the same all-reduced anchor gradients
    assert np.array_equal(dk0, other[0]) and np.array_equal(dv0, other[1])
    assert np.allclose(dk0, gk[0], rtol=1e-10, atol=1e-12) and np.allclose(dv0, gv[0], rtol=1e-10, atol=1e-12)
