"""GPU: segment plans (documents given per token, interleaved chunks;
"When Precision Meets Position", architecture page, §3.4 "AnchorAttention with
Interleaved Chunks" and "Mask construction") against the fp64 oracle, in the
caller's token order, with the same tolerances as the contiguous path."""
import numpy as np
import pytest
import torch

import oracle as orc
from aa_synth import interleaved_chunks
from gpu_common import REL_L2, check_forward, f64, inputs, rel_l2, rope_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def aa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import packed_sequence_rope_gb300 as pkg
    return pkg


CASES = [
    # name, lengths, chunks, Hq, Hkv, D, base, mode, pos, layout
    ("anchor_reset_gqa", [200, 37, 410, 3, 150], 4, 4, 2, 128, 5e5, orc.MASK_ANCHOR, orc.POS_RESET,
     orc.ROPE_ADJACENT),
    ("anchor_continuous", [300, 120, 90], 3, 2, 2, 128, 1e4, orc.MASK_ANCHOR, orc.POS_CONTINUOUS,
     orc.ROPE_ADJACENT),
    ("intra_doc_d64_half", [128, 129, 250], 5, 2, 1, 64, 1e4, orc.MASK_INTRA_DOC, orc.POS_RESET, orc.ROPE_HALF),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_segments_fwd_bwd_elementwise(aa, case):
    name, lengths, chunks, Hq, Hkv, D, base, mode, pos, layout = case
    doc = interleaved_chunks(lengths, chunks, np.random.default_rng(len(name)))
    T = doc.size
    q, k, v, do = inputs(T, Hq, Hkv, D, seed=41)
    with aa.Plan(None, T, Hq, Hkv, D, base, mode, pos, layout, doc_of_token=doc) as p:
        o, lse = p.fwd(q, k, v)
        dq, dk, dv = p.bwd(q, k, v, o, lse, do)
        torch.cuda.synchronize()
        p.check_device_error()
    prob = orc.Problem(None, T, Hq, Hkv, D, base, mode, pos, layout, doc_of_token=doc)
    O, L = orc.forward(prob, q.cpu(), k.cpu(), v.cpu())
    check_forward(o, lse, O, L, tag=name)
    gq, gk, gv = orc.backward(prob, q.cpu(), k.cpu(), v.cpu(), do.cpu())
    for nm, got, ref in (("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
        e = rel_l2(got, ref)
        assert e <= REL_L2, f"{name} {nm} rel-L2 {e:.3e}"


def test_segments_rope_apply_uses_caller_positions(aa):
    doc = interleaved_chunks([100, 80, 60], 3, np.random.default_rng(3))
    T, H, D = doc.size, 2, 128
    x = torch.randn(T, H, D, device="cuda").to(torch.bfloat16)
    with aa.Plan(None, T, H, H, D, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, doc_of_token=doc, pos_shift=9) as p:
        y = p.rope_apply(x)
        torch.cuda.synchronize()
    pos = orc.segment_position_ids(doc, orc.POS_RESET, 9)
    ref = orc.rotate(f64(x), pos, 1e4)
    assert (np.abs(f64(y) - ref) <= rope_bound(ref, f64(x))).all()


def test_contiguous_segments_bit_identical_to_cu_plan(aa):
    cu, T, Hq, Hkv, D = [1, 90, 91, 400, 640], 640, 2, 1, 128
    doc = np.zeros(T, np.int32)
    for kk in range(1, len(cu)):
        doc[cu[kk - 1]:cu[kk]] = 7 * kk      # any ids >= 1
    q, k, v, do = inputs(T, Hq, Hkv, D, seed=42)
    with aa.Plan(cu, T, Hq, Hkv, D, 1e4) as p0, aa.Plan(None, T, Hq, Hkv, D, 1e4, doc_of_token=doc) as p1:
        o0, l0 = p0.fwd(q, k, v)
        o1, l1 = p1.fwd(q, k, v)
        _, dk0, dv0 = p0.bwd(q, k, v, o0, l0, do)
        _, dk1, dv1 = p1.bwd(q, k, v, o1, l1, do)
        torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert torch.equal(dk0, dk1) and torch.equal(dv0, dv1)


def test_segments_static_workspace_backward(aa):
    doc = interleaved_chunks([70, 50, 40], 3, np.random.default_rng(4))
    T, H, D = doc.size, 2, 64
    q, k, v, do = inputs(T, H, H, D, seed=43)
    with aa.Plan(None, T, H, H, D, 1e4, doc_of_token=doc) as p:
        o, lse = p.fwd(q, k, v)
        dq0, dk0, dv0 = p.bwd(q, k, v, o, lse, do)
        dq1, dk1, dv1 = p.bwd_static_workspace(q, k, v, o, lse, do)
        torch.cuda.synchronize()
    assert torch.equal(dk0, dk1) and torch.equal(dv0, dv1)
    assert rel_l2(dq0, f64(dq1)) <= 1e-6


def test_full_size_interleaved_chunks_bench_path(aa):
    # the benchmark's --chunks 4 layout: the 64K packing's 38 documents cut
    # into 4 chunks each and interleaved, through aa_fwd + aa_bwd_from_fwd.
    # The kernels run on the tokens grouped by document (in order of first
    # appearance) and meet the caller's order only through their row maps, so
    # the contiguous plan on the grouped inputs gives O, LSE, dk and dv bit for
    # bit and dq up to the order of its fp32 additions; and one document is
    # checked against the oracle in the caller's order.
    from aa_synth import WORKLOADS, make_qkv, workload_cu_doclens
    w = WORKLOADS["llama7b_64k"]
    T, Hq, Hkv, D = w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    doc = interleaved_chunks(np.diff(workload_cu_doclens(w)), 4, np.random.default_rng(0))
    assert doc.size == T
    q, k, v, do = make_qkv(w, device="cuda")
    outs = []
    with aa.Plan(None, T, Hq, Hkv, D, w.rope_base, doc_of_token=doc) as p:
        fws = p.alloc_fwd_workspace(q.device)
        o, lse = p.fwd(q, k, v, workspace=fws)
        outs = [o, lse, *p.bwd_from_fwd(fws, v, o, lse, do)]
        torch.cuda.synchronize()
        p.check_device_error()
        del fws
    first = {}
    for i, d in enumerate(doc[1:].tolist(), start=1):
        first.setdefault(d, i)
    order = sorted(first, key=first.get)
    perm = np.concatenate([[0]] + [np.flatnonzero(doc == d) for d in order])
    cu_g = np.concatenate([[1], 1 + np.cumsum([int((doc == d).sum()) for d in order])]).astype(np.int32)
    pg = torch.as_tensor(perm, device=q.device)
    with aa.Plan(cu_g, T, Hq, Hkv, D, w.rope_base) as p:
        fws = p.alloc_fwd_workspace(q.device)
        o_g, lse_g = p.fwd(q[pg], k[pg], v[pg], workspace=fws)
        dq_g, dk_g, dv_g = p.bwd_from_fwd(fws, v[pg], o_g, lse_g, do[pg])
        torch.cuda.synchronize()
        p.check_device_error()
        del fws
    o, lse, dq, dk, dv = outs
    assert torch.equal(o[pg], o_g)
    assert torch.equal(lse[:, pg], lse_g)
    assert torch.equal(dk[pg], dk_g)
    assert torch.equal(dv[pg], dv_g)
    # dq: the fp32 accumulator receives the same contributions in another order
    # (k additions per value: relative error ~ k 2^-24, far below bf16's half
    # ulp 2^-9), so after the bf16 rounding a value moves by at most one ulp;
    # the absolute floor covers sums that cancel to near zero
    a, b = dq[pg].double(), dq_g.double()
    mag = torch.maximum(a.abs(), b.abs()).clamp_min(1e-30)
    bound = torch.exp2(torch.floor(torch.log2(mag)) - 7) + 1e-6 * b.abs().max()  # bf16 spacing at |x|
    bad = int(((a - b).abs() > bound).sum())
    assert bad == 0, f"dq: {bad} values beyond one bf16 ulp of the contiguous plan's"
    # one document against the oracle: [anchor + its tokens in the caller's
    # order] is that document laid out contiguously (positions count its tokens)
    d = order[len(order) // 2]
    idx = np.concatenate([[0], np.flatnonzero(doc == d)])
    n = idx.size - 1
    it = torch.as_tensor(idx, device=q.device)
    heads = torch.tensor([0, Hq - 1], device=q.device)
    sub = [x[it][:, heads].cpu() for x in (q, k, v, do)]
    prob = orc.Problem([1, 1 + n], 1 + n, 2, 2, D, w.rope_base)
    O, L = orc.forward(prob, *sub[:3])
    check_forward(o[it[1:]][:, heads], lse[heads][:, it[1:]], O[1:], L[:, 1:], tag=f"document {d}")
    gq, gk, gv = orc.backward(prob, *sub)
    for nm, got, ref in (("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
        err = rel_l2(got[it[1:]][:, heads], ref[1:])
        assert err <= REL_L2, f"document {d} {nm} rel-L2 {err:.3e}"
