"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Element-wise at sizes the oracle finishes in seconds (several tiles, ragged
tails, documents shorter than a tile, GQA, every mask/position/RoPE mode),
sampled at the full workload sizes, plus run-to-run determinism and
fused-vs-unfused RoPE bit identity.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from aa_synth import WORKLOADS, make_qkv, workload_cu_doclens
from gpu_common import (REL_L2, check_forward, f64, inputs, problem, rel_l2, rope_bound)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def aa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import packed_sequence_rope_gb300 as pkg
    return pkg


# --------------------------------------------------------------------------- RoPE
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("layout", [orc.ROPE_ADJACENT, orc.ROPE_HALF])
@pytest.mark.parametrize("shift", [0, 120000])
def test_rope_apply_matches_oracle(aa, D, layout, shift):
    T, H = 777, 3
    cu = [1, 200, 201, 777]
    x = torch.randn(T, H, D, device="cuda").to(torch.bfloat16)
    with aa.Plan(cu, T, H, H, D, 5e5, orc.MASK_ANCHOR, orc.POS_CONTINUOUS, layout, pos_shift=shift) as p:
        y = p.rope_apply(x)
        back = p.rope_apply(y, inverse=True)
        torch.cuda.synchronize()
    pos = orc.position_ids(cu, T, orc.MASK_ANCHOR, orc.POS_CONTINUOUS, shift)
    ref = orc.rotate(f64(x), pos, 5e5, layout)
    assert (np.abs(f64(y) - ref) <= rope_bound(ref, f64(x), layout)).all()
    ref_back = orc.rotate(f64(y), pos, 5e5, layout, inverse=True)
    assert (np.abs(f64(back) - ref_back) <= rope_bound(ref_back, f64(y), layout)).all()


def test_rope_none_is_copy(aa):
    x = torch.randn(300, 2, 64, device="cuda").to(torch.bfloat16)
    with aa.Plan([1, 300], 300, 2, 2, 64, 1e4, rope_layout=orc.ROPE_NONE) as p:
        assert torch.equal(p.rope_apply(x), x)


# --------------------------------------------------------------------------- fwd/bwd small
CASES = [
    # name, cu, T, Hq, Hkv, D, base, mode, pos, layout
    ("tiny", [1, 32, 96, 192, 256], 256, 1, 1, 64, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_ADJACENT),
    ("ragged_gqa", [1, 5, 140, 141, 400, 1000, 1301], 1301, 4, 2, 128, 5e6, orc.MASK_ANCHOR, orc.POS_RESET,
     orc.ROPE_ADJACENT),
    ("continuous", [1, 300, 301, 700, 1100], 1100, 2, 2, 128, 1e4, orc.MASK_ANCHOR, orc.POS_CONTINUOUS,
     orc.ROPE_ADJACENT),
    ("intra_doc", [1, 129, 500, 900], 900, 2, 1, 128, 1e4, orc.MASK_INTRA_DOC, orc.POS_RESET, orc.ROPE_ADJACENT),
    ("causal", None, 700, 2, 2, 128, 1e4, orc.MASK_CAUSAL, orc.POS_RESET, orc.ROPE_ADJACENT),
    ("half_d64", [1, 64, 65, 333, 640], 640, 2, 2, 64, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_HALF),
    ("no_rope", [1, 50, 600], 600, 2, 1, 128, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_NONE),
    ("single_doc", [1, 513], 513, 2, 2, 128, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_ADJACENT),
    ("two_tokens", [1, 2], 2, 1, 1, 128, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_ADJACENT),
    # GQA with an even group: forward items of two heads on one query tile (here a single partial tile)
    ("two_tokens_gqa", [1, 2], 2, 4, 2, 128, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_ADJACENT),
    # an odd group (3 query heads per kv head): forward items of two query tiles of one head
    ("gqa_group3_d64", [1, 100, 130, 300], 300, 3, 1, 64, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_ADJACENT),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fwd_bwd_elementwise(aa, case):
    name, cu, T, Hq, Hkv, D, base, mode, pos, layout = case
    q, k, v, do = inputs(T, Hq, Hkv, D, seed=len(name))
    with aa.Plan(cu, T, Hq, Hkv, D, base, mode, pos, layout) as p:
        o, lse = p.fwd(q, k, v)
        dq, dk, dv = p.bwd(q, k, v, o, lse, do)
        torch.cuda.synchronize()
        p.check_device_error()
    prob = problem(cu, T, Hq, Hkv, D, base, mode, pos, layout)
    O, L = orc.forward(prob, q.cpu(), k.cpu(), v.cpu())
    check_forward(o, lse, O, L, tag=name)
    gq, gk, gv = orc.backward(prob, q.cpu(), k.cpu(), v.cpu(), do.cpu())
    for nm, got, ref in (("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
        e = rel_l2(got, ref)
        assert e <= REL_L2, f"{name} {nm} rel-L2 {e:.3e}"


def test_anchor_row_and_gradients_of_anchor(aa):
    # the anchor row returns v_0 exactly (up to bf16 rounding of a copy)
    T, H, D = 1000, 2, 128
    cu = [1, 100, 450, 1000]
    q, k, v, do = inputs(T, H, H, D, seed=7)
    with aa.Plan(cu, T, H, H, D, 1e4) as p:
        o, lse = p.fwd(q, k, v)
        dq, dk, dv = p.bwd(q, k, v, o, lse, do)
        torch.cuda.synchronize()
    assert torch.equal(o[0], v[0])
    gq, gk, gv = orc.backward(problem(cu, T, H, H, D, 1e4), q.cpu(), k.cpu(), v.cpu(), do.cpu())
    assert rel_l2(dk[0], gk[0]) <= REL_L2 and rel_l2(dv[0], gv[0]) <= REL_L2


def test_determinism_and_fused_equals_unfused(aa):
    T, Hq, Hkv, D = 1500, 4, 2, 128
    cu = [1, 90, 600, 1100, 1500]
    q, k, v, do = inputs(T, Hq, Hkv, D, seed=3)
    with aa.Plan(cu, T, Hq, Hkv, D, 5e6) as p, \
            aa.Plan(cu, T, Hq, Hkv, D, 5e6, rope_layout=orc.ROPE_NONE) as pn:
        o1, l1 = p.fwd(q, k, v)
        o2, l2 = p.fwd(q, k, v)
        _, dk1, dv1 = p.bwd(q, k, v, o1, l1, do)
        _, dk2, dv2 = p.bwd(q, k, v, o1, l1, do)
        # unfused: rotate with aa_rope_apply, then attention with RoPE disabled
        o3, l3 = pn.fwd(p.rope_apply(q), p.rope_apply(k), v)
        torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


# --------------------------------------------------------------------------- full sizes, sampled
def _sample_rows(cu, T, n, seed):
    rng = np.random.default_rng(seed)
    starts = np.asarray(cu[:-1], dtype=np.int64)
    rows = np.unique(np.concatenate([[0, 1, T - 1], starts, rng.integers(0, T, n)]))
    return rows


@pytest.mark.parametrize("name", ["llama7b_8k", "llama7b_64k", "gqa_128k"])
def test_full_size_forward_sampled(aa, name):
    w = WORKLOADS[name]
    cu = workload_cu_doclens(w)
    q, k, v, do = make_qkv(w, device="cuda", with_grad_out=False)
    with aa.Plan(cu, w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.rope_base) as p:
        o, lse = p.fwd(q, k, v)
        torch.cuda.synchronize()
        p.check_device_error()
    rows = _sample_rows(cu, w.total_tokens, 96, 0)
    prob = problem(cu, w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.rope_base)
    O, L = orc.forward(prob, q.cpu(), k.cpu(), v.cpu(), rows=rows)
    check_forward(o, lse, O, L, rows=rows, tag=name)


def test_full_size_backward_documents(aa):
    # documents are independent apart from the anchor: the oracle restricted
    # to one document's rows gives that document's complete dq, dk, dv
    w = WORKLOADS["llama7b_8k"]
    cu = workload_cu_doclens(w)
    T = w.total_tokens
    q, k, v, do = make_qkv(w, device="cuda")
    with aa.Plan(cu, T, w.num_q_heads, w.num_kv_heads, w.head_dim, w.rope_base) as p:
        o, lse = p.fwd(q, k, v)
        dq, dk, dv = p.bwd(q, k, v, o, lse, do)
        torch.cuda.synchronize()
        p.check_device_error()
    prob = problem(cu, T, w.num_q_heads, w.num_kv_heads, w.head_dim, w.rope_base)
    lens = np.diff(cu)
    picks = [int(np.argmin(lens)), int(np.argmax(lens)), len(lens) - 1]
    for d in sorted(set(picks)):
        a, b = int(cu[d]), int(cu[d + 1])
        rows = np.arange(a, b)
        gq, gk, gv = orc.backward(prob, q.cpu(), k.cpu(), v.cpu(), do.cpu(), rows=rows)
        for nm, got, ref in (("dq", dq[a:b], gq[a:b]), ("dk", dk[a:b], gk[a:b]), ("dv", dv[a:b], gv[a:b])):
            e = rel_l2(got, ref)
            assert e <= REL_L2, f"doc {d} {nm} rel-L2 {e:.3e}"


# --------------------------------------------------------------------------- explicit frequency tables
def _scaled_theta(D, base):
    # a non-default table: the lowest-frequency half of the pairs slowed down 8x
    # (the kind of per-pair rescaling RoPE variants apply)
    th = orc.rope_theta(D, base)
    th[D // 4:] /= 8.0
    return th


@pytest.mark.parametrize("layout", [orc.ROPE_ADJACENT, orc.ROPE_HALF])
def test_rope_apply_custom_theta_matches_oracle(aa, layout):
    T, H, D = 600, 2, 128
    cu = [1, 250, 600]
    theta = _scaled_theta(D, 1e4)
    x = torch.randn(T, H, D, device="cuda").to(torch.bfloat16)
    with aa.Plan(cu, T, H, H, D, 1e4, orc.MASK_ANCHOR, orc.POS_CONTINUOUS, layout, pos_shift=3000,
                 theta=theta) as p:
        y = p.rope_apply(x)
        torch.cuda.synchronize()
    pos = orc.position_ids(cu, T, orc.MASK_ANCHOR, orc.POS_CONTINUOUS, 3000)
    ref = orc.rotate(f64(x), pos, 1e4, layout, theta=theta)
    assert (np.abs(f64(y) - ref) <= rope_bound(ref, f64(x), layout)).all()


def test_fwd_bwd_custom_theta_elementwise(aa):
    cu, T, Hq, Hkv, D = [1, 77, 400, 700], 700, 2, 1, 128
    theta = _scaled_theta(D, 5e5)
    q, k, v, do = inputs(T, Hq, Hkv, D, seed=31)
    with aa.Plan(cu, T, Hq, Hkv, D, 5e5, theta=theta) as p:
        o, lse = p.fwd(q, k, v)
        dq, dk, dv = p.bwd(q, k, v, o, lse, do)
        torch.cuda.synchronize()
        p.check_device_error()
    prob = orc.Problem(cu, T, Hq, Hkv, D, 5e5, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_ADJACENT, theta=theta)
    O, L = orc.forward(prob, q.cpu(), k.cpu(), v.cpu())
    check_forward(o, lse, O, L, tag="custom_theta")
    gq, gk, gv = orc.backward(prob, q.cpu(), k.cpu(), v.cpu(), do.cpu())
    for nm, got, ref in (("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
        assert rel_l2(got, ref) <= REL_L2, nm


def test_default_theta_table_is_bit_identical_to_base(aa):
    cu, T, H, D = [1, 300, 500], 500, 2, 64
    q, k, v, _ = inputs(T, H, H, D, seed=32)
    with aa.Plan(cu, T, H, H, D, 1e4) as p0, aa.Plan(cu, T, H, H, D, 1e4, theta=orc.rope_theta(D, 1e4)) as p1:
        o0, l0 = p0.fwd(q, k, v)
        o1, l1 = p1.fwd(q, k, v)
        torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_batched_rows_as_one_packing(aa):
    # two packed rows run separately, and concatenated after one shared anchor
    rows = [[1, 300, 310, 700], [1, 128, 600]]
    Hq, Hkv, D = 2, 2, 128
    per = [inputs(cu[-1], Hq, Hkv, D, seed=51 + b) for b, cu in enumerate(rows)]
    for i in range(3):                      # the rows share the anchor's q, k, v
        per[1][i][0] = per[0][i][0]
    outs = []
    for cu, (q, k, v, do) in zip(rows, per):
        with aa.Plan(cu, cu[-1], Hq, Hkv, D, 1e4) as p:
            o, lse = p.fwd(q, k, v)
            outs.append((o, lse) + p.bwd(q, k, v, o, lse, do))
    cat = lambda i: torch.cat([per[0][i][:1]] + [p_[i][1:] for p_ in per]).contiguous()
    q, k, v, do = (cat(i) for i in range(4))
    do[0] = per[0][3][0] + per[1][3][0]
    T = q.shape[0]
    cu = [1] + rows[0][1:] + [c + rows[0][-1] - 1 for c in rows[1][1:]]
    with aa.Plan(cu, T, Hq, Hkv, D, 1e4) as p:
        o, lse = p.fwd(q, k, v)
        dq, dk, dv = p.bwd(q, k, v, o, lse, do)
        torch.cuda.synchronize()
    off = 1
    for (o_r, l_r, dq_r, dk_r, dv_r), cu_r in zip(outs, rows):
        n = cu_r[-1] - 1
        sl = slice(off, off + n)
        assert (o[sl].float() - o_r[1:].float()).abs().max().item() <= 2e-2
        assert (lse[:, sl] - l_r[:, 1:]).abs().max().item() <= 1e-3
        for got, ref in ((dq[sl], dq_r[1:]), (dk[sl], dk_r[1:]), (dv[sl], dv_r[1:])):
            assert rel_l2(got, f64(ref)) <= REL_L2
        off += n
    assert rel_l2(dk[0:1], f64(outs[0][3][0:1] + outs[1][3][0:1])) <= REL_L2
    assert rel_l2(dv[0:1], f64(outs[0][4][0:1] + outs[1][4][0:1])) <= REL_L2


@pytest.mark.parametrize("name", ["llama7b_64k", "gqa_128k"])
def test_full_size_backward_documents_long(aa, name):
    # documents are independent apart from the anchor (pinned in the oracle
    # tests: a packing equals per-document runs), so the gradients of one
    # document's tokens at full size equal the oracle's on [anchor + that
    # document] alone, with the same reset positions
    w = WORKLOADS[name]
    cu = workload_cu_doclens(w)
    T = w.total_tokens
    q, k, v, do = make_qkv(w, device="cuda")
    with aa.Plan(cu, T, w.num_q_heads, w.num_kv_heads, w.head_dim, w.rope_base) as p:
        o, lse = p.fwd(q, k, v)
        dq, dk, dv = p.bwd(q, k, v, o, lse, do)
        torch.cuda.synchronize()
        p.check_device_error()
    lens = np.diff(cu)
    order = np.argsort(lens)
    picks = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])} if lens.max() <= 4096
                   else {int(order[0]), int(order[len(order) // 2])})
    host = [t.cpu() for t in (q, k, v, do)]
    for d in picks:
        a, b = int(cu[d]), int(cu[d + 1])
        idx = torch.from_numpy(np.concatenate([[0], np.arange(a, b)]))
        sub = orc.Problem([1, b - a + 1], b - a + 1, w.num_q_heads, w.num_kv_heads, w.head_dim, w.rope_base)
        gq, gk, gv = orc.backward(sub, *(t[idx] for t in host))
        for nm, got, ref in (("dq", dq[a:b], gq[1:]), ("dk", dk[a:b], gk[1:]), ("dv", dv[a:b], gv[1:])):
            e = rel_l2(got, ref)
            assert e <= REL_L2, f"{name} doc {d} ({b - a} tokens) {nm} rel-L2 {e:.3e}"
