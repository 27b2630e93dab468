"""GPU: aa_bwd_from_fwd, the backward pass that reads the rotated Q and K aa_fwd
left in its workspace instead of rotating q and k again ("When Precision Meets
Position", architecture page, §3.4 "AnchorAttention: The Shared Anchor
Design" for the mask, Eq. 6 of §3.4 "Rotary Positional Embedding (RoPE)" for
the rotation).

Its gradients are those of aa_bwd: dk and dv bit for bit (the same rotated
operands go through the same kernels), dq up to the order of its fp32 atomic
additions; and they meet the fp64 oracle at the parity tolerances. Plans
without RoPE are refused, and a short workspace is refused before any launch.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from aa_synth import interleaved_chunks
from gpu_common import REL_L2, f64, inputs, rel_l2

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
    # name, cu, T, Hq, Hkv, D, base, mode, pos, layout
    ("anchor_gqa_d128", [1, 90, 300, 301, 700, 1000], 1000, 4, 2, 128, 5e5, orc.MASK_ANCHOR, orc.POS_RESET,
     orc.ROPE_ADJACENT),
    ("intra_doc_continuous_d64_half", [1, 129, 400], 400, 2, 2, 64, 1e4, orc.MASK_INTRA_DOC, orc.POS_CONTINUOUS,
     orc.ROPE_HALF),
    ("causal_gqa_d128", None, 300, 2, 1, 128, 1e4, orc.MASK_CAUSAL, orc.POS_RESET, orc.ROPE_ADJACENT),
]


def _same_as_bwd(got, ref, tag):
    assert torch.equal(got[1], ref[1]), f"{tag}: dk differs from aa_bwd"
    assert torch.equal(got[2], ref[2]), f"{tag}: dv differs from aa_bwd"
    e = rel_l2(got[0], f64(ref[0]))
    assert e <= 1e-6, f"{tag}: dq rel-L2 {e:.3e} against aa_bwd"


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_matches_bwd_and_oracle(aa, case):
    name, cu, T, Hq, Hkv, D, base, mode, pos, layout = case
    q, k, v, do = inputs(T, Hq, Hkv, D, seed=51)
    with aa.Plan(cu, T, Hq, Hkv, D, base, mode, pos, layout) as p:
        fws = p.alloc_fwd_workspace(q.device)
        o, lse = p.fwd(q, k, v, workspace=fws)
        ref = p.bwd(q, k, v, o, lse, do)
        got = p.bwd_from_fwd(fws, v, o, lse, do)
        torch.cuda.synchronize()
        p.check_device_error()
        assert p.bwd_from_fwd_workspace_bytes() < p.workspace_bytes()
    _same_as_bwd(got, ref, name)
    prob = orc.Problem(cu, T, Hq, Hkv, D, base, mode, pos, layout)
    grads = orc.backward(prob, q.cpu(), k.cpu(), v.cpu(), do.cpu())
    for nm, g, r in zip(("dq", "dk", "dv"), got, grads):
        e = rel_l2(g, r)
        assert e <= REL_L2, f"{name} {nm} rel-L2 {e:.3e}"


def test_segments_match_bwd(aa):
    doc = interleaved_chunks([200, 37, 410, 3, 150], 4, np.random.default_rng(7))
    T, Hq, Hkv, D = doc.size, 4, 2, 128
    q, k, v, do = inputs(T, Hq, Hkv, D, seed=52)
    with aa.Plan(None, T, Hq, Hkv, D, 5e5, doc_of_token=doc) as p:
        fws = p.alloc_fwd_workspace(q.device)
        o, lse = p.fwd(q, k, v, workspace=fws)
        ref = p.bwd(q, k, v, o, lse, do)
        got = p.bwd_from_fwd(fws, v, o, lse, do)
        torch.cuda.synchronize()
        p.check_device_error()
    _same_as_bwd(got, ref, "segments")
    prob = orc.Problem(None, T, Hq, Hkv, D, 5e5, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_ADJACENT,
                       doc_of_token=doc)
    grads = orc.backward(prob, q.cpu(), k.cpu(), v.cpu(), do.cpu())
    for nm, g, r in zip(("dq", "dk", "dv"), got, grads):
        assert rel_l2(g, r) <= REL_L2, nm


def test_rope_none_is_refused(aa):
    q, k, v, do = inputs(256, 1, 1, 64, seed=53)
    with aa.Plan([1, 100, 256], 256, 1, 1, 64, 1e4, rope_layout=orc.ROPE_NONE) as p:
        fws = torch.empty(256, device="cuda", dtype=torch.uint8)
        o, lse = p.fwd(q, k, v)
        with pytest.raises(aa.AAError, match="AA_ROPE_NONE"):
            p.bwd_from_fwd(fws, v, o, lse, do)


def test_short_workspace_is_refused(aa):
    q, k, v, do = inputs(256, 2, 2, 128, seed=54)
    with aa.Plan([1, 100, 256], 256, 2, 2, 128, 1e4) as p:
        fws = p.alloc_fwd_workspace(q.device)
        o, lse = p.fwd(q, k, v, workspace=fws)
        small = torch.empty(256, device="cuda", dtype=torch.uint8)
        with pytest.raises(aa.AAError, match="smaller than aa_bwd_from_fwd_workspace_bytes"):
            p.bwd_from_fwd(fws, v, o, lse, do, workspace=small)


# --------------------------------------------------------------------------- full size, the timed path
FULL = [
    # workload, query heads checked (all of their kv groups' query heads, so
    # the kv heads' dk / dv are complete)
    ("llama7b_64k", [0, 17]),
    ("gqa_128k", [4, 5, 6, 7]),   # kv head 1 and its whole query group
]


@pytest.mark.parametrize("name, heads", FULL, ids=[f[0] for f in FULL])
def test_full_size_training_step(aa, name, heads):
    # The benchmark's step at full size: aa_fwd, then aa_bwd_from_fwd on the
    # forward's workspace. Documents are independent apart from the anchor
    # (architecture page, §3.4 "AnchorAttention", "Mask construction": every
    # row sees column 0, nothing crosses documents), so
    #  - the longest document's dq, dk, dv equal the oracle's on [anchor + that
    #    document] alone (its key ranges span the most tiles), and
    #  - the anchor's dk_0, dv_0 are the sum, over every document, of the
    #    oracle's anchor gradients from that document's rows, plus the anchor
    #    row's own term (counted once): the full reduction over all T rows.
    from aa_synth import WORKLOADS, make_qkv, workload_cu_doclens
    w = WORKLOADS[name]
    cu = workload_cu_doclens(w)
    T, Hq, Hkv, D = w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    group = Hq // Hkv
    kv = sorted({h // group for h in heads})
    assert sorted(heads) == [h for g in kv for h in range(g * group, (g + 1) * group)]
    q, k, v, do = make_qkv(w, device="cuda")
    with aa.Plan(cu, T, Hq, Hkv, D, w.rope_base) as p:
        fws = p.alloc_fwd_workspace(q.device)
        o, lse = p.fwd(q, k, v, workspace=fws)
        dq, dk, dv = p.bwd_from_fwd(fws, v, o, lse, do)
        torch.cuda.synchronize()
        p.check_device_error()
        del fws
    hq = torch.tensor(heads)
    hk = torch.tensor(kv)
    host = (q.cpu()[:, hq], k.cpu()[:, hk], v.cpu()[:, hk], do.cpu()[:, hq])
    dq, dk, dv = dq.cpu()[:, hq], dk.cpu()[:, hk], dv.cpu()[:, hk]
    del q, k, v, do, o, lse
    torch.cuda.empty_cache()
    lens = np.diff(cu)
    longest = int(np.argmax(lens))
    gk0 = np.zeros((len(kv), D))
    gv0 = np.zeros((len(kv), D))
    for d in range(len(lens)):
        a, b = int(cu[d]), int(cu[d + 1])
        idx = torch.from_numpy(np.concatenate([[0], np.arange(a, b)]))
        sub = orc.Problem([1, b - a + 1], b - a + 1, len(heads), len(kv), D, w.rope_base)
        rows = np.arange(0 if d == 0 else 1, b - a + 1)   # the anchor row once, with the first document
        gq, gk, gv = orc.backward(sub, *(t[idx] for t in host), rows=rows)
        gk0 += gk[0]
        gv0 += gv[0]
        if d == longest:
            for nm, got, ref in (("dq", dq[a:b], gq[1:]), ("dk", dk[a:b], gk[1:]), ("dv", dv[a:b], gv[1:])):
                e = rel_l2(got, ref)
                assert e <= REL_L2, f"{name} longest document ({b - a} tokens) {nm} rel-L2 {e:.3e}"
    for nm, got, ref in (("dk_0", dk[0], gk0), ("dv_0", dv[0], gv0)):
        e = rel_l2(got, ref)
        assert e <= REL_L2, f"{name} anchor {nm} over all {T} rows: rel-L2 {e:.3e}"


def test_training_step_replays_from_a_cuda_graph(aa):
    # The training step (aa_fwd + aa_bwd_from_fwd) issues only stream-ordered
    # work (kernel launches and the work counters' async resets), so a caller
    # may capture it in a CUDA graph: each replay re-runs the whole step and
    # gives the eager step's O, LSE, dk and dv bit for bit and its dq up to the
    # order of the fp32 dQ additions (within one bf16 ulp of each value).
    cu, T, Hq, Hkv, D = [1, 90, 600, 1100, 1500], 1500, 4, 2, 128
    q, k, v, do = inputs(T, Hq, Hkv, D, seed=61)
    with aa.Plan(cu, T, Hq, Hkv, D, 5e6) as p:
        fws = p.alloc_fwd_workspace(q.device)
        ws = torch.empty(p.bwd_from_fwd_workspace_bytes(), device=q.device, dtype=torch.uint8)
        o, lse = torch.empty_like(q), torch.empty(Hq, T, device=q.device, dtype=torch.float32)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        outs = (o, lse, dq, dk, dv)

        def step():
            p.fwd(q, k, v, o, lse, fws)
            p.bwd_from_fwd(fws, v, o, lse, do, dq, dk, dv, ws)

        step()
        torch.cuda.synchronize()
        p.check_device_error()
        ref = [t.clone() for t in outs]
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        torch.cuda.synchronize()
        for _ in range(2):
            for t in outs:
                t.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            p.check_device_error()
            for name, got, want in zip(("o", "lse", "dk", "dv"), (o, lse, dk, dv), (ref[0], ref[1], ref[3], ref[4])):
                assert torch.equal(got, want), f"graph replay: {name} differs from the eager step"
            a, b = dq.double(), ref[2].double()
            mag = torch.maximum(a.abs(), b.abs()).clamp_min(1e-30)
            bound = torch.exp2(torch.floor(torch.log2(mag)) - 7) + 1e-6 * b.abs().max()
            assert bool(((a - b).abs() <= bound).all()), "graph replay: dq beyond one bf16 ulp of the eager step"
