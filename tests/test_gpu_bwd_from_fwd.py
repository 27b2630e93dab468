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
