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
