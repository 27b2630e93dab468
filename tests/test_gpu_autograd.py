"""GPU: the autograd entry (packed_sequence_rope_gb300.anchor_attention).

It marshals one aa_fwd call and one aa_bwd_from_fwd (or aa_bwd) call, so its
gradients are the library's: dk and dv bit for bit those of the direct calls
(the same kernels on the same operands), dq within one bf16 ulp (the order of
its fp32 additions varies), and all of them within the parity tolerance of the
fp64 oracle ("When Precision Meets Position", architecture page, §3.4
"AnchorAttention: The Shared Anchor Design"; Eq. 6 of §3.4 "Rotary Positional
Embedding (RoPE)").
"""
import pytest
import torch

import oracle as orc
from gpu_common import REL_L2, inputs, problem, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def aa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import packed_sequence_rope_gb300 as pkg
    return pkg


def _within_one_ulp(a, b):
    a, b = a.double(), b.double()
    mag = torch.maximum(a.abs(), b.abs()).clamp_min(1e-30)
    bound = torch.exp2(torch.floor(torch.log2(mag)) - 7) + 1e-6 * b.abs().max()
    return bool(((a - b).abs() <= bound).all())


CASES = [
    # name, cu, T, Hq, Hkv, D, base, mode, pos, layout
    ("anchor_gqa_d128", [1, 90, 600, 1100, 1500], 1500, 4, 2, 128, 5e6, orc.MASK_ANCHOR, orc.POS_RESET,
     orc.ROPE_ADJACENT),
    ("intra_doc_continuous_d64_half", [1, 129, 400], 400, 2, 2, 64, 1e4, orc.MASK_INTRA_DOC, orc.POS_CONTINUOUS,
     orc.ROPE_HALF),
    ("anchor_no_rope", [1, 200, 333], 333, 2, 1, 128, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_NONE),
]


@pytest.mark.parametrize("keep_rotated", [True, False])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_autograd_matches_direct_calls_and_oracle(aa, case, keep_rotated):
    name, cu, T, Hq, Hkv, D, base, mode, pos, layout = case
    q0, k0, v0, do = inputs(T, Hq, Hkv, D, seed=71)
    with aa.Plan(cu, T, Hq, Hkv, D, base, mode, pos, layout) as p:
        q, k, v = (x.clone().requires_grad_(True) for x in (q0, k0, v0))
        o, lse = aa.anchor_attention(p, q, k, v, keep_rotated=keep_rotated, return_lse=True)
        assert not lse.requires_grad
        (o.float() * do.float()).sum().backward()
        torch.cuda.synchronize()
        p.check_device_error()
        # the direct calls on the same inputs
        o_ref, lse_ref = p.fwd(q0, k0, v0)
        dq_ref, dk_ref, dv_ref = p.bwd(q0, k0, v0, o_ref, lse_ref, do)
        torch.cuda.synchronize()
        p.check_device_error()
    assert torch.equal(o.detach(), o_ref) and torch.equal(lse, lse_ref)
    assert torch.equal(k.grad, dk_ref), f"{name}: dk differs from aa_bwd"
    assert torch.equal(v.grad, dv_ref), f"{name}: dv differs from aa_bwd"
    assert _within_one_ulp(q.grad, dq_ref), f"{name}: dq beyond one bf16 ulp of aa_bwd"
    prob = problem(cu, T, Hq, Hkv, D, base, mode, pos, layout)
    gq, gk, gv = orc.backward(prob, q0.cpu(), k0.cpu(), v0.cpu(), do.cpu())
    for nm, got, ref in (("dq", q.grad, gq), ("dk", k.grad, gk), ("dv", v.grad, gv)):
        e = rel_l2(got, ref)
        assert e <= REL_L2, f"{name}: {nm} rel-L2 {e:.3e} against the oracle"


def test_autograd_through_a_following_op(aa):
    # the op composes with ordinary torch ops: a loss on a projection of O
    T, Hq, Hkv, D = 700, 2, 2, 128
    cu = [1, 300, 700]
    q0, k0, v0, do = inputs(T, Hq, Hkv, D, seed=72)
    gen = torch.Generator(device=q0.device).manual_seed(5)
    w = torch.randn(D, 16, device=q0.device, dtype=torch.float32, generator=gen)
    with aa.Plan(cu, T, Hq, Hkv, D, 5e6) as p:
        q, k, v = (x.clone().requires_grad_(True) for x in (q0, k0, v0))
        o = aa.anchor_attention(p, q, k, v)
        upstream = []
        o.register_hook(lambda g: upstream.append(g.detach().clone()))
        loss = (o.float() @ w).square().sum()
        loss.backward()
        torch.cuda.synchronize()
        p.check_device_error()
        # the gradient autograd brought to O, through the direct calls
        assert len(upstream) == 1 and upstream[0].dtype == torch.bfloat16
        o_ref, lse_ref = p.fwd(q0, k0, v0)
        dq_ref, dk_ref, dv_ref = p.bwd(q0, k0, v0, o_ref, lse_ref, upstream[0].contiguous())
        torch.cuda.synchronize()
    assert torch.equal(k.grad, dk_ref) and torch.equal(v.grad, dv_ref)
    assert _within_one_ulp(q.grad, dq_ref)


def test_autograd_on_a_segment_plan(aa):
    # documents given per token (interleaved chunks): the entry goes through
    # the same calls, so its gradients are aa_bwd's and meet the oracle in the
    # caller's token order
    import numpy as np
    from aa_synth import interleaved_chunks
    doc = interleaved_chunks([200, 37, 410, 3, 150], 4, np.random.default_rng(9))
    T, Hq, Hkv, D = doc.size, 4, 2, 128
    q0, k0, v0, do = inputs(T, Hq, Hkv, D, seed=73)
    with aa.Plan(None, T, Hq, Hkv, D, 5e5, doc_of_token=doc) as p:
        q, k, v = (x.clone().requires_grad_(True) for x in (q0, k0, v0))
        o = aa.anchor_attention(p, q, k, v)
        (o.float() * do.float()).sum().backward()
        torch.cuda.synchronize()
        p.check_device_error()
        o_ref, lse_ref = p.fwd(q0, k0, v0)
        dq_ref, dk_ref, dv_ref = p.bwd(q0, k0, v0, o_ref, lse_ref, do)
        torch.cuda.synchronize()
        p.check_device_error()
    assert torch.equal(o.detach(), o_ref)
    assert torch.equal(k.grad, dk_ref) and torch.equal(v.grad, dv_ref)
    assert _within_one_ulp(q.grad, dq_ref)
    prob = orc.Problem(None, T, Hq, Hkv, D, 5e5, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_ADJACENT,
                       doc_of_token=doc)
    gq, gk, gv = orc.backward(prob, q0.cpu(), k0.cpu(), v0.cpu(), do.cpu())
    for nm, got, ref in (("dq", q.grad, gq), ("dk", k.grad, gk), ("dv", v.grad, gv)):
        assert rel_l2(got, ref) <= REL_L2, nm
