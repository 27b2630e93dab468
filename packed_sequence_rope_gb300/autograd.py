"""PyTorch autograd entry: fused RoPE + AnchorAttention as a differentiable op.

Argument marshalling only, like the rest of the binding: the forward is one
aa_fwd call and the backward one aa_bwd_from_fwd call (or aa_bwd), so every
step runs in the library's kernels. The mask, positions and RoPE come from
the plan ("When Precision Meets Position", architecture page, §3.4
"AnchorAttention: The Shared Anchor Design" and Eq. 6 of §3.4 "Rotary
Positional Embedding (RoPE)").

    with Plan(cu_doclens, T, Hq, Hkv, D, rope_base) as plan:
        o = anchor_attention(plan, q, k, v)     # q, k, v: [T, H, D] bf16, requires_grad
        loss = f(o); loss.backward()            # q.grad, k.grad, v.grad w.r.t. the un-rotated q, k, v

keep_rotated=True (the default) keeps the forward's workspace, which holds
the rotated Q and K (T * (Hq + Hkv) * D * 2 bytes), until the backward and
uses aa_bwd_from_fwd; keep_rotated=False saves q and k instead and lets aa_bwd
rotate them again (less memory held between the passes, two more rotation
passes). The plan must outlive the backward.
"""
import torch

from .binding import ROPE_NONE

__all__ = ["AnchorAttentionFn", "anchor_attention"]


class AnchorAttentionFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, plan, q, k, v, keep_rotated=True):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        fws = plan.alloc_fwd_workspace(q.device)
        o, lse = plan.fwd(q, k, v, workspace=fws)
        ctx.plan = plan
        # without RoPE the forward rotates nothing, and aa_bwd_from_fwd refuses such plans
        ctx.keep_rotated = bool(keep_rotated) and plan.cfg.rope_layout != ROPE_NONE
        if ctx.keep_rotated:
            ctx.fws = fws
            ctx.save_for_backward(v, o, lse)
        else:
            ctx.save_for_backward(q, k, v, o, lse)
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        do = do.contiguous()
        if ctx.keep_rotated:
            v, o, lse = ctx.saved_tensors
            dq, dk, dv = ctx.plan.bwd_from_fwd(ctx.fws, v, o, lse, do)
            ctx.fws = None
        else:
            q, k, v, o, lse = ctx.saved_tensors
            dq, dk, dv = ctx.plan.bwd(q, k, v, o, lse, do)
        return None, dq, dk, dv, None


def anchor_attention(plan, q, k, v, keep_rotated=True, return_lse=False):
    """O (and, if asked, the per-row log-sum-exp [Hq, T] fp32, not
    differentiable) of the plan's attention over q, k, v."""
    o, lse = AnchorAttentionFn.apply(plan, q, k, v, keep_rotated)
    return (o, lse) if return_lse else o
