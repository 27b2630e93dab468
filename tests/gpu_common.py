"""Shared helpers of the GPU parity tests (inputs, oracle comparison, tolerances).

Tolerances are the acceptance bounds for this path: O max-abs <= 2e-2 and
mean-abs <= 2e-3 against the fp64 oracle; dQ/dK/dV relative L2 <= 3e-2;
LSE max-abs <= 1e-2 (an extra check). Metadata is compared bit-exactly.
"""
import numpy as np
import torch

import oracle as orc
from aa_synth import gaussian_bf16

O_MAX, O_MEAN, LSE_MAX, REL_L2 = 2e-2, 2e-3, 1e-2, 3e-2


def inputs(T, Hq, Hkv, D, seed, device="cuda"):
    q = gaussian_bf16((T, Hq, D), 10 * seed + 1, device)
    k = gaussian_bf16((T, Hkv, D), 10 * seed + 2, device)
    v = gaussian_bf16((T, Hkv, D), 10 * seed + 3, device)
    do = gaussian_bf16((T, Hq, D), 10 * seed + 4, device)
    return q, k, v, do


def problem(cu, T, Hq, Hkv, D, base, mode=orc.MASK_ANCHOR, pos=orc.POS_RESET, layout=orc.ROPE_ADJACENT,
            shift=0):
    return orc.Problem(cu, T, Hq, Hkv, D, base, mode, pos, layout, pos_shift=shift)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_forward(o, lse, O_ref, L_ref, rows=None, tag=""):
    o = f64(o)
    lse = f64(lse)
    if rows is not None:
        o, lse = o[rows], lse[:, rows]
    err = np.abs(o - O_ref)
    lerr = np.abs(lse - L_ref)
    assert err.max() <= O_MAX, f"{tag} O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{tag} O mean-abs {err.mean():.3e}"
    assert lerr.max() <= LSE_MAX, f"{tag} LSE max-abs {lerr.max():.3e}"
    return float(err.max()), float(err.mean())


def rel_l2(got, ref):
    got = f64(got) if isinstance(got, torch.Tensor) else got
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


# Error of the library's fp32 rotation before its bf16 rounding, in units of
# u = 2^-24 times the pair's magnitude. A tile row's (cos, sin) is either a
# two-level table value (two fp64 -> fp32 roundings and one fp32 angle
# addition: at most 3u per component, 3*sqrt(2)u for the pair) or the previous
# row's value advanced by one complex step (cos theta_p, sin theta_p): the
# step's own fp32 rounding (sqrt(2)u/2) plus the product's roundings (2*sqrt(2)u)
# add at most 4.3u per step, and a 16-row unit takes at most 15 steps from its
# table value. The rotation itself adds at most 3u. Total < 4.3 + 15 * 4.3 + 3
# = 72u; the bound takes 96u (a third of margin).
ROT_U = 96 * 2.0 ** -24


def bf16_ulp(x):
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 1e-30)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def pair_norm(x, layout=orc.ROPE_ADJACENT):
    """|(a, b)| of the rotated pair each element of x [..., d] belongs to."""
    d = x.shape[-1]
    if layout == orc.ROPE_ADJACENT:
        n = np.sqrt(x[..., 0::2] ** 2 + x[..., 1::2] ** 2)
        return np.repeat(n, 2, axis=-1)
    n = np.sqrt(x[..., : d // 2] ** 2 + x[..., d // 2:] ** 2)
    return np.concatenate([n, n], axis=-1)


def rope_bound(ref, x, layout=orc.ROPE_ADJACENT):
    """Bound on |library rotation (bf16) - exact rotation| elementwise: the fp32
    rotation's error plus one bf16 rounding of its result (a full ulp of the
    reference covers a result that crosses a binade boundary)."""
    return bf16_ulp(ref) + ROT_U * pair_norm(x, layout)
