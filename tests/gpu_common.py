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
