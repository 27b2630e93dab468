"""Shift-discrepancy measurements with this library's kernels.

Kernel-level version of the protocol behind Figure 1 of "When Precision Meets
Position" (architecture page, §3.4 "Diagnostic Methodology: Measuring the
Breakdown"): one sequence of length L = 4096 under the causal mask, Δ2 = 16
fixed and Δ1 swept, Eq. 4's D for each pair; Eq. 5's D_logit for
(Δ1, Δ2) = (0, 16) as L grows from 64 to 8192. There are no model weights
here: q and k are seeded N(0, 1) bf16 tensors shaped like one attention layer
(32 heads, d = 128, RoPE base 1e4), averaged over a few seeds. A last block
compares the masks on a 64K packing (causal over the packing against
AnchorAttention with reset or continuous position IDs).

    python -m packed_sequence_rope_gb300.diagnostics [--seeds N]

Prints one JSON object per measurement.
"""
from __future__ import annotations

import argparse
import json

import numpy as np

from . import binding as B
from aa_synth import WORKLOADS, gaussian_bf16, workload_cu_doclens

MASK_CAUSAL, MASK_ANCHOR = 0, 2
POS_RESET, POS_CONTINUOUS = 0, 1
DELTA1 = [0, 2, 4, 6, 8, 10, 12, 14, 15, 17, 18, 20, 22, 50, 100, 200, 500, 1000, 2000]
LENGTHS = [64, 128, 256, 512, 1024, 2048, 4096, 8192]


def _measure(cu, T, H, d, base, mode, pos_mode, d1, d2, seeds, timing=False):
    import torch
    p1 = B.Plan(cu, T, H, H, d, base, mode, pos_mode, pos_shift=d1)
    p2 = B.Plan(cu, T, H, H, d, base, mode, pos_mode, pos_shift=d2)
    vals, ms = [], None
    with p1, p2:
        for s in range(seeds):
            q = gaussian_bf16((T, H, d), 1000 + 2 * s, "cuda")
            k = gaussian_bf16((T, H, d), 1001 + 2 * s, "cuda")
            _, _, res = p1.shift_diag(p2, q, k)
            vals.append(res[:2].cpu().numpy())
            if timing and s == 0:
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                ev[0].record()
                p1.shift_diag(p2, q, k)
                ev[1].record()
                torch.cuda.synchronize()
                ms = ev[0].elapsed_time(ev[1])
        p1.check_device_error()
    v = np.mean(vals, axis=0)
    return float(v[0]), float(v[1]), ms


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--seeds", type=int, default=4)
    args = ap.parse_args(argv)
    H, d, base = 32, 128, 1e4
    for d1 in DELTA1:
        D, Dl, ms = _measure(None, 4096, H, d, base, MASK_CAUSAL, POS_RESET, d1, 16, args.seeds, timing=d1 == 0)
        rec = {"figure": "D vs delta1", "L": 4096, "delta1": d1, "delta2": 16, "D": D, "D_logit": Dl}
        if ms is not None:
            rec["ms_per_call"] = round(ms, 3)
        print(json.dumps(rec), flush=True)
    for L in LENGTHS:
        D, Dl, _ = _measure(None, L, H, d, base, MASK_CAUSAL, POS_RESET, 0, 16, args.seeds)
        print(json.dumps({"figure": "D_logit vs length", "L": L, "delta1": 0, "delta2": 16, "D": D,
                          "D_logit": Dl}), flush=True)
    w = WORKLOADS["llama7b_64k"]
    cu = workload_cu_doclens(w)
    for name, mode, pos in (("causal", MASK_CAUSAL, POS_RESET), ("anchor+reset", MASK_ANCHOR, POS_RESET),
                            ("anchor+continuous", MASK_ANCHOR, POS_CONTINUOUS)):
        D, Dl, ms = _measure(cu, w.total_tokens, w.num_q_heads, w.head_dim, w.rope_base, mode, pos, 0, 16, 1,
                             timing=True)
        print(json.dumps({"figure": "64K packing", "mask": name, "delta1": 0, "delta2": 16, "D": D,
                          "D_logit": Dl, "ms_per_call": round(ms, 3)}), flush=True)


if __name__ == "__main__":
    main()
