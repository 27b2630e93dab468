"""Timing of segment plans (documents given per token) against the same
documents packed contiguously, on the 64K packing: fwd + bwd effective TFLOP/s
(14 * D * Hq * visible pairs / time; both layouts have the same pairs). The
step is aa_fwd + aa_bwd_from_fwd (the training step), or aa_fwd + aa_bwd with
--bwd recompute.

    python -m packed_sequence_rope_gb300.segment_bench [--chunks 4] [--steps 10] [--bwd recompute]

Prints one JSON object per layout.
"""
from __future__ import annotations

import argparse
import json

import numpy as np

from . import binding as B
from aa_synth import WORKLOADS, gaussian_bf16, interleaved_chunks, workload_cu_doclens


def _time(plan, q, k, v, do, steps, recompute):
    import torch
    fws = plan.alloc_fwd_workspace(q.device)
    if recompute:
        bws = plan.alloc_workspace(q.device)
        bwd = lambda o, lse: plan.bwd(q, k, v, o, lse, do, workspace=bws)
    else:
        bws = torch.empty(max(plan.bwd_from_fwd_workspace_bytes(), 256), device=q.device, dtype=torch.uint8)
        bwd = lambda o, lse: plan.bwd_from_fwd(fws, v, o, lse, do, workspace=bws)
    o, lse = plan.fwd(q, k, v, workspace=fws)
    for _ in range(3):
        o, lse = plan.fwd(q, k, v, o=o, lse=lse, workspace=fws)
        bwd(o, lse)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    ev[0].record()
    for _ in range(steps):
        o, lse = plan.fwd(q, k, v, o=o, lse=lse, workspace=fws)
        bwd(o, lse)
    ev[1].record()
    torch.cuda.synchronize()
    plan.check_device_error()
    return ev[0].elapsed_time(ev[1]) / steps


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--chunks", type=int, default=4)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--bwd", choices=["from_fwd", "recompute"], default="from_fwd")
    args = ap.parse_args(argv)
    w = WORKLOADS["llama7b_64k"]
    cu = workload_cu_doclens(w)
    T, Hq, Hkv, D = w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    doc = interleaved_chunks(np.diff(cu), args.chunks, np.random.default_rng(0))
    q = gaussian_bf16((T, Hq, D), 1, "cuda")
    k = gaussian_bf16((T, Hkv, D), 2, "cuda")
    v = gaussian_bf16((T, Hkv, D), 3, "cuda")
    do = gaussian_bf16((T, Hq, D), 4, "cuda")
    for name, kw in (("contiguous", dict(cu_doclens=cu)), (f"interleaved x{args.chunks}", dict(doc_of_token=doc))):
        cu_arg = kw.pop("cu_doclens", None)
        with B.Plan(cu_arg, T, Hq, Hkv, D, w.rope_base, **kw) as p:
            pairs = p.stats()["unmasked_pairs"]
            ms = _time(p, q, k, v, do, args.steps, args.bwd == "recompute")
        print(json.dumps({"layout": name, "workload": "llama7b_64k", "bwd": args.bwd, "ms_per_fwd_bwd": round(ms, 3),
                          "tflops": round(14 * D * Hq * pairs / (ms * 1e-3) / 1e12, 1), "pairs_per_head": pairs}),
              flush=True)


if __name__ == "__main__":
    main()
