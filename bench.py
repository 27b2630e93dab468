"""Benchmark: fused RoPE + AnchorAttention forward + backward on one GB300.

A step is one aa_fwd + one aa_bwd_from_fwd over one synthetic packing (the
64K long-context training shape by default: T = 65536, 32 heads MHA, head_dim
128, RoPE base 5e6, log-normal document lengths with median 1500): the
forward rotates Q and K once and the backward reads them from the forward's
workspace, as a training step that keeps that workspace for the backward
does (--bwd recompute times aa_bwd, which rotates them again). Inputs (Q, K,
V, dO: 2 GiB) are far larger than L2, so no flush runs between steps.

Metric: effective TFLOP/s = 14 * D * Hq * P / (t_fwd + t_bwd), where P counts
the visible (query, key) pairs of the mask, anchor pairs included (4*D flops
per pair forward, 10*D backward); masked or padded work is not credited.

The default line also carries `other_configs`: GQA 128K and the 64K
mask-paradigm sweep (a few steps each, after the main timed region).
--chunks N times the same documents cut into N chunks each and interleaved
(a segment plan, documents given per token).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas, weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from aa_synth import WORKLOADS, make_qkv, workload_cu_doclens  # noqa: E402

METRIC = "AnchorAttention fwd+bwd effective TFLOP/s @64K packed bf16; % of GB300 BF16 peak"
UNIT = "TFLOP/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), float(d["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    return rank, world


def _max_over_ranks(x, world):
    import torch
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _barrier(world):
    import torch
    if world > 1:
        torch.distributed.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def code_hash(path):
    """sha256 of a C/CUDA source with its // comments and all whitespace removed:
    it changes when the code does, not when a comment is edited."""
    import hashlib
    import re
    text = open(path, encoding="utf-8").read()
    code = "".join(re.sub(r"//.*", "", line) for line in text.splitlines())
    return hashlib.sha256(re.sub(r"\s+", "", code).encode()).hexdigest()


def _captured_traffic(key):
    """DRAM bytes per launch of the dominant kernel from the committed ncu capture
    (profiles/traffic.json), or None when there is none or the kernel's code has
    changed since the counters were taken."""
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(tpath)).get(key)
        if code_hash(os.path.join(ROOT, rec["kernel_source"])) != rec["code_sha256"]:
            return None
        return int(rec["bytes"])
    except Exception:
        return None


# ----------------------------------------------------------------------------- our path
def run_ours(args):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import packed_sequence_rope_gb300 as aa

    rank, world = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    cu = workload_cu_doclens(w)
    T, Hq, Hkv, D = w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    mask = {"anchor": aa.MASK_ANCHOR, "intra_doc": aa.MASK_INTRA_DOC, "causal": aa.MASK_CAUSAL}[args.mask]
    pos = {"reset": aa.POS_RESET, "continuous": aa.POS_CONTINUOUS}[args.pos]
    q, k, v, do = make_qkv(w, device=dev)
    layout = "contiguous"
    if args.chunks > 0:
        # the same documents cut into chunks and interleaved (a segment plan:
        # documents given per token); the visible pairs are unchanged
        from aa_synth import interleaved_chunks
        doc = interleaved_chunks(np.diff(cu), args.chunks, np.random.default_rng(0))
        plan = aa.Plan(None, T, Hq, Hkv, D, w.rope_base, mask, pos, doc_of_token=doc)
        layout = f"interleaved chunks x{args.chunks}"
    else:
        plan = aa.Plan(cu, T, Hq, Hkv, D, w.rope_base, mask, pos)
    st = plan.stats()
    work = plan.work()
    P = st["unmasked_pairs"]
    flops_fwd = 4.0 * D * Hq * P
    flops_bwd = 10.0 * D * Hq * P
    o = torch.empty_like(q)
    lse = torch.empty(Hq, T, device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fws = plan.alloc_fwd_workspace(dev)
    stream = torch.cuda.current_stream()
    bwd = _bwd_call(plan, args.bwd, q, k, v, o, lse, do, dq, dk, dv, fws, dev)
    # fwd: K and Q rotation + attention; bwd: (K and Q rotation,) prep, tile
    # kernel, dq finalize (+ anchor)
    n_launch_per_step = 3 + 3 + (2 if args.bwd == "recompute" else 0) + (1 if mask == aa.MASK_ANCHOR else 0)
    if args.chunks > 0:
        # the forward gathers v into its grouped order (aa_bwd gathers it again)
        n_launch_per_step += 1 + (0 if args.bwd == "from_fwd" else 1)

    def step():
        plan.fwd(q, k, v, o, lse, fws)
        bwd()

    for _ in range(args.warmup):
        step()
    plan.check_device_error()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    # torch creates events lazily and only times events it has recorded: record
    # the hook's pair once here so the library re-records existing handles
    for e in ev:
        e[2].record(stream)
        e[3].record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    _barrier(world)
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        e = ev[s]
        e[0].record(stream)
        plan.fwd(q, k, v, o, lse, fws)
        e[1].record(stream)
        plan.set_bwd_timing_events(e[2], e[3])
        bwd()
        e[4].record(stream)
    t_stop.record(stream)
    _barrier(world)
    clk = clocks.stop()
    plan.set_bwd_timing_events(None, None)
    plan.check_device_error()
    total_ms = t_start.elapsed_time(t_stop)
    t_fwd = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)]
    t_bwd = [ev[s][1].elapsed_time(ev[s][4]) for s in range(args.steps)]
    t_bwd_main = [ev[s][2].elapsed_time(ev[s][3]) for s in range(args.steps)]
    total_ms = _max_over_ranks(total_ms, world)
    ms_step = total_ms / args.steps
    value = world * (flops_fwd + flops_bwd) / (ms_step * 1e-3) / 1e12
    burst, sustained, hbm, peak_src = _peaks()
    fwd_ms = float(np.mean(t_fwd))
    bwd_ms = float(np.mean(t_bwd))
    bwd_main_ms = float(np.mean(t_bwd_main))
    # dominant kernel: the backward tile kernel (10*D flops per visible pair)
    dom_flops = flops_bwd
    dom_ms = bwd_main_ms
    dom_name = "attn_bwd_kernel"
    if fwd_ms > bwd_main_ms:
        dom_flops, dom_ms, dom_name = flops_fwd, fwd_ms, "attn_fwd_kernel"
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    traffic = _captured_traffic(f"{args.workload}:{dom_name}")

    extra = {}
    if args.compare_causal and mask != aa.MASK_CAUSAL and rank == 0:
        extra["speedup_vs_causal"] = _causal_speedup(aa, w, q, k, v, do, dev, ms_step, args)
    if args.other_configs and rank == 0 and world == 1 and args.chunks == 0 and w.name == "llama7b_64k":
        causal = extra.get("speedup_vs_causal", {}).get("causal_ms_per_step")
        del q, k, v, do, o, lse, dq, dk, dv, fws, bwd
        torch.cuda.empty_cache()
        t0 = time.perf_counter()
        extra["other_configs"] = _other_configs(aa, dev, args, causal)
        extra["other_configs"]["wall_s"] = round(time.perf_counter() - t0, 1)

    e2e = _e2e(aa, plan, w, dev, args, flops_fwd + flops_bwd, world) if not args.no_e2e else None
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu = cpu_baseline(w, cu, mask, pos, budget_s=args.cpu_budget)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V/dO, seeded log-normal document lengths)",
        "config": {"workload": w.name, "layout": layout, "total_tokens": T, "num_q_heads": Hq, "num_kv_heads": Hkv,
                   "head_dim": D, "rope_base": w.rope_base, "mask": args.mask, "pos": args.pos,
                   "documents": int(len(cu) - 1), "unmasked_pairs_per_head": P,
                   "l2": "inputs (2 GiB) larger than L2; no flush", "parallelism": f"replicas x{world}"},
        "bwd_entry": "aa_bwd_from_fwd" if args.bwd == "from_fwd" else "aa_bwd",
        "fwd_ms": round(fwd_ms, 4), "bwd_ms": round(bwd_ms, 4), "bwd_main_kernel_ms": round(bwd_main_ms, 4),
        "fwd_tflops": round(flops_fwd / (fwd_ms * 1e-3) / 1e12, 2),
        "bwd_tflops": round(flops_bwd / (bwd_ms * 1e-3) / 1e12, 2),
        "pct_of_bf16_peak_burst": round(100 * value / world / burst, 2),
        "pct_of_bf16_peak_sustained": round(100 * value / world / sustained, 2),
        "skipped_tile_fraction": round(1 - st["live_tiles"] / st["causal_tiles"], 4),
        "tiles": {"live": st["live_tiles"], "causal": st["causal_tiles"], "fwd_tiles": work["fwd_tiles"],
                  "bwd_tiles": work["bwd_tiles"]},
        "roofline": {"bound": "tensor", "kernel": dom_name, "achieved": round(achieved, 2),
                     "peak": burst, "unit": "TFLOP/s", "frac": round(achieved / burst, 4),
                     "peak_kind": f"bf16 burst ({peak_src}): the timed region is short and runs at the "
                                  f"maximum clock", "frac_of_sustained": round(achieved / sustained, 4),
                     "traffic": traffic,
                     "traffic_source": "DRAM bytes per launch from the committed ncu capture of this kernel "
                                       "(profiles/traffic.json, checked against a hash of the kernel source's code; "
                                       "null once the code changed), not measured in this run"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": n_launch_per_step * args.steps,
        "clocks": clk,
        "context": "pages: >50% training-time saving vs full attention (~4.5 -> ~2 days per 1B tokens, "
                   "64K, 8x A100, Ulysses); not comparable hardware",
    }
    line.update(extra)
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def _time_steps(plan, fwd, bwd, steps, warmup):
    """Mean ms per fwd+bwd step (CUDA events on the current stream) after
    `warmup` untimed steps; the library's error word is checked after both."""
    import torch
    for _ in range(warmup):
        fwd()
        bwd()
    plan.check_device_error()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(steps):
        fwd()
        bwd()
    z.record()
    torch.cuda.synchronize()
    plan.check_device_error()
    return a.elapsed_time(z) / steps


def _other_configs(aa, dev, args, causal_ms_64k):
    """The secondary configurations, a few timed steps each: GQA 128K, and the
    mask-paradigm sweep at 64K (document-length medians 512 / 1500 (the main
    packing) / 4096 / one document under CAUSAL, INTRA_DOC + RESET, ANCHOR +
    RESET and ANCHOR + CONTINUOUS) with the skipped-tile fraction and the
    speedup over the same kernels on the causal mask. The causal step ignores
    the documents, so one causal timing (the main workload's, same shape)
    serves every 64K sweep point; the main packing's ANCHOR + RESET point is
    the headline line itself."""
    import torch
    out = {}
    runs = [("gqa_128k", "anchor", "reset")]
    for wname in ("sweep_64k_m512", "llama7b_64k", "sweep_64k_m4096", "sweep_64k_single"):
        if wname != "llama7b_64k":
            runs += [(wname, "intra_doc", "reset"), (wname, "anchor", "reset")]
        runs.append((wname, "anchor", "continuous"))
    for name, mname, pname in runs:
        w = WORKLOADS[name]
        cu = workload_cu_doclens(w)
        T, Hq, Hkv, D = w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
        mask = {"anchor": aa.MASK_ANCHOR, "intra_doc": aa.MASK_INTRA_DOC}[mname]
        pos = {"reset": aa.POS_RESET, "continuous": aa.POS_CONTINUOUS}[pname]
        q, k, v, do = make_qkv(w, device=dev)
        with aa.Plan(cu, T, Hq, Hkv, D, w.rope_base, mask, pos) as p:
            st = p.stats()
            o = torch.empty_like(q)
            lse = torch.empty(Hq, T, device=dev, dtype=torch.float32)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            fws = p.alloc_fwd_workspace(dev)
            bwd = _bwd_call(p, args.bwd, q, k, v, o, lse, do, dq, dk, dv, fws, dev)
            ms = _time_steps(p, lambda: p.fwd(q, k, v, o, lse, fws), bwd, args.other_steps, 2)
            flops = 14.0 * D * Hq * st["unmasked_pairs"]
            rec = {"mask": mname, "pos": pname, "documents": int(len(cu) - 1), "ms_per_step": round(ms, 3),
                   "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
                   "skipped_tile_fraction": round(1 - st["live_tiles"] / st["causal_tiles"], 4)}
            if w.total_tokens == 65536 and causal_ms_64k:
                rec["speedup_vs_causal"] = round(causal_ms_64k / ms, 3)
            out[f"{name}:{mname}" + (":continuous" if pname == "continuous" else "")] = rec
            del bwd, fws, o, lse, dq, dk, dv
        del q, k, v, do
        torch.cuda.empty_cache()
    if causal_ms_64k:
        w = WORKLOADS["llama7b_64k"]
        out["sweep_64k:causal"] = {"mask": "causal", "ms_per_step": round(causal_ms_64k, 3),
                                   "tflops": round(14.0 * w.head_dim * w.num_q_heads * w.total_tokens
                                                   * (w.total_tokens + 1) / 2 / (causal_ms_64k * 1e-3) / 1e12, 2),
                                   "skipped_tile_fraction": 0.0, "speedup_vs_causal": 1.0,
                                   "note": "the causal mask ignores the documents: one timing for every 64K point"}
    return out


def _bwd_call(plan, kind, q, k, v, o, lse, do, dq, dk, dv, fws, dev):
    """The step's backward call with its workspace: aa_bwd_from_fwd reading the
    rotated Q and K from the forward workspace `fws`, or aa_bwd (recompute)."""
    import torch
    if kind == "from_fwd":
        ws = torch.empty(max(plan.bwd_from_fwd_workspace_bytes(), 256), device=dev, dtype=torch.uint8)
        return lambda: plan.bwd_from_fwd(fws, v, o, lse, do, dq, dk, dv, ws)
    ws = plan.alloc_workspace(dev)
    return lambda: plan.bwd(q, k, v, o, lse, do, dq, dk, dv, ws)


def _causal_speedup(aa, w, q, k, v, do, dev, ms_anchor, args):
    import torch
    T, Hq, Hkv, D = w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    with aa.Plan(None, T, Hq, Hkv, D, w.rope_base, aa.MASK_CAUSAL) as pc:
        o = torch.empty_like(q)
        lse = torch.empty(Hq, T, device=dev, dtype=torch.float32)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        fws = pc.alloc_fwd_workspace(dev)
        bwd = _bwd_call(pc, args.bwd, q, k, v, o, lse, do, dq, dk, dv, fws, dev)
        for _ in range(1):
            pc.fwd(q, k, v, o, lse, fws)
            bwd()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = 2
        a.record()
        for _ in range(n):
            pc.fwd(q, k, v, o, lse, fws)
            bwd()
        b.record()
        torch.cuda.synchronize()
        pc.check_device_error()
        ms_causal = a.elapsed_time(b) / n
        del bwd
    return {"causal_ms_per_step": round(ms_causal, 3), "speedup": round(ms_causal / ms_anchor, 3)}


def _gpu_numa_node(dev):
    """The NUMA node the GPU's PCI function reports (sysfs) and that node's
    CPUs, or (None, None) where the system does not say."""
    import torch
    try:
        pr = torch.cuda.get_device_properties(dev)
        bdf = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bdf}/numa_node") as f:
            node = int(f.read())
        if node < 0:
            return None, None
        cpus = set()
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            for part in f.read().strip().split(","):
                lo, _, hi = part.partition("-")
                cpus.update(range(int(lo), int(hi or lo) + 1))
        return node, cpus
    except (OSError, ValueError, AttributeError):
        return None, None


def _link_probe(h_src, d_dst, d_src, h_dst):
    """Host link bandwidth with the e2e run's own pinned buffers (GB/s): one
    copy host -> device, one device -> host, then both at once (each rate
    over the pair's common wall time). Outside the timed region."""
    import torch
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    nb_in, nb_out = h_src.numel() * h_src.element_size(), d_src.numel() * d_src.element_size()

    def timed(pairs):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in pairs]
        torch.cuda.synchronize()
        for (a, z), (st, dst, src) in zip(ev, pairs):
            a.record(st)
            with torch.cuda.stream(st):
                dst.copy_(src, non_blocking=True)
            z.record(st)
        torch.cuda.synchronize()
        return [a.elapsed_time(z) for a, z in ev]

    timed([(s1, d_dst, h_src), (s2, h_dst, d_src)])  # warm-up
    t_in = timed([(s1, d_dst, h_src)])[0]
    t_out = timed([(s2, h_dst, d_src)])[0]
    both = max(timed([(s1, d_dst, h_src), (s2, h_dst, d_src)]))
    gbs = lambda b, ms: round(b / (ms * 1e-3) / 1e9, 1)
    return {"h2d": gbs(nb_in, t_in), "d2h": gbs(nb_out, t_out),
            "h2d_concurrent": gbs(nb_in, both), "d2h_concurrent": gbs(nb_out, both), "bytes_each": int(nb_in)}


def _e2e(aa, plan, w, dev, args, flops, world):
    """Same step through the public C-ABI with host buffers: every step copies its
    Q/K/V/dO in from pinned host memory, runs fwd + bwd, and copies O, LSE, dQ,
    dK, dV back to pinned host memory, all inside the timed region. The steps
    are pipelined the way a training input pipeline is: step i + 1's inputs go
    in on one stream and step i - 1's results come out on another while step i
    computes (device inputs and outputs double-buffered; events order each
    buffer's reuse)."""
    import torch
    T, Hq, Hkv, D = w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    # pinned host buffers on the GPU's own NUMA node where the system names
    # one (pages land on the node of the thread that first writes them)
    node, cpus = _gpu_numa_node(dev)
    old_aff = os.sched_getaffinity(0)
    if cpus and cpus & old_aff:
        try:
            os.sched_setaffinity(0, cpus & old_aff)
        except OSError:  # a placement hint only
            pass
    try:
        hq, hk, hv, hdo = (t.pin_memory() for t in make_qkv(w, device="cpu"))
        h_out = (torch.empty_like(hq).pin_memory(), torch.empty(Hq, T, dtype=torch.float32).pin_memory(),
                 torch.empty_like(hq).pin_memory(), torch.empty_like(hk).pin_memory(),
                 torch.empty_like(hv).pin_memory())
        for t in h_out:
            t.zero_()
    finally:
        try:
            os.sched_setaffinity(0, old_aff)
        except OSError:
            pass
    h_in = (hq, hk, hv, hdo)
    d_in = [tuple(torch.empty_like(t, device=dev) for t in h_in) for _ in range(2)]
    d_out = [(torch.empty_like(d_in[b][0]), torch.empty(Hq, T, device=dev, dtype=torch.float32),
              torch.empty_like(d_in[b][0]), torch.empty_like(d_in[b][1]), torch.empty_like(d_in[b][2]))
             for b in range(2)]
    fws = plan.alloc_fwd_workspace(dev)
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bwds = []
    for b in range(2):
        q, k, v, do = d_in[b]
        o, lse, dq, dk, dv = d_out[b]
        bwds.append(_bwd_call(plan, args.bwd, q, k, v, o, lse, do, dq, dk, dv, fws, dev))
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    link = _link_probe(hq, d_in[0][0], d_out[0][0], h_out[0])
    link["gpu_numa_node"] = node
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]

    def step(i):
        b = i % 2
        if used[b]:  # buffer b's previous step has been computed and read back
            s_in.wait_event(comp_done[b])
        with torch.cuda.stream(s_in):
            for d_, h_ in zip(d_in[b], h_in):
                d_.copy_(h_, non_blocking=True)
            in_done[b].record(s_in)
        s_comp.wait_event(in_done[b])
        if used[b]:
            s_comp.wait_event(out_done[b])
        with torch.cuda.stream(s_comp):
            q, k, v, _ = d_in[b]
            o, lse = d_out[b][0], d_out[b][1]
            plan.fwd(q, k, v, o, lse, fws, stream=s_comp)
            bwds[b]()
            comp_done[b].record(s_comp)
        s_out.wait_event(comp_done[b])
        with torch.cuda.stream(s_out):
            for h_, d_ in zip(h_out, d_out[b]):
                h_.copy_(d_, non_blocking=True)
            out_done[b].record(s_out)
        used[b] = True

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    n = max(4, args.steps)  # the same K steps as the device-timed value (pipeline fill and drain included)
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(n):
        step(i)
    for b in range(2):
        s_out.wait_event(out_done[b])
    z.record(s_out)
    torch.cuda.synchronize()
    plan.check_device_error()
    ms = _max_over_ranks(a.elapsed_time(z) / n, world)
    return {"value": round(world * flops / (ms * 1e-3) / 1e12, 2), "unit": UNIT, "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipelined": "inputs of step i+1 in and results of step i-1 out on their own streams while step i computes",
            "steps": n,
            "link_gbs": link,
            "link_bound_ms": round(1e3 * max(h2d / (link["h2d_concurrent"] * 1e9), d2h / (link["d2h_concurrent"] * 1e9)), 3)}


# ----------------------------------------------------------------------------- CPU oracle
def cpu_baseline(w, cu, mask, pos, budget_s=15.0):
    """Time the fp64 oracle (as it stands) on whole documents of the same
    packing, one head, until ~budget_s of CPU work; report effective TFLOP/s
    over the visible pairs it processed, scaled per the metric's definition."""
    import torch
    import oracle as orc
    T, D = w.total_tokens, w.head_dim
    qh, kh, vh, doh = make_qkv(w, device="cpu")
    q, k, v, do = (t[:, :1].contiguous() for t in (qh, kh, vh, doh))
    prob = orc.Problem(cu, T, 1, 1, D, w.rope_base, mask, pos)
    lens = np.diff(cu)
    order = np.argsort(lens)
    pairs = 0
    docs = 0
    t0 = time.perf_counter()
    for d in order[len(order) // 4:]:
        a, b = int(cu[d]), int(cu[d + 1])
        rows = np.arange(a, b)
        orc.forward(prob, q, k, v, rows=rows)
        orc.backward(prob, q, k, v, do, rows=rows)
        n = b - a
        pairs += n * (n + 1) // 2 + (n if mask == 2 else 0)
        docs += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(14.0 * D * pairs / dt / 1e12, 6), "unit": UNIT, "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"fp64 numpy oracle fwd+bwd, 1 head, {docs} whole documents of the {w.name} packing "
                      f"({pairs} visible pairs), {dt:.1f} s; BLAS threads = all host cores"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    cu = workload_cu_doclens(w)
    mask = {"anchor": 2, "intra_doc": 1, "causal": 0}[args.mask]
    pos = {"reset": 0, "continuous": 1}[args.pos]
    budget = max(1.0, min(60.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(w, cu, mask, pos, budget_s=budget)
    vals = [cpu_baseline(w, cu, mask, pos, budget_s=budget) for _ in range(args.steps)]
    v = float(np.mean([x["value"] for x in vals]))
    cb = dict(vals[-1])
    cb["value"] = round(v, 6)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "total_tokens": w.total_tokens, "num_q_heads": w.num_q_heads,
                       "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "mask": args.mask, "pos": args.pos},
            "cpu_baseline": cb,
            "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama7b_64k", choices=sorted(WORKLOADS))
    ap.add_argument("--mask", default="anchor", choices=["anchor", "intra_doc", "causal"])
    ap.add_argument("--pos", default="reset", choices=["reset", "continuous"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--compare-causal", action=argparse.BooleanOptionalAction, default=True)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--bwd", choices=["from_fwd", "recompute"], default="from_fwd",
                    help="backward entry point: aa_bwd_from_fwd (default) or aa_bwd")
    ap.add_argument("--chunks", type=int, default=0,
                    help="cut every document into this many chunks and interleave them (a segment plan)")
    ap.add_argument("--other-configs", action=argparse.BooleanOptionalAction, default=True,
                    help="also time GQA 128K and the 64K mask sweep (default workload, one GPU)")
    ap.add_argument("--other-steps", type=int, default=3)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
