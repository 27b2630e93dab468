"""The multi-rank bench plumbing (replicas under torchrun) on CPU with gloo:
the step time every rank reports is the maximum over ranks, and the
reference arm prints only on rank 0."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    r, w = bench._dist()
    t = bench._max_over_ranks(10.0 + 5 * rank, w)
    bench._barrier(w)
    q.put((r, w, t))
    torch.distributed.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 2, 15.0), (1, 2, 15.0)]


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny_256"], capture_output=True, text=True, env=env,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_json_line():
    # single process: one JSON line with the bench contract's keys; the
    # reference arm's cpu_baseline and e2e restate its own value
    import json
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny_256", "--cpu-budget", "1"], capture_output=True,
                       text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["config"]["workload"] == "tiny_256"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_traffic_record_follows_code_not_comments(tmp_path):
    # the stored DRAM traffic stays valid across comment edits of the kernel
    # source and is dropped once its code changes
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k(int* x) {\n  x[0] = 1;  // one\n}\n")
    h0 = bench.code_hash(str(src))
    src.write_text("// a kernel\n__global__ void k(int* x) {\n    x[0] = 1;   // the first element\n}\n")
    assert bench.code_hash(str(src)) == h0
    src.write_text("__global__ void k(int* x) {\n  x[0] = 2;\n}\n")
    assert bench.code_hash(str(src)) != h0
    rec = bench._captured_traffic("llama7b_64k:attn_bwd_kernel")
    assert rec is None or rec > 0
