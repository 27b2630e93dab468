"""GPU: the benchmark's own JSON line carries every key of its contract.

`python bench.py` prints one JSON line per run; this runs it with few steps on
the 64K workload and checks the keys, their types and the relations between
them: the device-timed value from ms_per_step and the visible pairs
(14·D·Hq·P flops per step), the dominant kernel's roofline fraction, the end-to-end
figure with the bytes it copies, the kernel launches and the clock record.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "4", "--warmup", "3", "--no-other-configs",
         "--no-compare-causal", "--cpu-budget", "2"],
        cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_contract_keys_and_types(line):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 4 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["dtype"] == "bf16"
    assert line["unit"] == "TFLOP/s" and line["value"] > 0 and line["ms_per_step"] > 0
    cfg = line["config"]
    assert cfg["workload"] == "llama7b_64k" and cfg["total_tokens"] == 65536 and cfg["head_dim"] == 128
    # value = 14 D Hq P flops per step over the measured step time
    flops = 14.0 * cfg["head_dim"] * cfg["num_q_heads"] * cfg["unmasked_pairs_per_head"]
    assert abs(flops / (line["ms_per_step"] * 1e-3) / 1e12 - line["value"]) <= 1e-3 * line["value"] + 0.05


def test_roofline_e2e_launches_and_clocks(line):
    rf = line["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in rf, key
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s"
    assert abs(rf["achieved"] / rf["peak"] - rf["frac"]) <= 1e-3
    assert 0.0 < rf["frac"] < 1.5
    e2e = line["e2e"]
    T, Hq, Hkv, D = (line["config"][k] for k in ("total_tokens", "num_q_heads", "num_kv_heads", "head_dim"))
    # in: q, k, v, dout; out: o, lse, dq, dk, dv (bf16 tensors, fp32 lse)
    assert e2e["h2d_bytes_per_step"] == 2 * T * D * (Hq + Hkv + Hkv + Hq)
    assert e2e["d2h_bytes_per_step"] == 2 * T * D * (Hq + Hq + Hkv + Hkv) + 4 * Hq * T
    assert 0 < e2e["value"] <= line["value"] and e2e["unit"] == line["unit"]
    assert line["gpu_launches"] == 7 * line["steps"]
    ck = line["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(ck)
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0
