"""The bench's CPU-side pieces: the reference arm's JSON line carries the contract's keys
(it times the oracle on host cores), and the algorithmic work the roofline fractions
divide by matches the workloads' stated sizes."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from swin_window_attention_gb300 import inputs  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "swin_l224_sweep_fwd"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["gpu_launches"] == 0 and d["dtype"] == "f64"


@pytest.mark.parametrize("name,mb", [("swin_l224_s1", 308.96), ("swin_l224_s2", 154.42), ("swin_l224_s3", 77.36),
                                     ("swin_l224_s4", 39.03), ("swin_b224_s1", 411.70)])
def test_forward_bytes_match_the_workload_table(name, mb):
    """qkv read + output write at 8C bytes per token (bf16) + dense bias + mask (s > 0); the
    table's figures also count the [(2M-1)^2, nH] bias table, which the forward does not
    read (it reads the precomputed bias)."""
    wl = inputs.BY_NAME[name]
    table = (2 * wl.M - 1) ** 2 * wl.nH * 4
    assert abs((bench.fwd_bytes(wl) + table) / 1e6 - mb) < 0.006


def test_step_bytes_and_tokens_of_the_sweep():
    sweep = [inputs.BY_NAME[n] for n in bench.SWEEP]
    assert sum(w.tokens for w in sweep) == 266560
    assert abs(sum(bench.fwd_bytes(w) + (2 * w.M - 1) ** 2 * w.nH * 4 for w in sweep) / 1e6 - 579.8) < 0.05


def test_gemm_roofline_takes_the_larger_time():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0}
    r = bench.gemm_roofline(10e9, 1e12, 20.0, peaks)  # 10 ms of HBM, 10 ms of tensor: tie -> hbm
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.5) < 1e-9
    r = bench.gemm_roofline(1e9, 2e12, 40.0, peaks)  # 1 ms of HBM, 20 ms of tensor
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.5) < 1e-9
    wl = inputs.BY_NAME["swin_l224_s1"]
    assert bench.qkv_flops(wl) == 2 * wl.tokens * wl.C * 3 * wl.C
    assert bench.fwd_fp8_bytes(wl) < bench.fwd_bytes(wl)
