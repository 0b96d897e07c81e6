"""The benchmark's output on a B300: each pass prints exactly one JSON line that carries
every key of its contract, with numbers that agree with one another (throughput against
the step time and the work, the roofline fraction against its parts, end-to-end bytes
counted from the copied tensors)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu

KEYS = ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
        "e2e", "gpu_launches", "clocks"]
ROOFLINE = ["bound", "achieved", "peak", "unit", "frac", "traffic"]


def _run(*args):
    out = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-3000:]
    return json.loads(lines[0])


def _check_common(line, steps):
    for k in KEYS:
        assert k in line, k
    roof = line["roofline"]
    for k in ROOFLINE:
        assert k in roof, k
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    assert line["n_gpus"] == 1 and line["steps"] == steps and line["warmup"] >= 3
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["gpu_launches"] >= steps
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert "workload" in line["config"]
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    clk = line["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clk)


def test_forward_line():
    line = _run("--workload", "t2048_w256_s64", "--steps", "4", "--warmup", "3",
                "--cpu-budget", "2", "--no-secondary")
    _check_common(line, 4)
    c = line["config"]
    flops = 4.0 * c["d"] * c["B"] * c["H"] * c["pairs_per_head"]
    assert line["value"] == pytest.approx(flops / (line["ms_per_step"] / 1e3) / 1e12, rel=1e-6)
    # a 2048-token step is bound by HBM traffic: GB/s of Q, K, V, O and LSE bytes
    roof = line["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    algo = c["B"] * c["H"] * c["T"] * (4 * c["d"] * 2 + 4)
    assert roof["achieved"] == pytest.approx(algo / (line["ms_per_step"] / 1e3) / 1e9, rel=1e-6)
    assert "secondary" not in line
    # inputs in, output and LSE out: bf16 q, k, v and O, fp32 LSE
    elems = c["B"] * c["H"] * c["T"] * c["d"]
    assert line["e2e"]["h2d_bytes_per_step"] == 3 * 2 * elems
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["cores"] >= 1 and cpu["sample"]


def test_forward_line_secondary_workloads():
    """The default forward run also times the other workloads, each with its own clocks,
    and compares the 128K / 8K cost ratio with their pair ratio."""
    line = _run("--workload", "t512_w128_s64", "--steps", "3", "--warmup", "3",
                "--no-cpu-baseline")
    sec = line["secondary"]
    for name in ["t128k_w4096_s1024", "t8k_full_causal", "t16k_r256_s16_g128",
                 "t2048_w256_s0", "t4096_bigbird", "t32k_w512_d2"]:
        e = sec[name]
        assert e["ms_per_step"] > 0 and 0 < e["frac"] == pytest.approx(e["achieved"] / e["peak"])
        assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(e["clocks"])
        flops = 4.0 * e["d"] * e["B"] * e["H"] * e["pairs_per_head"]
        assert e["tflops"] == pytest.approx(flops / (e["ms_per_step"] / 1e3) / 1e12, rel=1e-6)
    assert sec["t2048_w256_s0"]["bound"] == "hbm" and sec["t16k_r256_s16_g128"]["bound"] == "tensor"
    dens = sec["density"]
    assert dens["pairs_ratio_128k_over_8k"] == pytest.approx(536_420_352 / 33_558_528)
    # density-proportional cost: the 128K step costs about its pair ratio in SM cycles
    assert 0.5 * dens["pairs_ratio_128k_over_8k"] < dens["cycles_ratio"] < 2 * dens["pairs_ratio_128k_over_8k"]


def test_backward_line():
    line = _run("--pass", "bwd", "--workload", "t2048_w256_s64", "--steps", "4", "--warmup", "3")
    _check_common(line, 4)
    c = line["config"]
    flops = 10.0 * c["d"] * c["B"] * c["H"] * c["pairs_per_head"]
    assert line["value"] == pytest.approx(flops / (line["ms_per_step"] / 1e3) / 1e12, rel=1e-6)
    elems = c["B"] * c["H"] * c["T"] * c["d"]
    # q, k, v, O, dO (bf16) and LSE (fp32) in; dQ, dK, dV out
    assert line["e2e"]["h2d_bytes_per_step"] == 5 * 2 * elems + 4 * c["B"] * c["H"] * c["T"]
    assert line["e2e"]["d2h_bytes_per_step"] == 3 * 2 * elems


def test_decode_line():
    line = _run("--pass", "decode", "--decode-workload", "decode_b8_w4096", "--steps", "5",
                "--warmup", "3")
    _check_common(line, 5)
    c = line["config"]
    assert line["roofline"]["bound"] == "hbm" and line["unit"] == "GB/s"
    kv = c["B"] * c["Hkv"] * c["window"] * c["d"] * 2 * 2
    assert line["value"] * line["ms_per_step"] / 1e3 * 1e9 >= kv  # at least the cache is counted
    assert line["gpu_launches"] == 2 * 5
