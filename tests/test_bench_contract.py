"""The benchmark's JSON line: the keys and units every run prints, on both arms.

The reference arm (the fp64 oracle on the host cores) runs on CPU; the GPU arm runs a short q_proj
benchmark and a short run of the seven-projection layer at an eighth of its tokens, and checks the
roofline, CPU-baseline, end-to-end, clock and launch-count records.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*argv, timeout=600):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], cwd=ROOT, capture_output=True,
                         text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _common(d, steps, warmup):
    assert d["metric"].startswith("packed multi-LoRA fwd+bwd tokens/s")
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == steps and d["warmup"] == warmup and d["n_gpus"] == 1 and d["scaling"] == "strong"
    assert d["vs_baseline"] is None
    e = d["e2e"]
    assert set(e) >= {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"} and e["unit"] == "tokens/s"
    c = d["cpu_baseline"]
    assert set(c) >= {"value", "unit", "cores", "kind", "sample"} and c["kind"] == "oracle" and c["cores"] >= 1


def test_reference_arm_line():
    d = _run("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1", "--ref-budget-s", "5")
    _common(d, 2, 1)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    assert d["cpu_baseline"]["value"] == d["value"] == d["e2e"]["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("tiny_f32")
    # the arm times a token sample of the workload: a step's tokens over its time
    assert d["ms_per_step"] > 0 and "tokens" in d["cpu_baseline"]["sample"]


@pytest.mark.gpu
def test_gpu_arm_line():
    d = _run("--workload", "qproj", "--steps", "5", "--warmup", "3", "--cpu-seconds", "1")
    _common(d, 5, 3)
    assert "impl" not in d and d["dtype"] == "bf16" and "MLORA_REUSE_STAGING" in d["options"]
    assert d["config"]["workload"] == "llama3_8b_q_proj_4096x4096_8ad_16384tok"
    assert d["config"]["tokens_per_step"] == 16384
    assert d["ms_per_step"] == pytest.approx(16384 / d["value"] * 1e3, rel=1e-6)
    # 7 launches a step with staging reuse and the AdamW shadow refresh (the first pack is in warm-up)
    assert d["gpu_launches"] == 7 * 5
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"]) and 0.2 < r["frac"] < 1.3
    assert r["kernel"] in ("fwd_gemm", "bwd_gemm")
    e = d["e2e"]
    # X, dY in and Y, dX out, bf16, every step
    assert e["h2d_bytes_per_step"] == 16384 * (4096 + 4096) * 2
    assert e["d2h_bytes_per_step"] == 16384 * (4096 + 4096) * 2
    assert 0 < e["value"] < d["value"] * 1.05
    clk = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clk)
    assert set(d["kernels"]) >= {"shrink", "fwd_gemm", "dH", "dB", "bwd_gemm", "dA", "adamw"}


def test_both_arms_report_the_same_config():
    sys.path.insert(0, ROOT)
    import bench
    for name in ("tiny", "qproj", "layer"):
        wl = bench.workload(name)
        c = bench.config_of(wl, 1)
        assert c == bench.config_of(bench.workload(name), 1) and "options" not in c
        assert c["tokens_per_step"] == wl.N
    c = bench.config_of(bench.workload("layer"), 1)
    assert [p["name"] for p in c["projections"]] == ["q", "k", "v", "o", "gate", "up", "down"]
    assert c["jobs"] == 32 and c["adapters"] == 7 * 32 and c["parallelism"] == "one GPU"


@pytest.mark.gpu
def test_gpu_arm_line_layer():
    """The seven-projection layer (an eighth of its tokens): one step is every projection's forward,
    backward and AdamW, each kernel aggregated over the projections."""
    d = _run("--workload", "layer_eighth", "--steps", "3", "--warmup", "3", "--cpu-seconds", "1",
             "--ref-tokens-per-job", "4")
    _common(d, 3, 3)
    c = d["config"]
    assert len(c["projections"]) == 7 and c["jobs"] == 32
    assert d["ms_per_step"] == pytest.approx(c["tokens_per_step"] / d["value"] * 1e3, rel=1e-6)
    # 7 launches per projection and step with staging reuse and the shadow refresh
    assert d["gpu_launches"] == 7 * 7 * 3
    r = d["roofline"]
    assert r["kernel"] in ("fwd_gemm", "bwd_gemm") and r["launches_per_step"] == 7
    for k in ("shrink", "fwd_gemm", "dH", "dB", "bwd_gemm", "dA", "adamw"):
        assert d["kernels"][k]["launches_per_step"] == 7
        assert set(d["kernels"][k]["by_projection"]) == {"q", "k", "v", "o", "gate", "up", "down"}
    e = d["e2e"]
    N = c["tokens_per_step"]
    width_in = sum(p["d_in"] + p["d_out"] for p in c["projections"])
    assert e["h2d_bytes_per_step"] == N * width_in * 2 == e["d2h_bytes_per_step"]


def test_clock_summary_keeps_the_timed_region():
    """The clock record summarises the samples that arrived inside the timed region, with the
    throttle reasons seen there; with none inside it says so and falls back to the nearest ones."""
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    c.proc = object()
    c.t0, c.t1 = 100.0, 101.0
    idle = "0, 1980, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    capped = "0, 1500, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active"
    hot = "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    c.rows = [(99.5, idle), (100.2, capped), (100.4, hot), (100.6, hot), (101.5, idle), (100.8, "garbled")]
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1390.0 and "note" not in s
    c.rows = [(99.5, idle)]
    s = c.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 1980.0 and "note" in s


@pytest.mark.gpu
def test_gpu_sweep_lines():
    """The packed-vs-sequential sweep on one layer shape at two job counts: one JSON line per point,
    the pack agreeing with the per-adapter PyTorch comparator to bf16 output rounding."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--sweep", "--sweep-layers",
                          "qwen2.5_3b_attn_2048x2048", "--sweep-jobs", "1,4", "--sweep-steps", "2"], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [json.loads(l) for l in out.stdout.splitlines() if l.startswith("{")]
    assert [d["jobs"] for d in lines] == [1, 4]
    for d in lines:
        assert d["sweep"] == "packed_vs_sequential" and d["tokens"] == 1024 * d["jobs"] and d["rank"] == 64
        assert d["packed_ms"] > 0 and d["one_plan_per_job_ms"] > 0 and d["torch_per_adapter_ms"] > 0
        assert d["agreement_rel_frobenius"]["Y"] < 2e-2 and d["agreement_rel_frobenius"]["dX"] < 2e-2
