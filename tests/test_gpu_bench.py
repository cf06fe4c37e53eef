"""bench.py's own arm on the GPU: a short run prints one JSON line with the
contract's keys (roofline of the dominant kernel, end-to-end leg with its
copied bytes, launch count, clocks sampled in the timed region)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_keeps_the_contract():
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5",
                        "--warmup", "3", "--no-cpu-baseline"],
                       capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["steps"] == 5 and d["warmup"] == 3
    assert d["n_gpus"] == 1 and d["scaling"] == "weak" and "workload" in d["config"]
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 4 * d["steps"]  # two softmax launches and two TopK per step
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    pw = d["per_workload"]
    for key in ("softmax_4096x32000_f32", "softmax_8192x128256_bf16", "topk_256x50257_f32_K8",
                "topk_256x50257_f32_K64", "softmax_64x1024_f32", "causal_1048576x128_f32",
                "increasing_65536x4096_f32", "softmax_4096x50257_f32",
                "softmax_8192x128256_bf16_stream_poly"):
        assert pw[key]["gbs"] > 0 and pw[key]["ms"] > 0, key
    step = ("softmax_4096x32000_f32", "softmax_8192x128256_bf16", "topk_256x50257_f32_K8",
            "topk_256x50257_f32_K64")
    for key in step:  # own-loop times plus the in-step attribution
        assert pw[key]["in_step_ms"] > 0 and pw[key]["timing"], key
    assert abs(sum(pw[key]["in_step_share"] for key in step) - 1.0) < 1e-3
    assert pw[r["workload"]]["timed_region_ms"] > 0  # the roofline kernel, timed in the timed region
    assert e["link"]["h2d_gbs"] > 0 and e["link"]["d2h_gbs"] > 0 and e["frac_of_link_bound"] > 0
    assert d["unfused_baselines"]["softmax_4096x32000_f32"]["safe_over_online"] > 0
    assert d["stats_and_causal"]["causal_1048576x128_f32"]["read_over_mask"] > 0
    assert d["attention"]["cases"]["d128_full"]["tflops"] > 0
