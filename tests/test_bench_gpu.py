"""bench.py's JSON line on a real GPU: one short run on the tiny shard, every
key the line promises present and consistent (CPU-side pieces of the bench are
covered by test_bench_helpers.py and test_multirank_cpu.py)."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_bench_line_contract():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "1", "--steps", "20", "--warmup", "3",
           "--no-e2e", "--cpu-seconds", "2", "--extra="]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "clocks", "gpu_launches"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and abs(d["value"] - d["config"]["elements"] / (d["ms_per_step"] * 1e-3)) <= 0.01 * d["value"]
    assert d["config"]["workload"].startswith("tiny") and d["config"]["groups"] == 1
    rf = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in rf, k
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    cb = d["cpu_baseline"]
    for k in ("value", "unit", "cores", "kind", "sample"):
        assert k in cb, k
    assert cb["kind"] == "oracle" and cb["value"] > 0 and set(cb["by_workload"]) == {
        "workload_1", "workload_3", "workload_4", "workload_5"}
    assert d["gpu_launches"] == 20 * (4 + 2)          # 4 accumulate passes, norm finish, fused step
    assert set(d["kernels"]) == {"accumulate_0", "accumulate_1", "accumulate_2", "accumulate_3", "norm_final", "step"}
    assert "cuda_graph_replay" in d["variants"] and "zero_offload" in d["variants"]
