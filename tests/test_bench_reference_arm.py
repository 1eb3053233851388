"""The reference arm of bench.py on the CPU: `--impl reference` times the
fp64 oracle on the host cores and prints the same JSON line as the GPU arm,
for the same metric, unit and workload, with `"impl": "reference"`."""
import json
import os
import subprocess
import sys

import bench
import synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "3", "--ref-rows", "64"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    line = json.loads(lines[0])
    w = synthetic.WORKLOADS[bench.WORKLOAD]

    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s"
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] == 3
    assert line["vs_baseline"] is None and line["data"] == "synthetic"
    assert line["value"] > 0 and line["ms_per_step"] > 0
    cfg = line["config"]
    assert cfg["workload"].startswith("long-sequence causal self-attention")
    assert (cfg["b"], cfg["h"], cfg["n_q"], cfg["n_k"], cfg["d_k"], cfg["d_v"]) == \
        (w.b, w.h, w.n_q, w.n_k, w.d_k, w.d_v)
    base = line["cpu_baseline"]
    assert base["kind"] == "oracle" and base["cores"] >= 1 and base["value"] == line["value"]
    assert "64 query rows" in base["sample"]
    assert isinstance(base["cpu"], str) and base["cpu"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == "TFLOP/s"
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["gpu_launches"] == 0


def test_row_flops_over_every_row_match_the_metric():
    """Summed over every query row, the reference arm's per-row FLOP equals the
    metric's 4 b h n_q n_k d / 2 for causal attention, up to the diagonal:
    row i sees i + 1 keys, so the sum is n (n + 1) / 2 keys per head, not n^2 / 2."""
    import numpy as np
    w = synthetic.WORKLOADS[bench.WORKLOAD]
    rows = np.arange(w.b * w.h * w.n_q, dtype=np.int64)
    ratio = bench._rows_flops(w, rows) / bench.metric_flops(w)
    assert abs(ratio - (w.n_q + 1) / w.n_q) < 1e-12
