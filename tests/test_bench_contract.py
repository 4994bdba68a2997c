"""The reference arm of bench.py (the CPU oracle timed on a bounded sample)
prints one JSON line with the contract's keys; it needs no GPU."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "single_256x256",
                        "--steps", "2", "--warmup", "1"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["unit"] == "params/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert "workload" in d["config"]


def test_algorithmic_bytes_of_the_vit_b16_list():
    """Per kernel: K0 reads g (4 B per element), K1 reads p, g, m0..2, v
    (24 B), K2 reads them again and writes p, m0..2, v (44 B); a [1 x n]
    view's per-element column accumulators add 24 B to K0 (read, write) and
    12 B to K1 and K2 (read).  The step's dependency-forced floor is 72 B
    per element of a 2-D tensor and 104 B of a [1 x n] view: 6.23 GB per
    step of the ViT-B/16 list, 0.916 ms at 6,795 GB/s."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    states = [dict(zip(("rows", "cols"), synth.rows_cols(s))) for _, s in synth.vit_b16_shapes()]
    k0, k1, k2 = bench.algorithmic_bytes(states)
    n2 = sum(s["rows"] * s["cols"] for s in states if s["rows"] > 1)
    n1 = sum(s["cols"] for s in states if s["rows"] == 1)
    assert n1 + n2 == 86_415_592
    assert (k0, k1, k2) == (4 * n2 + 28 * n1, 24 * n2 + 36 * n1, 44 * n2 + 56 * n1)
    floor = bench.step_floor_bytes(states)
    assert floor == 72 * n2 + 104 * n1 == 6_225_862_208
    assert abs(floor / 6795.1e9 * 1e3 - 0.9162) < 1e-4
