"""bench.py on CPU: the reference arm (the oracle timed on the host cores) prints one JSON
line with the contract's keys, the same metric and workload naming as the GPU arm, and
under a multi-rank launch only rank 0 prints; the acceptance curve is computed from the
histogram as the DMTP blog defines it. No GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny",
                        "--steps", "2", "--warmup", "3"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_reference_line_keys():
    sys.path.insert(0, ROOT)
    import bench
    from synth import CONFIGS
    lines = _run()
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0
    assert d["config"]["workload"] == bench.workload_name(CONFIGS["tiny"], 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_other_ranks_print_nothing():
    assert _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []


def test_acceptance_curve_from_histogram():
    """P(accept length >= k) from per-n counts: a hand-worked histogram."""
    sys.path.insert(0, ROOT)
    import bench
    # 10 sequence-rounds: 4 accepted no draft (length 1), 3 accepted 2 (length 3),
    # 2 accepted 6 (length 7), 1 accepted all 7 (length 8)
    a = bench.acceptance([4, 0, 3, 0, 0, 0, 2, 1])
    assert a["hist_n_accepted"] == [4, 0, 3, 0, 0, 0, 2, 1]
    assert a["p_len_ge"] == [1.0, 0.6, 0.6, 0.3, 0.3, 0.3, 0.3, 0.1]
    assert a["first_candidate"] == pytest.approx(0.6)           # 1 - 4/10
    assert bench.acceptance([0] * 8)["p_len_ge"] == [0.0] * 8
    assert bench.acceptance([0] * 8)["first_candidate"] == 0.0
