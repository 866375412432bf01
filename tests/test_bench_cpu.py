"""Host-side arithmetic of bench.py: the valid-rows roofline terms of ragged batches."""
import dataclasses

import pytest

import bench
from rank_linear_complexity_gb300.workloads import WORKLOADS


@pytest.mark.parametrize("idx", range(len(WORKLOADS)))
def test_valid_rows_equal_the_dense_figures_at_full_length(idx):
    w = WORKLOADS[idx]
    dense = bench.algorithmic(w)
    va = bench.valid_rows_algorithmic(w, [w.n] * w.b)
    assert va["total_bytes"] == dense["total_bytes"]
    assert va["total_flop"] == dense["total_flop"]


def test_valid_rows_scale_with_the_valid_rows_only():
    w = dataclasses.replace(WORKLOADS[4], b=2)          # bf16, per-head, ragged
    full = bench.valid_rows_algorithmic(w, [w.n, w.n])
    half = bench.valid_rows_algorithmic(w, [w.n, 0])     # one sequence empty
    es, units_rows = 2, w.h * w.n
    assert full["total_flop"] - half["total_flop"] == 8.0 * units_rows * w.k * w.d
    # Q, K and V of the empty sequence are not read; its O is still written
    assert full["total_bytes"] - half["total_bytes"] == 3 * units_rows * w.d * es
    clamped = bench.valid_rows_algorithmic(w, [w.n + 5, -3])
    assert clamped == half


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON line
    with the fields the measurement contract asks for; a tiny time budget here."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "3", "--ref-budget-s", "3"],
                         capture_output=True, text=True, timeout=600, cwd=root,
                         env=dict(os.environ, RANK="0", WORLD_SIZE="1"))
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["unit"] == "Mtokens/s" and j["value"] > 0
    assert j["steps"] == 2 and j["warmup"] == 3 and j["higher_is_better"] is True
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["cpu_baseline"]["value"] == j["value"]
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert j["config"]["workload"] == "bf16_b16h12_n4096_k256_layerwise"
