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
