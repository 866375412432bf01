"""The approximation-error leg of the benchmark on the GPU, at one small (n, k).

"Linformer 요약 설명", section Self-Attention is Low Rank: the first theorem projects
the attention output with a random k x n matrix of N(0, 1/k) entries; by the
Johnson-Lindenstrauss lemma each entry of P R^T R V deviates from P V by about
||p_i|| ||v_c|| / sqrt(k).  approx_error_rows() measures that deviation (jl_t1) and
the deviation of the library's output from the method computed exactly in fp64
(kernel_dev).  The lemma's rate fixes jl_t1 to within a constant factor of 1/sqrt(k)
(the CPU tests pin the factor near one); the kernel's own rounding must stay far below
the method's error.
"""
import math

import pytest

import bench

pytestmark = pytest.mark.gpu


def test_approx_error_rows_small():
    n, k = 512, 64
    rows = bench.approx_error_rows([n], [k], units=4)
    assert len(rows) == 1
    r = rows[0]
    assert r["n"] == n and r["k"] == k
    assert r["kernel_dev"] <= 1e-3, r
    rate = 1.0 / math.sqrt(k)
    assert 0.7 * rate <= r["jl_t1"] <= 1.4 * rate, r
    assert r["rel_lin"] > 100 * r["kernel_dev"], r
