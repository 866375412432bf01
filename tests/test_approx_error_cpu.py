"""The approximation-error measurement (bench.py --approx-error) on the CPU.

Its fp64 references are pinned to the oracle (the exact attention and the method
itself), and its error measures to cases with a known answer: an identity projection
(k = n, E = F = I) reproduces attention exactly, and the first theorem's
construction P R^T R V obeys the Johnson-Lindenstrauss rate, error ~ 1/sqrt(k)
whatever n ("Linformer ... 요약 설명", section "Self-Attention is Low Rank").
"""
import numpy as np
import torch

import bench
from oracle import oracle as orc
from rank_linear_complexity_gb300.workloads import BF16, LAYERWISE
from tests.parity import case_inputs


def test_references_match_the_oracle():
    x = case_inputs(1, 2, 96, 64, 16, LAYERWISE, BF16, seed=7)
    _, O = bench.full_attention64(x["Q"][0], x["K"][0], x["V"][0])
    for i in range(2):
        ref = orc.full_attention(x["Q"][0, i], x["K"][0, i], x["V"][0, i])
        assert np.abs(O[i].numpy() - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
    OL = bench.linformer64(x["Q"][0], x["K"][0], x["V"][0], x["E"])
    refL, _ = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], None, None, LAYERWISE)
    assert np.abs(OL.numpy() - refL[0]).max() <= 1e-12 * max(1.0, np.abs(refL).max())


def test_identity_projection_is_exact():
    g = torch.Generator().manual_seed(3)
    Q, K, V = (torch.randn(2, 48, 64, generator=g, dtype=torch.float64) for _ in range(3))
    r = bench.approx_errors(Q, K, V, torch.eye(48, dtype=torch.float64))
    assert r["jl_t1"] < 1e-12 and r["rel_lin"] < 1e-12 and r["jl_lin"] < 1e-12


def test_first_theorem_error_follows_the_lemma():
    g = torch.Generator().manual_seed(5)
    errs = {}
    for n in (256, 1024):
        Q, K, V = (torch.randn(1, n, 64, generator=g, dtype=torch.float64) for _ in range(3))
        for k in (16, 64):
            R = torch.randn(k, n, generator=g, dtype=torch.float64) / k ** 0.5
            errs[n, k] = bench.approx_errors(Q, K, V, R)["jl_t1"]
    for (n, k), e in errs.items():
        assert 0.7 / k ** 0.5 < e < 1.4 / k ** 0.5, (n, k, e)  # about 1/sqrt(k)
    for k in (16, 64):  # and not growing with n
        assert errs[1024, k] < 1.3 * errs[256, k]
