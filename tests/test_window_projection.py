"""Pooling and convolution compression ("Linformer ... 요약 설명", section "Additional
Efficiency Techniques").  With a window of s = n / k positions moved by s, both are
linear maps k x n; the oracle's projection through such a map must equal the block
means (pooling) or the strided convolution computed directly (CPU), and the library's
device-built map and forward through it must match (GPU)."""
import numpy as np
import pytest
import torch

import rank_linear_complexity_gb300.linformer as lf
from oracle import oracle as orc
from rank_linear_complexity_gb300.workloads import BF16, LAYERWISE, HEADWISE
from tests.parity import case_inputs, check, host64, to_device


def window_matrix(n, k, weights=None):
    s = n // k
    w = np.full(s, 1.0 / s) if weights is None else np.asarray(weights, np.float64)
    P = np.zeros((k, n))
    for j in range(k):
        P[j, j * s:(j + 1) * s] = w
    return P


@pytest.mark.parametrize("weights", [None, [0.5, -0.25, 1.0, 0.125]])
def test_oracle_projection_through_a_window_is_pooling_or_convolution(weights):
    n, k, d = 64, 16, 64
    x = case_inputs(1, 2, n, d, k, LAYERWISE, BF16, seed=11)
    P = torch.tensor(window_matrix(n, k, weights), dtype=torch.float64)
    _, _, Kb, Vb = orc.linformer_fwd(x["Q"], x["K"], x["V"], P, None, None, LAYERWISE,
                                     return_proj=True)
    s = n // k
    w = np.full(s, 1.0 / s) if weights is None else np.asarray(weights)
    for X, got in ((x["K"], Kb), (x["V"], Vb)):
        X64 = X.double().numpy().reshape(1, 2, k, s, d)
        direct = np.einsum("bhjtc,t->bhjc", X64, w)  # window j: sum_t w_t X[j s + t]
        assert np.abs(got - direct).max() <= 1e-12 * max(1.0, np.abs(direct).max())


@pytest.mark.gpu
@pytest.mark.parametrize("n,k,weights", [(512, 128, None), (384, 128, None),
                                         (1024, 256, [0.25, 0.5, 0.125, -0.5])])
def test_device_window_matrix(n, k, weights):
    w = None if weights is None else torch.tensor(weights, dtype=torch.float32, device="cuda")
    P = lf.window_projection(n, k, w)
    torch.cuda.synchronize()
    ref = torch.tensor(window_matrix(n, k, weights), dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(P.cpu(), ref)
    assert lf.linformer_window_projection(P, None, n, 100, BF16, None) == -2  # n % k != 0


@pytest.mark.gpu
@pytest.mark.parametrize("mode,weights", [(LAYERWISE, None), (HEADWISE, [0.5, 0.25, 0.125, 0.125])])
def test_forward_through_a_window_matches_oracle(mode, weights):
    b, h, n, d, k = 2, 3, 1024, 64, 256
    x = case_inputs(b, h, n, d, k, mode, BF16, seed=21)
    g = to_device(x, torch.device("cuda:0"))
    w = None if weights is None else torch.tensor(weights, dtype=torch.float32, device="cuda")
    P = lf.window_projection(n, k, w)
    O = lf.attention(g["Q"], g["K"], g["V"], P, P if mode == HEADWISE else None, None, mode)
    torch.cuda.synchronize()
    Pc = P.cpu()
    ref, _ = orc.linformer_fwd(x["Q"], x["K"], x["V"], Pc, Pc if mode == HEADWISE else None,
                               None, mode)
    check(host64(O), ref, BF16, f"window mode {mode}")
