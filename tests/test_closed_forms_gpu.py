"""GPU forward against closed forms computed here in fp64, without the oracle, and a
full grid of sharing mode x data type x ragged lengths against the oracle.

Closed forms ("Linformer(Self-Attention with Linear Complexity) 요약 설명", section Model:
Kbar = E K and Vbar = F V over the valid rows, O = softmax(Q Kbar^T / sqrt(d)) Vbar, padded
query rows zero):
  * Q = 0: every score is 0, the softmax is uniform over the k projected positions, so
    every valid row of O is the mean of the rows of Vbar = F V;
  * k = 1: the softmax of one column is 1, so every valid row of O is the one row of
    Vbar, whatever Q and K are.
"""
import numpy as np
import pytest
import torch

import rank_linear_complexity_gb300.linformer as lf
from oracle import oracle as orc
from rank_linear_complexity_gb300.workloads import (BF16, BF16_F32OUT, F32, HEADWISE, KV,
                                                    LAYERWISE, PER_HEAD)
from tests.parity import case_inputs, check, host64, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
MODES = [PER_HEAD, KV, HEADWISE, LAYERWISE]


def run(x, mode, dtype):
    g = to_device(x, DEV)
    O = lf.attention(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], mode,
                     out_fp32=(dtype == BF16_F32OUT))
    torch.cuda.synchronize()
    assert lf.linformer_debug_read_device_status() == 0
    return host64(O)


def f_hat(x, mode, head):
    """The value projection of head `head` as float64 [k][n] (F, or E where F = E)."""
    P = x["F"] if x["F"] is not None else x["E"]
    P = P.double().numpy()
    return P[head] if mode in (PER_HEAD, KV) else P


def vbar_rows(x, mode):
    """Vbar = F V over the valid rows, float64 [b][h][k][d], written out here."""
    V = x["V"].double().numpy()
    b, h, n, d = V.shape
    L = x["lengths"].numpy() if x["lengths"] is not None else np.full(b, n)
    out = []
    for bi in range(b):
        Lb = int(min(max(L[bi], 0), n))
        out.append([f_hat(x, mode, hi)[:, :Lb] @ V[bi, hi, :Lb] for hi in range(h)])
    return np.array(out), L


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dtype,k", [(BF16, 256), (BF16_F32OUT, 96), (F32, 64)])
def test_zero_queries_give_the_mean_of_vbar(mode, dtype, k):
    b, h, n, d = 2, 3, 700, 64
    x = case_inputs(b, h, n, d, k, mode, dtype, ragged=True, seed=500 + k + mode)
    x["Q"] = torch.zeros_like(x["Q"])
    vb, L = vbar_rows(x, mode)
    ref = np.zeros((b, h, n, d))
    for bi in range(b):
        ref[bi, :, :int(L[bi])] = vb[bi].mean(axis=1)[:, None, :]
    check(run(x, mode, dtype), ref, dtype, f"Q = 0, mode {mode}, k {k}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dtype", [BF16, BF16_F32OUT, F32])
def test_one_projected_position_gives_vbar(mode, dtype):
    b, h, n, d, k = 2, 3, 520, 64, 1
    x = case_inputs(b, h, n, d, k, mode, dtype, ragged=True, seed=600 + mode)
    vb, L = vbar_rows(x, mode)
    ref = np.zeros((b, h, n, d))
    for bi in range(b):
        ref[bi, :, :int(L[bi])] = vb[bi][:, 0, None, :]
    check(run(x, mode, dtype), ref, dtype, f"k = 1, mode {mode}")


@pytest.mark.parametrize("ragged", [False, True])
@pytest.mark.parametrize("dtype", [BF16, BF16_F32OUT, F32])
@pytest.mark.parametrize("mode", MODES)
def test_mode_dtype_grid(mode, dtype, ragged):
    """Every sharing mode with every data type, with and without lengths: n = 1000 (seven
    full query tiles and a ragged one), k = 176 (a half of four chunks and one of two)."""
    b, h, n, d, k = 2, 3, 1000, 64, 176
    x = case_inputs(b, h, n, d, k, mode, dtype, ragged=ragged, seed=700 + 10 * mode + dtype)
    ref = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], mode)[0]
    check(run(x, mode, dtype), ref, dtype, f"mode {mode} dtype {dtype} ragged {ragged}")
