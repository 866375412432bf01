"""GPU parity of the dense softmax attention (linformer_dense_attn_fwd, through the C
ABI) against the fp64 dense oracle, at the fp32 bar of the forward:
max|O_gpu - O_ref| <= 1e-4 * max|O_ref|."""
import numpy as np
import pytest
import torch

import rank_linear_complexity_gb300.linformer as lf
from oracle import dense
from rank_linear_complexity_gb300.workloads import F32, PER_HEAD, make_inputs
from tests.parity import check, host64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def inputs(b, h, n, d, lengths=None, seed=0):
    x = make_inputs(b, h, n, d, 1, PER_HEAD, F32, seed=seed)
    L = None if lengths is None else torch.tensor(lengths, dtype=torch.int32)
    return x["Q"], x["K"], x["V"], L


def run(Q, K, V, L):
    O = lf.dense_attention(Q.to(DEV), K.to(DEV), V.to(DEV), None if L is None else L.to(DEV))
    torch.cuda.synchronize()
    return host64(O)


CASES = [
    # (b, h, n, d, lengths)
    (2, 3, 200, 32, [150, 37]),
    (1, 2, 777, 64, None),          # ragged tiles, n not a multiple of 4 (scalar loads)
    (2, 2, 512, 64, [512, 0]),      # a full and an empty sequence
    (1, 1, 1000, 128, None),
    (1, 1, 1, 1, None),             # the smallest problem
    (2, 12, 512, 64, None),         # n = 512, RoBERTa-base heads
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}h{c[1]}n{c[2]}d{c[3]}{'r' if c[4] else ''}"
                                             for c in CASES])
def test_dense_matches_oracle(case):
    b, h, n, d, lengths = case
    Q, K, V, L = inputs(b, h, n, d, lengths, seed=n)
    check(run(Q, K, V, L), dense.dense_fwd(Q, K, V, L), F32, str(case))


def test_padded_rows_may_hold_anything():
    Q, K, V, L = inputs(2, 2, 300, 64, [211, 64], seed=5)
    ref = dense.dense_fwd(Q, K, V, L)
    for bi, n_valid in enumerate([211, 64]):
        for t in (Q, K, V):
            t[bi, :, n_valid:] = float("nan")
    check(run(Q, K, V, L), ref, F32, "poisoned")


def test_workspace_is_the_score_matrices():
    """The pool's high-water mark during one call is the n x n scores of every unit."""
    b, h, n, d = 1, 4, 1024, 64
    Q, K, V, L = inputs(b, h, n, d, seed=6)
    torch.cuda.synchronize()
    lf.linformer_pool_peak_bytes(reset=True)
    run(Q, K, V, L)
    assert lf.linformer_pool_peak_bytes() >= b * h * n * n * 4


@pytest.mark.parametrize("n,units", [(4096, 12), (65536, 1)])
def test_inference_table_sizes_sampled_rows(n, units):
    """The sizes the inference comparison times (n = 4096 with 12 heads, n = 65536 with
    one): sampled query rows against the oracle (each row stands alone), plus finite
    values everywhere."""
    b, h, d = 1, units, 64
    Q, K, V, L = inputs(b, h, n, d, seed=n + 1)
    O = lf.dense_attention(Q.to(DEV), K.to(DEV), V.to(DEV))
    torch.cuda.synchronize()
    assert torch.isfinite(O).all()
    rows = np.unique(np.r_[0, 1, n // 2, n - 1, np.random.default_rng(n).integers(0, n, 20)])
    heads = [0, h - 1]
    got = O[:, heads][:, :, torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    ref = dense.dense_fwd(Q[:, heads], K[:, heads], V[:, heads], rows=rows)
    check(got, ref, F32, f"n={n}")
