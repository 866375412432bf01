"""GPU parity of the backward (linformer_attn_bwd, through the C ABI) against the
fp64 backward oracle, on the same seeded inputs.

Tolerance: every gradient G satisfies max|G_gpu - G_ref| <= 2e-4 * max|G_ref|.  The
kernels compute in fp32 with a chain of three dependent products (scores, score
gradient, projection gradient), each a sum of at most max(n, k, d, units) terms; the
rounding of one such sum is at most depth * 2^-24 of its absolute terms (~6e-5 at
depth 1000), so three in sequence stay within 2e-4 of the largest gradient.
"""
import numpy as np
import pytest
import torch

import rank_linear_complexity_gb300.linformer as lf
from oracle import backward as bw
from rank_linear_complexity_gb300.workloads import (F32, HEADWISE, KV, LAYERWISE, PER_HEAD,
                                                    output_gradient)
from tests.parity import case_inputs, host64, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BWD_REL = 2e-4
NAMES = ("dQ", "dK", "dV", "dE", "dF")


def gpu_grads(x, dO, mode):
    g = to_device(x, DEV)
    out = lf.attention_backward(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"],
                                dO.to(DEV), mode)
    torch.cuda.synchronize()
    return [None if t is None else host64(t) for t in out]


def check_grads(got, ref, what):
    for name, a, r in zip(NAMES, got, ref):
        assert (a is None) == (r is None), f"{what} {name}: presence differs"
        if r is None:
            continue
        assert a.shape == r.shape, (what, name, a.shape, r.shape)
        assert np.isfinite(a).all(), f"{what} {name}: non-finite"
        err = float(np.abs(a - r).max()) if r.size else 0.0
        bound = BWD_REL * max(float(np.abs(r).max()) if r.size else 0.0, 1e-30)
        assert err <= bound, f"{what} {name}: max|err| {err:.3e} > {bound:.3e}"


CASES = [
    # (b, h, n, d, k, share_mode, ragged)
    (2, 4, 512, 64, 128, PER_HEAD, False),    # the fp32 evaluation workload
    (2, 3, 200, 32, 48, PER_HEAD, True),
    (2, 3, 200, 32, 48, KV, True),
    (2, 3, 200, 32, 48, HEADWISE, True),
    (2, 3, 200, 32, 48, LAYERWISE, True),
    (1, 3, 520, 64, 128, KV, False),          # several 64-row tiles and an 8-row tail
    (2, 2, 130, 128, 300, HEADWISE, False),   # k > n, d = 128
    (3, 2, 777, 64, 96, LAYERWISE, True),
    (1, 1, 1, 1, 1, PER_HEAD, False),         # the smallest problem
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}h{c[1]}n{c[2]}d{c[3]}k{c[4]}m{c[5]}"
                                             f"{'r' if c[6] else ''}" for c in CASES])
def test_backward_matches_oracle(case):
    b, h, n, d, k, mode, ragged = case
    x = case_inputs(b, h, n, d, k, mode, F32, ragged=ragged, seed=17 + n)
    dO = output_gradient(b, h, n, d, seed=5 + n)
    ref = bw.linformer_bwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], dO, mode)
    check_grads(gpu_grads(x, dO, mode), ref, str(case))


@pytest.mark.parametrize("mode", [PER_HEAD, LAYERWISE])
def test_empty_and_full_sequences(mode):
    """lengths 0 (no valid token: every gradient of that batch is zero) and n."""
    b, h, n, d, k = 3, 2, 96, 64, 32
    x = case_inputs(b, h, n, d, k, mode, F32, lengths=[0, n, 37], seed=2)
    dO = output_gradient(b, h, n, d, seed=3)
    ref = bw.linformer_bwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], dO, mode)
    got = gpu_grads(x, dO, mode)
    check_grads(got, ref, f"mode {mode}")
    for t in got[:3]:
        assert not t[0].any()


@pytest.mark.parametrize("mode", [KV, HEADWISE])
def test_padded_rows_may_hold_anything(mode):
    """NaN in the rows t >= L of Q, K, V and dO changes no gradient."""
    b, h, n, d, k = 2, 2, 160, 64, 64
    x = case_inputs(b, h, n, d, k, mode, F32, lengths=[100, 41], seed=9)
    dO = output_gradient(b, h, n, d, seed=10)
    ref = bw.linformer_bwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], dO, mode)
    poisoned = dict(x)
    dOp = dO.clone()
    for name in ("Q", "K", "V"):
        poisoned[name] = x[name].clone()
    for bi, L in enumerate([100, 41]):
        for t in (poisoned["Q"], poisoned["K"], poisoned["V"], dOp):
            t[bi, :, L:, :] = float("nan")
    check_grads(gpu_grads(poisoned, dOp, mode), ref, f"poisoned mode {mode}")


def test_backward_launches_through_the_library():
    """The gradients come from the library's kernels (the per-kernel counter moves)."""
    b, h, n, d, k = 1, 2, 64, 64, 32
    x = case_inputs(b, h, n, d, k, PER_HEAD, F32, seed=4)
    dO = output_gradient(b, h, n, d, seed=4)
    lf.linformer_profile_enable(True)
    try:
        gpu_grads(x, dO, PER_HEAD)
        stats = lf.linformer_profile_collect()
    finally:
        lf.linformer_profile_enable(False)
    assert stats.get("backward_kernels", (0, 0))[1] >= 10


def test_full_size_layerwise():
    """b=16, h=12, n=4096, d=64, k=256, one shared projection (the
    backward's benchmark workload, no padding): every gradient against the oracle."""
    b, h, n, d, k = 16, 12, 4096, 64, 256
    x = case_inputs(b, h, n, d, k, LAYERWISE, F32, seed=77)
    dO = output_gradient(b, h, n, d, seed=78)
    ref = bw.linformer_bwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], dO, LAYERWISE)
    check_grads(gpu_grads(x, dO, LAYERWISE), ref, "full size")
