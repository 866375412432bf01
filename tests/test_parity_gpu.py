"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Small cases are compared element by element over the whole output; the five
evaluation workloads run at full size in the same call the benchmark times and
are compared element by element with the whole-problem oracle as well (it runs
on all host cores in seconds), plus exact zeros on the padded rows.
"""
import numpy as np
import pytest
import torch

import rank_linear_complexity_gb300.linformer as lf
from oracle import oracle as orc
from rank_linear_complexity_gb300.workloads import (BF16, BF16_F32OUT, F32, HEADWISE, KV,
                                                    LAYERWISE, PER_HEAD, WORKLOADS,
                                                    workload_inputs)
from tests.parity import case_inputs, check, host64, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def run(x, share_mode, dtype):
    g = to_device(x, DEV)
    O = lf.attention(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], share_mode,
                     out_fp32=(dtype == BF16_F32OUT))
    torch.cuda.synchronize()
    assert lf.linformer_debug_read_device_status() == 0
    return O


def oracle_full(x, share_mode):
    O, _ = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], share_mode)
    return O


def with_dtype(x, dtype):
    return x


# --- small and edge shapes, whole output compared ------------------------------------

SMALL = [
    # (b, h, n, d, k, share_mode, dtype, ragged)
    (2, 4, 512, 64, 128, PER_HEAD, F32, False),       # the fp32 evaluation workload
    (2, 3, 320, 64, 128, LAYERWISE, BF16, False),     # 2.5 query tiles
    (2, 3, 320, 64, 256, PER_HEAD, BF16, True),
    (1, 4, 1000, 64, 64, KV, BF16, False),
    (3, 2, 777, 64, 96, HEADWISE, BF16_F32OUT, True),
    (2, 2, 384, 64, 200, HEADWISE, BF16, False),
    (1, 2, 300, 32, 40, PER_HEAD, BF16, False),       # d != 64: SIMT kernels
    (1, 2, 130, 128, 300, KV, F32, False),            # k > 256 on SIMT
    (2, 2, 250, 64, 64, LAYERWISE, BF16, True),       # n not a multiple of 8
]


@pytest.mark.parametrize("case", SMALL, ids=[f"b{c[0]}h{c[1]}n{c[2]}d{c[3]}k{c[4]}m{c[5]}t{c[6]}"
                                             f"{'r' if c[7] else ''}" for c in SMALL])
def test_small_cases_match_oracle(case):
    b, h, n, d, k, mode, dtype, ragged = case
    x = case_inputs(b, h, n, d, k, mode, dtype, ragged=ragged, seed=hash(case) % 1000)
    O = run(x, mode, dtype)
    check(host64(O), oracle_full(x, mode), dtype, str(case))


EDGE_N = [1, 2, 3, 5, 8, 127, 129, 136]
EDGE_K = [1, 2, 16, 64, 255, 256]


@pytest.mark.parametrize("n", EDGE_N)
@pytest.mark.parametrize("k", EDGE_K)
def test_edge_shapes(n, k):
    idx = EDGE_N.index(n) * len(EDGE_K) + EDGE_K.index(k)
    mode = idx % 4
    dtype = (BF16, BF16_F32OUT, BF16, F32)[idx % 4]
    x = case_inputs(2, 2, n, 64, k, mode, dtype, seed=idx)
    O = run(x, mode, dtype)
    check(host64(O), oracle_full(x, mode), dtype, f"n={n} k={k} mode={mode}")


@pytest.mark.parametrize("n", [8, 136, 256])
def test_k_equals_n(n):
    x = case_inputs(1, 2, n, 64, n if n <= 256 else 256, PER_HEAD, BF16, seed=n)
    O = run(x, PER_HEAD, BF16)
    check(host64(O), oracle_full(x, PER_HEAD), BF16, f"k=n={n}")


@pytest.mark.parametrize("mode", [PER_HEAD, KV, HEADWISE, LAYERWISE])
@pytest.mark.parametrize("dtype", [BF16, F32])
def test_lengths_edges(mode, dtype):
    n = 200
    x = case_inputs(4, 2, n, 64, 64, mode, dtype, seed=5 + mode, lengths=[0, 1, n - 1, n])
    O = run(x, mode, dtype)
    ref = oracle_full(x, mode)
    check(host64(O), ref, dtype, f"lengths mode={mode}")
    assert (host64(O)[0] == 0).all() and (host64(O)[1, :, 1:] == 0).all()


# --- invariants on the GPU -----------------------------------------------------------

def test_padded_rows_cannot_leak():
    n = 640
    x = case_inputs(3, 2, n, 64, 128, PER_HEAD, BF16, seed=9, lengths=[640, 333, 129])
    O1 = run(x, PER_HEAD, BF16)
    y = {kk: (v.clone() if v is not None else None) for kk, v in x.items()}
    for bi, L in enumerate([640, 333, 129]):
        y["K"][bi, :, L:] = float("nan")
        y["V"][bi, :, L:] = float("inf")
        y["Q"][bi, :, L:] = float("nan")
    O2 = run(y, PER_HEAD, BF16)
    assert torch.equal(O1, O2)


def test_deterministic_bitwise():
    x = case_inputs(4, 3, 1024, 64, 256, LAYERWISE, BF16, seed=11)
    O1 = run(x, LAYERWISE, BF16)
    O2 = run(x, LAYERWISE, BF16)
    assert torch.equal(O1, O2)


def test_sharing_mode_consistency():
    x = case_inputs(2, 3, 512, 64, 128, HEADWISE, BF16, seed=12)
    O_hw = run(x, HEADWISE, BF16)
    y = dict(x)
    y["E"] = x["E"].unsqueeze(0).repeat(3, 1, 1).contiguous()
    y["F"] = x["F"].unsqueeze(0).repeat(3, 1, 1).contiguous()
    O_ph = run(y, PER_HEAD, BF16)
    check(host64(O_ph), host64(O_hw), BF16, "per-head with equal E_h vs headwise")
    z = dict(x)
    z["F"] = None
    O_lw = run(z, LAYERWISE, BF16)
    w = dict(x)
    w["F"] = x["E"]
    O_hw2 = run(w, HEADWISE, BF16)
    check(host64(O_lw), host64(O_hw2), BF16, "layerwise vs headwise with F = E")


@pytest.mark.parametrize("mode", [PER_HEAD, KV, HEADWISE, LAYERWISE])
def test_projection_entry_point(mode):
    x = case_inputs(2, 3, 1000, 64, 128, mode, BF16, ragged=True, seed=20 + mode)
    g = to_device(x, DEV)
    Kb, Vb = lf.projection(g["K"], g["V"], g["E"], g["F"], g["lengths"], mode)
    torch.cuda.synchronize()
    _, _, rK, rV = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], mode,
                                     return_proj=True)
    for got, ref in ((host64(Kb), rK), (host64(Vb), rV)):
        assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max() + 1e-6


@pytest.mark.parametrize("b,n,d,dtype,ragged", [(2, 512, 64, BF16, False),   # two chunks
                                                 (5, 512, 64, BF16, True),    # uneven chunks
                                                 (3, 130, 40, F32, False)])   # one chunk (rows
def test_host_entry_point_matches_device(b, n, d, dtype, ragged):          # not 256-B multiples)
    x = case_inputs(b, 2, n, d, 128, KV, dtype, ragged=ragged, seed=30 + b)
    O_dev = run(x, KV, dtype)
    pin = {kk: (v.pin_memory() if v is not None else None) for kk, v in x.items()}
    O_host = torch.empty(O_dev.shape, dtype=O_dev.dtype).pin_memory()
    st = lf.linformer_attn_fwd_host(pin["Q"], pin["K"], pin["V"], pin["E"], None,
                                    pin["lengths"], O_host, b, 2, n, d, 128, KV, dtype)
    assert st == 0, lf.status_string(st)
    assert torch.equal(O_host, O_dev.cpu())


# --- projection CTAs that take two units ----------------------------------------------
# More units than one wave of CTA slots, unsplit, E = F, no lengths: some CTAs project
# two members of a sharing group with one E tile.  k > 128 gives one CTA per SM (152
# slots), k <= 128 two (304 slots).

PAIRED = [
    # (b, h, n, k, share_mode)
    (16, 12, 512, 256, LAYERWISE),   # 192 units: 40 two-unit CTAs
    (16, 12, 512, 256, KV),          # per head: 4 two-member CTAs in each of 12 groups
    (13, 12, 384, 200, KV),          # odd members: 1 pair and 11 single CTAs per group
    (20, 16, 256, 64, LAYERWISE),    # 320 units, two CTAs per SM: 16 two-unit CTAs
    (20, 16, 256, 64, KV),
    (16, 12, 520, 256, LAYERWISE),   # last 64-row stage partly past n in both units of a pair
]


@pytest.mark.parametrize("case", PAIRED, ids=[f"b{c[0]}h{c[1]}n{c[2]}k{c[3]}m{c[4]}"
                                              for c in PAIRED])
def test_paired_projection_match_oracle(case):
    b, h, n, k, mode = case
    x = case_inputs(b, h, n, 64, k, mode, BF16, seed=50 + b + k)
    O = run(x, mode, BF16)
    check(host64(O), oracle_full(x, mode), BF16, str(case))


def test_paired_projection_outputs():
    b, h, n, k, mode = PAIRED[0]
    x = case_inputs(b, h, n, 64, k, mode, BF16, seed=60)
    g = to_device(x, DEV)
    Kb, Vb = lf.projection(g["K"], g["V"], g["E"], g["F"], g["lengths"], mode)
    torch.cuda.synchronize()
    _, _, rK, rV = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], mode,
                                     return_proj=True)
    for got, ref in ((host64(Kb), rK), (host64(Vb), rV)):
        assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max() + 1e-6


# --- the number of P.Vbar products ------------------------------------------------------

PV_CASE = (2, 3, 2048, 64, 128, PER_HEAD)  # Vbar ~ N(0, 16 vscale^2): max|Vbar| ~ 16 vscale


@pytest.mark.parametrize("terms,vscale", [(1, 1.0), (2, 1.0), (3, 1.0), (0, 2.0), (2, 2.0),
                                          (3, 2.0)])
def test_pv_products_match_oracle(terms, vscale):
    """Each forced product count where all of them meet the bar (vscale 1), and, with V
    doubled, the per-unit choice (which then takes two products) and its neighbours."""
    b, h, n, d, k, mode = PV_CASE
    x = case_inputs(b, h, n, d, k, mode, BF16, seed=40)
    x["V"] = (x["V"].float() * vscale).to(x["V"].dtype)  # a power of two: exact in bf16
    ref, _, _, rV = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"],
                                      mode, return_proj=True)
    vmax = np.abs(rV).reshape(b * h, -1).max(axis=1)
    if terms == 0:  # every unit inside the two-product band
        assert (vmax >= 24).all() and (vmax < 40).all(), vmax
    prev = lf.linformer_set_pv_terms(terms)
    try:
        O = run(x, mode, BF16)
    finally:
        lf.linformer_set_pv_terms(prev)
    check(host64(O), ref, BF16, f"terms={terms} vscale={vscale}")


@pytest.mark.parametrize("k", [1, 16, 40, 64, 100, 128, 200, 256])
def test_three_products_at_every_key_layout(k):
    """Three P.Vbar products forced where a key half has one, two, three or four chunks
    (up to k_pad = 128 the tile keeps P_lo after its P in its own buffer, both chunks
    read first; above, P_lo goes to the other buffer), with ragged lengths and a ragged
    last query tile."""
    b, h, n, d, mode = 2, 3, 1000, 64, PER_HEAD
    x = case_inputs(b, h, n, d, k, mode, BF16, ragged=True, seed=44)
    ref = oracle_full(x, mode)
    prev = lf.linformer_set_pv_terms(3)
    try:
        O = run(x, mode, BF16)
    finally:
        lf.linformer_set_pv_terms(prev)
    check(host64(O), ref, BF16, f"three products, k={k}")


# --- scores that grow along the keys ---------------------------------------------------

@pytest.mark.parametrize("mode", [PER_HEAD, HEADWISE])
@pytest.mark.parametrize("k", [128, 200, 256])
def test_scores_growing_along_the_keys(mode, k):
    """Rows of E scaled by 1, 4, 16, 64 for the first, second, ... 32-key chunk of each
    128-key half: every chunk's maximum score lies far above the previous chunks' (more
    than 2^15 in exp2 terms), so each half's maximum sits in its last chunk and nearly
    all of a row's weight on a few keys.  F is left alone (one P.Vbar product)."""
    b, h, n, d = 2, 3, 512, 64
    x = case_inputs(b, h, n, d, k, mode, BF16, seed=44)
    j = torch.arange(k)
    factor = torch.pow(4.0, torch.clamp((j % 128) // 32, max=3).float())  # exact in bf16
    x["E"] = (x["E"].float() * factor.view(*([1] * (x["E"].dim() - 2)), k, 1)).to(x["E"].dtype)
    ref = oracle_full(x, mode)
    O = run(x, mode, BF16)
    check(host64(O), ref, BF16, f"growing scores k={k} mode={mode}")


# --- the five evaluation workloads at full size, whole output ------------------------

def _report(entry):
    """Appends one JSON line of parity margins to $LINFORMER_PARITY_REPORT, if set."""
    import json
    import os
    path = os.environ.get("LINFORMER_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(entry) + "\n")
    print(entry)


@pytest.mark.parametrize("wi", range(len(WORKLOADS)), ids=[w.name for w in WORKLOADS])
def test_workload_full_output(wi):
    """Every element of the five evaluation workloads, in the launch configuration the
    benchmark times, against the whole-problem fp64 oracle on all host cores."""
    w = WORKLOADS[wi]
    x = workload_inputs(w)
    O = run(x, w.share_mode, w.dtype)
    lengths = x["lengths"].numpy() if x["lengths"] is not None else np.full(w.b, w.n)
    for bi in range(w.b):
        assert (O[bi, :, int(lengths[bi]):] == 0).all()
    got = host64(O)
    del O
    ref, used = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"],
                                  w.share_mode)
    e = check(got, ref, w.dtype, w.name)
    _report({"workload": w.name, "elements": int(ref.size), "oracle_threads": int(used),
             **{kk: (round(v, 6) if isinstance(v, float) else v) for kk, v in e.items()}})
