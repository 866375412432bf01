"""Robustness checks that need no GPU fault: a forced workspace-allocation failure,
guard rows around the output and after every workspace, and the invariance of the
output under a permutation of the projected positions.

* Allocation failure: with LINFORMER_FAIL_ALLOC=1 every workspace allocation of the
  library fails; each entry point must return LINFORMER_ERR_ALLOC (-7) before it
  launches anything, and leave its output untouched.
* Guard rows: O is a view into a larger buffer with guard rows before and after it,
  all filled with a pattern; after the call the guards must be unchanged.  With
  LINFORMER_WORKSPACE_GUARD=1 the library also puts 4 KB of a pattern after each
  workspace and checks it when the workspace is freed (a changed byte sets the device
  status word).  Shapes cover the tile edges of both kernels (n around multiples of
  128 and 64, k around multiples of 16 and 32), every sharing mode and output type.
* Permutation: the method sums over the k projected positions inside the softmax
  and in P.Vbar, so permuting the rows of E and F together ("Linformer 요약 설명",
  section Model: row j of E merges the n positions into compressed position j)
  cannot change O beyond rounding.
"""
import os

import numpy as np
import pytest
import torch

import rank_linear_complexity_gb300.linformer as lf
from oracle import oracle as orc
from rank_linear_complexity_gb300.workloads import (BF16, BF16_F32OUT, F32, HEADWISE, KV,
                                                    LAYERWISE, PER_HEAD, output_gradient)
from tests.parity import case_inputs, check, host64, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ERR_ALLOC = -7


@pytest.fixture
def env(monkeypatch):
    return monkeypatch


def _out_dtype(dtype):
    return torch.bfloat16 if dtype == BF16 else torch.float32


# --- forced allocation failure ---------------------------------------------------------

ALLOC_CASES = [
    # (b, h, n, d, k, mode, dtype): tensor-core path, fp32 SIMT path, bf16 SIMT path (whose
    # projection alone needs no workspace: linformer_project_fwd is not checked there)
    (2, 3, 256, 64, 128, LAYERWISE, BF16),
    (2, 2, 200, 64, 48, PER_HEAD, F32),
    (1, 2, 300, 32, 40, KV, BF16),
]


@pytest.mark.parametrize("case", ALLOC_CASES, ids=[f"n{c[2]}d{c[3]}k{c[4]}t{c[6]}"
                                                   for c in ALLOC_CASES])
def test_forced_allocation_failure_returns_before_launch(env, case):
    b, h, n, d, k, mode, dtype = case
    g = to_device(case_inputs(b, h, n, d, k, mode, dtype, seed=3), DEV)
    O = torch.full((b, h, n, d), float("nan"), dtype=_out_dtype(dtype), device=DEV)
    torch.cuda.synchronize()
    env.setenv("LINFORMER_FAIL_ALLOC", "1")
    launches = lf.linformer_launch_count()
    st = lf.linformer_attn_fwd(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], O,
                               b, h, n, d, k, mode, dtype)
    assert st == ERR_ALLOC, lf.status_string(st)
    if dtype == F32 or lf.linformer_select_path(b, h, n, d, k, mode, dtype) == lf.PATH_TENSOR:
        Kb = torch.empty((b, h, k, d), dtype=torch.float32, device=DEV)
        st = lf.linformer_project_fwd(g["K"], g["V"], g["E"], g["F"], g["lengths"], Kb,
                                      torch.empty_like(Kb), b, h, n, d, k, mode, dtype)
        assert st == ERR_ALLOC
    pin = {kk: (v.cpu().pin_memory() if v is not None else None) for kk, v in g.items()}
    Oh = torch.empty(O.shape, dtype=O.dtype).pin_memory()
    st = lf.linformer_attn_fwd_host(pin["Q"], pin["K"], pin["V"], pin["E"], pin["F"],
                                    pin["lengths"], Oh, b, h, n, d, k, mode, dtype)
    assert st == ERR_ALLOC
    assert lf.linformer_launch_count() == launches  # nothing was launched
    torch.cuda.synchronize()
    assert torch.isnan(O.float()).all()  # O untouched
    env.delenv("LINFORMER_FAIL_ALLOC")
    st = lf.linformer_attn_fwd(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], O,
                               b, h, n, d, k, mode, dtype)
    assert st == 0
    torch.cuda.synchronize()
    assert lf.linformer_debug_read_device_status() == 0


def test_forced_allocation_failure_backward_and_dense(env):
    b, h, n, d, k = 1, 2, 128, 64, 32
    g = to_device(case_inputs(b, h, n, d, k, PER_HEAD, F32, seed=4), DEV)
    dO = output_gradient(b, h, n, d, seed=5).to(DEV)
    out = [torch.empty_like(g[c]) for c in ("Q", "K", "V", "E", "F")]
    env.setenv("LINFORMER_FAIL_ALLOC", "1")
    launches = lf.linformer_launch_count()
    st = lf.linformer_attn_bwd(g["Q"], g["K"], g["V"], g["E"], g["F"], None, dO, *out,
                               b, h, n, d, k, PER_HEAD, F32)
    assert st == ERR_ALLOC
    st = lf.linformer_dense_attn_fwd(g["Q"], g["K"], g["V"], None, out[0], b, h, n, d, F32)
    assert st == ERR_ALLOC
    assert lf.linformer_launch_count() == launches


# --- guard rows --------------------------------------------------------------------------

GUARD_ROWS = 8
GUARD_CASES = [
    # (b, h, n, k, mode, dtype, lengths)
    (2, 3, 8, 16, LAYERWISE, BF16, None),
    (2, 2, 127, 255, PER_HEAD, BF16, None),
    (1, 3, 128, 256, KV, BF16_F32OUT, None),
    (3, 2, 129, 200, HEADWISE, BF16, [129, 1, 64]),
    (2, 2, 640, 96, PER_HEAD, BF16, [640, 333]),
    (2, 2, 136, 33, KV, F32, [136, 70]),
    (2, 2, 250, 64, LAYERWISE, BF16, [250, 129]),        # n % 8 != 0: SIMT path
    (16, 12, 520, 256, LAYERWISE, BF16, None),           # two-unit projection CTAs
    (1, 4, 4096, 128, HEADWISE, BF16, None),             # split sequence: partial sums
]


@pytest.mark.parametrize("case", GUARD_CASES, ids=[f"b{c[0]}n{c[2]}k{c[3]}m{c[4]}t{c[5]}"
                                                   for c in GUARD_CASES])
def test_guard_rows_around_output_and_workspace(env, case):
    b, h, n, k, mode, dtype, lengths = case
    d = 64
    x = case_inputs(b, h, n, d, k, mode, dtype, seed=7 + n, lengths=lengths)
    g = to_device(x, DEV)
    odt = _out_dtype(dtype)
    rows = b * h * n
    buf = torch.empty((rows + 2 * GUARD_ROWS, d), dtype=odt, device=DEV)
    buf.view(torch.uint8 if odt == torch.bfloat16 else torch.int32).fill_(
        0x5A if odt == torch.bfloat16 else 0x5A5A5A5A)
    before = buf.clone()
    O = buf[GUARD_ROWS:GUARD_ROWS + rows].view(b, h, n, d)
    assert O.data_ptr() % 16 == 0
    env.setenv("LINFORMER_WORKSPACE_GUARD", "1")
    st = lf.linformer_attn_fwd(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], O,
                               b, h, n, d, k, mode, dtype)
    assert st == 0, lf.status_string(st)
    torch.cuda.synchronize()
    assert lf.linformer_debug_read_device_status() == 0  # workspace guards intact
    assert torch.equal(buf[:GUARD_ROWS], before[:GUARD_ROWS])
    assert torch.equal(buf[GUARD_ROWS + rows:], before[GUARD_ROWS + rows:])
    check(host64(O), orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"],
                                       mode)[0], dtype, str(case))


def test_guard_rows_around_projection_outputs(env):
    b, h, n, d, k = 2, 3, 1000, 64, 200
    x = case_inputs(b, h, n, d, k, PER_HEAD, BF16, ragged=True, seed=8)
    g = to_device(x, DEV)
    rows = b * h * k
    bufs = [torch.full((rows + 2 * GUARD_ROWS, d), -7.25, device=DEV) for _ in range(2)]
    Kb, Vb = (bb[GUARD_ROWS:GUARD_ROWS + rows].view(b, h, k, d) for bb in bufs)
    env.setenv("LINFORMER_WORKSPACE_GUARD", "1")
    st = lf.linformer_project_fwd(g["K"], g["V"], g["E"], g["F"], g["lengths"], Kb, Vb,
                                  b, h, n, d, k, PER_HEAD, BF16)
    assert st == 0
    torch.cuda.synchronize()
    assert lf.linformer_debug_read_device_status() == 0
    for bb in bufs:
        assert (bb[:GUARD_ROWS] == -7.25).all() and (bb[GUARD_ROWS + rows:] == -7.25).all()


# --- permutation of the projected positions ------------------------------------------------

@pytest.mark.parametrize("mode,dtype,k", [(PER_HEAD, BF16, 256), (KV, BF16, 200),
                                          (HEADWISE, BF16_F32OUT, 128), (LAYERWISE, BF16, 64),
                                          (PER_HEAD, F32, 96)])
def test_permuting_projected_positions_on_gpu(mode, dtype, k):
    b, h, n = 2, 3, 776 if dtype != F32 else 300
    x = case_inputs(b, h, n, 64, k, mode, dtype, ragged=True, seed=90 + k)
    perm = torch.from_numpy(np.random.default_rng(k).permutation(k))
    y = dict(x)
    y["E"] = x["E"].index_select(-2, perm).contiguous()
    if x["F"] is not None:
        y["F"] = x["F"].index_select(-2, perm).contiguous()
    outs = []
    for inp in (x, y):
        gi = to_device(inp, DEV)
        outs.append(lf.attention(gi["Q"], gi["K"], gi["V"], gi["E"], gi["F"], gi["lengths"],
                                 mode, out_fp32=(dtype == BF16_F32OUT)))
    torch.cuda.synchronize()
    ref = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], mode)[0]
    check(host64(outs[1]), ref, dtype, "permuted E/F against the unpermuted oracle")
    check(host64(outs[0]), ref, dtype, "unpermuted")


# --- forwards one after another in a stream --------------------------------------------------

def test_forwards_in_a_stream_see_inputs_written_between_them():
    """The projection is launched as a programmatic dependent of whatever kernel precedes it
    and waits for that grid before it reads or writes anything; the attention lets the
    next kernel launch early.  A forward that follows PyTorch kernels rewriting Q, K, V and
    E in place on the same stream must see the new values, and a forward launched right
    after another (its projection overlapping the previous attention's last CTAs) must
    give the same result.  Unsplit units, so no memset separates the launches."""
    b, h, n, d, k, mode = 4, 12, 2048, 64, 256, LAYERWISE
    x = case_inputs(b, h, n, d, k, mode, BF16, seed=77)
    y = case_inputs(b, h, n, d, k, mode, BF16, seed=78)
    g, gy = to_device(x, DEV), to_device(y, DEV)

    def fwd():
        return lf.attention(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], mode)

    O1 = fwd()
    for key in ("Q", "K", "V", "E"):  # elementwise kernels, not copies: 0 x + y == y exactly
        g[key].mul_(0).add_(gy[key])
    O2 = fwd()
    O3 = fwd()
    torch.cuda.synchronize()
    assert lf.linformer_debug_read_device_status() == 0
    check(host64(O1), orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"],
                                        mode)[0], BF16, "first forward")
    ref_y = orc.linformer_fwd(y["Q"], y["K"], y["V"], y["E"], y["F"], y["lengths"], mode)[0]
    check(host64(O2), ref_y, BF16, "forward after the inputs were rewritten")
    assert torch.equal(O2, O3), "back-to-back forwards differ"


@pytest.mark.parametrize("mode,k,forced", [(KV, 128, 0), (HEADWISE, 128, 3), (LAYERWISE, 256, 0)])
def test_many_forwards_back_to_back(mode, k, forced):
    """Hundreds of forwards in a row, each attention CTA working through many tiles: every
    bounded device wait must be met (the device status stays clear) and every call must
    give the same output.  With k_pad <= 128 a buffer's next score products wait only for
    its previous P.V, so a softmax may finish a tile while the epilogue is two tiles
    behind in the same buffer; a per-buffer barrier would then have run a phase past the
    epilogue's wait (the row sums' own four-slot barriers prevent that)."""
    b, h, n, d = 8, 12, 1024, 64
    x = case_inputs(b, h, n, d, k, mode, BF16, seed=91)
    g = to_device(x, DEV)

    def fwd():
        return lf.attention(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], mode)

    prev = lf.linformer_set_pv_terms(forced)  # 0: each unit's own choice
    try:
        O1 = fwd()
        for _ in range(300):
            O2 = fwd()
        torch.cuda.synchronize()
    finally:
        lf.linformer_set_pv_terms(prev)
    assert lf.linformer_debug_read_device_status() == 0
    assert torch.equal(O1, O2), "repeated forwards differ"
    check(host64(O1), orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"],
                                        mode)[0], BF16, "first of the repeated forwards")


def test_two_streams_and_the_projection_entry_point_interleaved():
    """Forwards on two streams at once (each stream's projection waits only for its own
    stream's previous kernel), and the projection-only entry point between forwards in
    one stream: every result against the oracle."""
    b, h, n, d, k, mode = 2, 12, 2048, 64, 256, PER_HEAD
    xs = [case_inputs(b, h, n, d, k, mode, BF16, seed=80 + i) for i in range(2)]
    gs = [to_device(x, DEV) for x in xs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = [[], []]
    for _ in range(3):
        for i in (0, 1):
            g = gs[i]
            with torch.cuda.stream(streams[i]):
                outs[i].append(lf.attention(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"],
                                            mode, stream=streams[i].cuda_stream))
    with torch.cuda.stream(streams[0]):
        g = gs[0]
        kb, vb = lf.projection(g["K"], g["V"], g["E"], g["F"], g["lengths"], mode,
                               stream=streams[0].cuda_stream)
        outs[0].append(lf.attention(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], mode,
                                    stream=streams[0].cuda_stream))
    torch.cuda.synchronize()
    assert lf.linformer_debug_read_device_status() == 0
    for i in (0, 1):
        x = xs[i]
        ref, _, rK, rV = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"],
                                           mode, return_proj=True)
        for j, O in enumerate(outs[i]):
            check(host64(O), ref, BF16, f"stream {i}, call {j}")
            assert torch.equal(O, outs[i][0]), f"stream {i}: call {j} differs from call 0"
        if i == 0:
            for got, want in ((kb, rK), (vb, rV)):
                w = np.asarray(want, np.float64)
                err = np.abs(host64(got) - w).max()
                assert err <= 1e-4 * max(np.abs(w).max(), 1e-30), err


@pytest.mark.parametrize("mode,k", [(LAYERWISE, 256), (PER_HEAD, 128)])
@pytest.mark.parametrize("entry", ["linformer_attn_fwd", "linformer_attn_fwd_noalloc"])
def test_forward_captured_in_a_cuda_graph(entry, mode, k):
    """A forward captured in a CUDA graph (its stream-ordered workspace, its programmatic
    launches) replays to the eager result bitwise, and sees inputs rewritten in place
    between replays; checked against the oracle too.  Both attention instantiations
    (k_pad > 128 and <= 128)."""
    fn = getattr(lf, entry)
    b, h, n, d = 2, 3, 1024, 64
    x = case_inputs(b, h, n, d, k, mode, BF16, seed=95)
    y = case_inputs(b, h, n, d, k, mode, BF16, seed=96)
    g, gy = to_device(x, DEV), to_device(y, DEV)

    def args(O, s):
        return (g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], O, b, h, n, d, k, mode,
                BF16, s)

    O_eager = torch.empty_like(g["Q"])
    assert fn(*args(O_eager, torch.cuda.current_stream().cuda_stream)) == 0  # first use: set-up
    torch.cuda.synchronize()
    O = torch.zeros_like(g["Q"])
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        assert fn(*args(O, s.cuda_stream)) == 0
    graph.replay()
    torch.cuda.synchronize()
    assert lf.linformer_debug_read_device_status() == 0
    assert torch.equal(O, O_eager)
    check(host64(O), orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"],
                                       mode)[0], BF16, f"{entry} replay")
    for key in ("Q", "K", "V", "E", "F"):
        if g[key] is not None:
            g[key].copy_(gy[key])
    graph.replay()
    torch.cuda.synchronize()
    assert lf.linformer_debug_read_device_status() == 0
    check(host64(O), orc.linformer_fwd(y["Q"], y["K"], y["V"], y["E"], y["F"], y["lengths"],
                                       mode)[0], BF16, f"{entry} replay after new inputs")
