"""Pins for the oracle's per-unit helpers, unit_projections and unit_rows (CPU only).

The GPU tests use these helpers wherever they need the reference output of a single
(batch, head) unit (rows of large fp32 problems, the backward's inputs).  Here they
are tied to the whole-problem routine oracle_linformer_fwd, which is pinned by the
hand-derived golden cases and the invariants of test_oracle.py: for every sharing
mode ("Linformer: Self-Attention with Linear Complexity - 中文验证版", section
方法适配: per head, key-value, headwise and layerwise sharing) and ragged valid
lengths ("Linformer 요약 설명", section Model, padding paragraph), every unit's
sampled rows, on both sides of its valid length, and its projections must agree.

Each head gets its own E and F, drawn independently, so that a helper that picked
the wrong head, or F where E belongs (or the reverse), gives a different answer;
the last test shows that two such plausible mistakes are indeed caught.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc

B, H, N, D, K = 3, 4, 96, 8, 16
LENGTHS = [96, 41, 0]  # full, ragged (rows on both sides of L), empty


def _inputs(mode, seed, torch_bf16=False):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((B, H, N, D))
    Kx = rng.standard_normal((B, H, N, D))
    V = rng.standard_normal((B, H, N, D))
    shp = (H, K, N) if mode in (orc.PER_HEAD, orc.KV) else (K, N)
    E = rng.standard_normal(shp) / np.sqrt(K)
    F = rng.standard_normal(shp) / np.sqrt(K)
    if mode in (orc.KV, orc.LAYERWISE):
        F = None
    lengths = np.array(LENGTHS, np.int32)
    if torch_bf16:  # the form the GPU tests pass in: torch bf16 tensors
        cv = lambda a: None if a is None else torch.from_numpy(a).to(torch.bfloat16)
        return {"Q": cv(Q), "K": cv(Kx), "V": cv(V), "E": cv(E), "F": cv(F),
                "lengths": torch.from_numpy(lengths)}
    return {"Q": Q, "K": Kx, "V": V, "E": E, "F": F, "lengths": lengths}


def _rows(L):
    picks = {0, N - 1, 1, N // 2, max(0, L - 1), min(N - 1, L), min(N - 1, L + 1)}
    return np.array(sorted(picks), np.int64)


def _whole(x, mode):
    return orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], mode,
                             return_proj=True)


@pytest.mark.parametrize("torch_bf16", [False, True], ids=["f64", "torch_bf16"])
@pytest.mark.parametrize("mode", [orc.PER_HEAD, orc.KV, orc.HEADWISE, orc.LAYERWISE])
def test_unit_rows_match_whole_problem(mode, torch_bf16):
    x = _inputs(mode, 10 + mode, torch_bf16)
    O, _, Kb, Vb = _whole(x, mode)
    for bi in range(B):
        L = LENGTHS[bi]
        for hi in range(H):
            rows = _rows(L)
            got, kb, vb = orc.unit_rows(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"],
                                        mode, bi, hi, rows)
            np.testing.assert_allclose(got, O[bi, hi][rows], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(kb, Kb[bi, hi], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(vb, Vb[bi, hi], rtol=1e-12, atol=1e-13)
            assert (got[rows >= L] == 0).all()  # padded query rows
            if L > 0:
                assert np.abs(got[rows < L]).max() > 0


@pytest.mark.parametrize("mode", [orc.PER_HEAD, orc.KV, orc.HEADWISE, orc.LAYERWISE])
def test_unit_projections_reproduce_the_whole_problem_projections(mode):
    """The pair a unit uses, applied by a library matmul over the valid rows, gives the
    Kbar and Vbar the whole-problem oracle computes for that unit."""
    x = _inputs(mode, 20 + mode)
    _, _, Kb, Vb = _whole(x, mode)
    for bi in range(B):
        L = LENGTHS[bi]
        for hi in range(H):
            Eh, Fh = orc.unit_projections(x["E"], x["F"], mode, hi)
            assert Eh.shape == (K, N) and Fh.shape == (K, N)
            np.testing.assert_allclose(Eh[:, :L] @ x["K"][bi, hi, :L], Kb[bi, hi],
                                       rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(Fh[:, :L] @ x["V"][bi, hi, :L], Vb[bi, hi],
                                       rtol=1e-10, atol=1e-12)


_UNIT_PROJECTIONS = orc.unit_projections  # the real helper, before any planted mistake


def _headwise_f_is_e(E, F, mode, head):
    Eh, Fh = _UNIT_PROJECTIONS(E, F, mode, head)
    return (Eh, Eh) if mode == orc.HEADWISE else (Eh, Fh)


def _head_dropped(E, F, mode, head):
    return _UNIT_PROJECTIONS(E, F, mode, 0)


@pytest.mark.parametrize("mistake,modes", [(_headwise_f_is_e, [orc.HEADWISE]),
                                           (_head_dropped, [orc.PER_HEAD, orc.KV])])
def test_planted_helper_mistakes_are_caught(monkeypatch, mistake, modes):
    """A unit_projections that used E for F in headwise mode, or always head 0, must fail
    the comparison above (planted in the oracle's helper, on the CPU)."""
    for mode in modes:
        x = _inputs(mode, 30 + mode)
        O, _, _, _ = _whole(x, mode)
        monkeypatch.setattr(orc, "unit_projections", mistake)
        caught = False
        for bi in range(B):
            for hi in range(H):
                rows = _rows(LENGTHS[bi])
                got, _, _ = orc.unit_rows(x["Q"], x["K"], x["V"], x["E"], x["F"],
                                          x["lengths"], mode, bi, hi, rows)
                if not np.allclose(got, O[bi, hi][rows], rtol=1e-12, atol=1e-13):
                    caught = True
        monkeypatch.undo()
        assert caught, f"{mistake.__name__} not caught in mode {mode}"
