"""Pins for the fp64 oracle (CPU only).

Each check ties the oracle to something other than itself:
  * hand-derived worked cases (tests/golden/*.json, each with its citation);
  * the special case k = n, E = F = I, which must reduce to ordinary softmax
    attention ("Linformer 요약 설명", section Transformer and Self-Attention),
    computed here by torch's library routine scaled_dot_product_attention;
  * the projection against a library matmul (numpy);
  * closed forms: Q = 0 gives the mean of Vbar; k = 1 gives F.V;
  * invariants: softmax rows sum to one; sharing-mode equalities; padded rows
    cannot influence the result; permuting the k projected positions changes
    nothing; linearity in V.
A final test plants plausible mistakes in copies of the oracle's C source and
checks that each one is caught by at least one of these pins.
"""
import glob
import json
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLDEN = sorted(glob.glob(os.path.join(os.path.dirname(__file__), "golden", "*.json")))


def _arr(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def _run_golden(path, lib=None):
    g = json.load(open(path))
    O, _ = orc.linformer_fwd(_arr(g["Q"]), _arr(g["K"]), _arr(g["V"]), _arr(g["E"]),
                             _arr(g["F"]), g["pad_lengths"], g["share_mode"], lib=lib)
    return O, _arr(g["expected_O"])


@pytest.mark.parametrize("path", GOLDEN, ids=[os.path.basename(p) for p in GOLDEN])
def test_golden_hand_derived(path):
    O, expected = _run_golden(path)
    np.testing.assert_allclose(O, expected, rtol=0, atol=1e-12)


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


@pytest.mark.parametrize("n,d", [(1, 1), (2, 3), (5, 4), (8, 16), (33, 8)])
def test_identity_projection_is_softmax_attention(n, d):
    """k = n, E = F = I: Linformer attention is plain scaled dot-product attention."""
    rng = np.random.default_rng(100 + n * 7 + d)
    Q, K, V = _rand(rng, 1, 1, n, d), _rand(rng, 1, 1, n, d), _rand(rng, 1, 1, n, d)
    I = np.eye(n)[None]
    O, _ = orc.linformer_fwd(Q, K, V, I, I, None, orc.PER_HEAD)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V)).numpy()
    np.testing.assert_allclose(O, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n,d", [(1, 2), (7, 3), (20, 8)])
def test_full_attention_matches_library(n, d):
    rng = np.random.default_rng(7 * n + d)
    Q, K, V = _rand(rng, n, d), _rand(rng, n, d), _rand(rng, n, d)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None])[0]
    np.testing.assert_allclose(orc.full_attention(Q, K, V), ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n,d,k,L", [(9, 4, 3, 9), (9, 4, 3, 5), (16, 8, 32, 11), (5, 2, 1, 0)])
def test_projection_matches_library_matmul(n, d, k, L):
    rng = np.random.default_rng(n * 100 + k)
    E, X = _rand(rng, k, n), _rand(rng, n, d)
    got = orc.project(E, X, L)
    np.testing.assert_allclose(got, E[:, :L] @ X[:L], rtol=1e-12, atol=1e-12)


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(3)
    n, d, k = 40, 8, 12
    Q, K, V = _rand(rng, n, d, scale=3), _rand(rng, n, d), _rand(rng, n, d)
    E = _rand(rng, k, n, scale=1 / np.sqrt(k))
    Kb, Vb = orc.project(E, K), orc.project(E, V)
    _, P = orc.attend(Q, Kb, Vb, return_p=True)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert (P >= 0).all()


def test_zero_query_gives_mean_of_vbar():
    rng = np.random.default_rng(4)
    b, h, n, d, k = 2, 3, 17, 5, 6
    Q = np.zeros((b, h, n, d))
    K, V = _rand(rng, b, h, n, d), _rand(rng, b, h, n, d)
    E, F = _rand(rng, h, k, n), _rand(rng, h, k, n)
    O, _ = orc.linformer_fwd(Q, K, V, E, F, None, orc.PER_HEAD)
    for bi in range(b):
        for hi in range(h):
            mean = (F[hi] @ V[bi, hi]).mean(axis=0)
            np.testing.assert_allclose(O[bi, hi], np.broadcast_to(mean, (n, d)),
                                       rtol=1e-12, atol=1e-12)


def test_single_projected_position_gives_f_times_v():
    rng = np.random.default_rng(5)
    b, h, n, d = 2, 2, 11, 3
    Q, K, V = _rand(rng, b, h, n, d), _rand(rng, b, h, n, d), _rand(rng, b, h, n, d)
    E, F = _rand(rng, 1, n), _rand(rng, 1, n)
    O, _ = orc.linformer_fwd(Q, K, V, E, F, None, orc.HEADWISE)
    for bi in range(b):
        for hi in range(h):
            np.testing.assert_allclose(O[bi, hi], np.broadcast_to(F @ V[bi, hi], (n, d)),
                                       rtol=1e-12, atol=1e-12)


def test_key_value_sharing_bitwise():
    rng = np.random.default_rng(6)
    b, h, n, d, k = 2, 3, 13, 4, 5
    Q, K = _rand(rng, b, h, n, d), _rand(rng, b, h, n, d)
    E = _rand(rng, h, k, n)
    # K = V with E = F: the two projections are the same numbers.
    _, _, Kb, Vb = orc.linformer_fwd(Q, K, K, E, None, None, orc.KV, return_proj=True)
    assert np.array_equal(Kb, Vb)
    # Key-value mode is per-head mode with F_h := E_h.
    V = _rand(rng, b, h, n, d)
    O_kv, _ = orc.linformer_fwd(Q, K, V, E, None, None, orc.KV)
    O_ph, _ = orc.linformer_fwd(Q, K, V, E, E.copy(), None, orc.PER_HEAD)
    assert np.array_equal(O_kv, O_ph)


def test_sharing_mode_equalities():
    rng = np.random.default_rng(8)
    b, h, n, d, k = 2, 3, 10, 4, 6
    Q, K, V = _rand(rng, b, h, n, d), _rand(rng, b, h, n, d), _rand(rng, b, h, n, d)
    E, F = _rand(rng, k, n), _rand(rng, k, n)
    O_hw, _ = orc.linformer_fwd(Q, K, V, E, F, None, orc.HEADWISE)
    O_ph, _ = orc.linformer_fwd(Q, K, V, np.stack([E] * h), np.stack([F] * h), None, orc.PER_HEAD)
    assert np.array_equal(O_hw, O_ph)
    O_lw, _ = orc.linformer_fwd(Q, K, V, E, None, None, orc.LAYERWISE)
    O_hw2, _ = orc.linformer_fwd(Q, K, V, E, E.copy(), None, orc.HEADWISE)
    assert np.array_equal(O_lw, O_hw2)
    # Distinct per-head projections really are picked per head.
    Eh, Fh = _rand(rng, h, k, n), _rand(rng, h, k, n)
    O, _ = orc.linformer_fwd(Q, K, V, Eh, Fh, None, orc.PER_HEAD)
    for hi in range(h):
        O1, _ = orc.linformer_fwd(Q[:, hi:hi + 1], K[:, hi:hi + 1], V[:, hi:hi + 1],
                                  Eh[hi], Fh[hi], None, orc.HEADWISE)
        assert np.array_equal(O[:, hi:hi + 1], O1)


def test_padding_garbage_invariance_and_truncation():
    rng = np.random.default_rng(9)
    b, h, n, d, k = 3, 2, 16, 4, 5
    Q, K, V = _rand(rng, b, h, n, d), _rand(rng, b, h, n, d), _rand(rng, b, h, n, d)
    E, F = _rand(rng, h, k, n), _rand(rng, h, k, n)
    lengths = np.array([16, 7, 1], np.int32)
    O, _ = orc.linformer_fwd(Q, K, V, E, F, lengths, orc.PER_HEAD)
    Kg, Vg, Qg = K.copy(), V.copy(), Q.copy()
    for bi, L in enumerate(lengths):
        Kg[bi, :, L:] = np.nan
        Vg[bi, :, L:] = 1e300
        Qg[bi, :, L:] = -np.inf
    Og, _ = orc.linformer_fwd(Qg, Kg, Vg, E, F, lengths, orc.PER_HEAD)
    assert np.array_equal(O, Og)
    for bi, L in enumerate(lengths):
        assert (O[bi, :, L:] == 0).all()
        Ot, _ = orc.linformer_fwd(Q[bi:bi + 1, :, :L], K[bi:bi + 1, :, :L], V[bi:bi + 1, :, :L],
                                  E[:, :, :L], F[:, :, :L], None, orc.PER_HEAD)
        np.testing.assert_allclose(O[bi, :, :L], Ot[0], rtol=1e-12, atol=1e-12)


def test_permuting_projected_positions():
    rng = np.random.default_rng(10)
    b, h, n, d, k = 1, 2, 12, 4, 7
    Q, K, V = _rand(rng, b, h, n, d), _rand(rng, b, h, n, d), _rand(rng, b, h, n, d)
    E, F = _rand(rng, h, k, n), _rand(rng, h, k, n)
    perm = rng.permutation(k)
    O1, _ = orc.linformer_fwd(Q, K, V, E, F, None, orc.PER_HEAD)
    O2, _ = orc.linformer_fwd(Q, K, V, E[:, perm], F[:, perm], None, orc.PER_HEAD)
    np.testing.assert_allclose(O1, O2, rtol=1e-12, atol=1e-12)


def test_linearity_in_v():
    rng = np.random.default_rng(11)
    b, h, n, d, k = 1, 2, 9, 3, 4
    Q, K, V = _rand(rng, b, h, n, d), _rand(rng, b, h, n, d), _rand(rng, b, h, n, d)
    E = _rand(rng, h, k, n)
    F = np.abs(_rand(rng, h, k, n))
    F /= F.sum(axis=2, keepdims=True)  # rows of F sum to one
    O, _ = orc.linformer_fwd(Q, K, V, E, F, None, orc.PER_HEAD)
    O3, _ = orc.linformer_fwd(Q, K, 3.0 * V, E, F, None, orc.PER_HEAD)
    np.testing.assert_allclose(O3, 3.0 * O, rtol=1e-12, atol=1e-12)
    c = np.array([0.5, -2.0, 7.0])
    Oc, _ = orc.linformer_fwd(Q, K, V + c, E, F, None, orc.PER_HEAD)
    np.testing.assert_allclose(Oc, O + c, rtol=1e-12, atol=1e-12)


def test_shape_example():
    """Shapes of the worked example: n=4096, d=64, k=256 (one unit, sampled rows)."""
    rng = np.random.default_rng(12)
    n, d, k = 4096, 64, 256
    E = _rand(rng, k, n, scale=1 / np.sqrt(k))
    K, V, Q = _rand(rng, n, d), _rand(rng, n, d), _rand(rng, n, d)
    Kb = orc.project(E, K)
    O, P = orc.attend(Q, Kb, orc.project(E, V), rows=np.array([0, 4095]), return_p=True)
    assert Kb.shape == (256, 64) and P.shape == (2, 256) and O.shape == (2, 64)


# --- planted mistakes: each must be caught by at least one pin ---------------------

MUTANTS = {
    "scale_1_over_d": ("const double scale = 1.0 / sqrt((double)d);\n    const double *q",
                       "const double scale = 1.0 / (double)d;\n    const double *q"),
    "transposed_E": ("acc += Ehat[(int64_t)j * n + t] * X[(int64_t)t * d + c];",
                     "acc += Ehat[(int64_t)t * n + j] * X[(int64_t)t * d + c];"),
    "F_replaced_by_E": ("*Fh = (share_mode == OR_KV || share_mode == OR_LAYERWISE) ? *Eh : F + off;",
                        "*Fh = *Eh;"),
    "padding_ignored_in_projection": ("for (int t = 0; t < L; ++t)\n            acc +=",
                                      "for (int t = 0; t < n; ++t)\n            acc +="),
    "padded_queries_not_zeroed": ("    if (i >= L) {\n        for (int c = 0; c < d; ++c) Orow[c] = 0.0;",
                                  "    if (0) {\n        for (int c = 0; c < d; ++c) Orow[c] = 0.0;"),
    "missing_normalisation": ("for (int j = 0; j < k; ++j) s[j] /= sum;", ""),
    "per_head_offset_dropped": ("? (int64_t)head * k * n : 0;", "? 0 : 0;"),
    "softmax_off_by_one_column": ("for (int j = 1; j < k; ++j) if (s[j] > m) m = s[j];\n    double sum = 0.0;\n    for (int j = 0; j < k; ++j)",
                                  "for (int j = 1; j < k; ++j) if (s[j] > m) m = s[j];\n    double sum = 0.0;\n    for (int j = 1; j < k; ++j)"),
    "lengths_not_clamped": ("return L < 0 ? 0 : (L > n ? n : L);", "return L > n ? n : (L < 0 ? 1 : L);"),
}


def _pins_pass(lib) -> bool:
    """Run the pins above against a given compiled oracle; False if any fails."""
    try:
        for path in GOLDEN:
            O, expected = _run_golden(path, lib=lib)
            if not np.allclose(O, expected, rtol=0, atol=1e-12):
                return False
        rng = np.random.default_rng(1)
        n, d = 6, 4
        Q, K, V = _rand(rng, 1, 1, n, d), _rand(rng, 1, 1, n, d), _rand(rng, 1, 1, n, d)
        I = np.eye(n)[None]
        O, _ = orc.linformer_fwd(Q, K, V, I, I, None, orc.PER_HEAD, lib=lib)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V)).numpy()
        if not np.allclose(O, ref, rtol=1e-12, atol=1e-12):
            return False
        E, X = _rand(rng, 3, 9), _rand(rng, 9, 2)
        if not np.allclose(orc.project(E, X, 5, lib=lib), E[:, :5] @ X[:5], atol=1e-12):
            return False
    except Exception:
        return False
    return True


def test_planted_mistakes_are_caught(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    assert _pins_pass(orc._load()), "the real oracle must pass every pin"
    src = open(orc._SRC).read()
    for name, (old, new) in MUTANTS.items():
        assert old in src, f"mutation {name} no longer applies to the oracle source"
        mutated = src.replace(old, new, 1)
        c_path = tmp_path / f"{name}.c"
        so_path = tmp_path / f"{name}.so"
        c_path.write_text(mutated)
        subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(so_path),
                        str(c_path), "-lm"], check=True)
        lib = orc._bind(str(so_path))
        assert not _pins_pass(lib), f"planted mistake '{name}' was not caught by any pin"
