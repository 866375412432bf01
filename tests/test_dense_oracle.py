"""The dense-attention oracle (oracle/dense.py) against what fixes it independently:
the Linformer C oracle with identity projections (k = n, E = F = I, where the method
is full attention), scalar loops on a tiny case, and closed forms."""
import math

import numpy as np
import pytest
import torch

from oracle import dense
from oracle import oracle as orc
from rank_linear_complexity_gb300.workloads import F32, PER_HEAD, make_inputs


def test_equals_linformer_with_identity_projections():
    b, h, n, d = 2, 3, 40, 16
    x = make_inputs(b, h, n, d, n, PER_HEAD, F32, seed=11)
    I = torch.eye(n).expand(h, n, n).contiguous()
    O_lin, _ = orc.linformer_fwd(x["Q"], x["K"], x["V"], I, I, None, PER_HEAD)
    O = dense.dense_fwd(x["Q"], x["K"], x["V"])
    assert np.abs(O - O_lin).max() <= 1e-12 * max(1.0, np.abs(O_lin).max())


def test_scalar_loops_on_a_tiny_case():
    rng = np.random.default_rng(0)
    b, h, n, d = 1, 2, 5, 3
    Q, K, V = (rng.standard_normal((b, h, n, d)) for _ in range(3))
    lengths = np.array([4])
    O = dense.dense_fwd(Q, K, V, lengths)
    for hi in range(h):
        for i in range(n):
            for c in range(d):
                if i >= 4:
                    want = 0.0
                else:
                    s = [sum(Q[0, hi, i, e] * K[0, hi, t, e] for e in range(d)) / math.sqrt(d)
                         for t in range(4)]
                    m = max(s)
                    w = [math.exp(v - m) for v in s]
                    want = sum(w[t] * V[0, hi, t, c] for t in range(4)) / sum(w)
                assert abs(O[0, hi, i, c] - want) < 1e-12


def test_zero_queries_average_the_valid_values():
    rng = np.random.default_rng(1)
    b, h, n, d = 2, 1, 12, 4
    Q = np.zeros((b, h, n, d))
    K, V = rng.standard_normal((b, h, n, d)), rng.standard_normal((b, h, n, d))
    O = dense.dense_fwd(Q, K, V, np.array([7, 12]))
    assert np.allclose(O[0, 0, :7], V[0, 0, :7].mean(axis=0), atol=1e-14)
    assert not O[0, 0, 7:].any()
    assert np.allclose(O[1, 0], V[1, 0].mean(axis=0), atol=1e-14)


def test_padding_is_truncation_and_ignores_padded_values():
    rng = np.random.default_rng(2)
    b, h, n, d, L = 1, 2, 20, 8, 13
    Q, K, V = (rng.standard_normal((b, h, n, d)) for _ in range(3))
    ref = dense.dense_fwd(Q[:, :, :L], K[:, :, :L], V[:, :, :L])
    Qp, Kp, Vp = Q.copy(), K.copy(), V.copy()
    for t in (Qp, Kp, Vp):
        t[:, :, L:] = np.nan
    O = dense.dense_fwd(Qp, Kp, Vp, np.array([L]))
    assert np.array_equal(O[:, :, :L], ref) and not O[:, :, L:].any()


def test_single_key_returns_its_value():
    rng = np.random.default_rng(3)
    Q, K, V = (rng.standard_normal((1, 1, 6, 5)) for _ in range(3))
    O = dense.dense_fwd(Q, K, V, np.array([1]))
    assert np.allclose(O[0, 0, 0], V[0, 0, 0], atol=1e-15)


@pytest.mark.parametrize("bad", ["keys_misaligned_with_values", "no_scale"])
def test_pins_catch_planted_mistakes(bad, monkeypatch):
    """An index mistake (keys paired with the wrong values) or a dropped 1/sqrt(d) in
    the oracle fails the identity pin."""
    real = dense.dense_fwd

    def wrong(Q, K, V, pad_lengths=None):
        Q64, K64, V64 = dense._f64(Q), dense._f64(K), dense._f64(V)
        if bad == "keys_misaligned_with_values":
            return real(Q64, K64[:, :, ::-1].copy(), V64)
        return real(Q64 * np.sqrt(Q64.shape[3]), K64, V64)

    monkeypatch.setattr(dense, "dense_fwd", wrong)
    with pytest.raises(AssertionError):
        test_equals_linformer_with_identity_projections()


def test_row_subsets_match_the_whole():
    rng = np.random.default_rng(4)
    Q, K, V = (rng.standard_normal((2, 2, 30, 8)) for _ in range(3))
    lengths = np.array([17, 30])
    full = dense.dense_fwd(Q, K, V, lengths)
    rows = np.array([0, 16, 17, 29])
    assert np.array_equal(dense.dense_fwd(Q, K, V, lengths, rows=rows), full[:, :, rows])
