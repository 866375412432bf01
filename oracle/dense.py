"""fp64 CPU oracle for dense softmax attention, the full-attention baseline of the
Linformer pages' inference comparison.

TEST INFRASTRUCTURE ONLY (like oracle.py): only the tests, ``__graft_entry__`` and
``bench.py``'s CPU legs may import it; the CUDA library never does.

Definition: the scaled dot-product attention of the PaperWeekly efficient-Transformer
survey, section 2.1, O = softmax(Q K^T / sqrt(d)) V per (batch, head), which the page
"Linformer 요약 설명", section Inference-time Efficiency Results, times the method
against (the standard Transformer).  With padding the usual key mask applies (a
reading: the pages do not spell it out): keys t >= L take no part and query rows
i >= L give O = 0.  numpy matrix products are the only library primitive.
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().float().cpu().numpy()
    return np.asarray(a, dtype=np.float64)


def dense_fwd(Q, K, V, pad_lengths=None, rows=None):
    """O [b][h][n][d] in float64; with `rows` (query row indices) only those rows,
    O [b][h][len(rows)][d] (each row of the definition stands alone)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    b, h, n, d = Q.shape
    pad = None if pad_lengths is None else np.asarray(_f64(pad_lengths)).astype(np.int64)
    rows = np.arange(n) if rows is None else np.asarray(rows)
    O = np.zeros((b, h, len(rows), d))
    for bi in range(b):
        L = n if pad is None else int(min(max(pad[bi], 0), n))
        live = np.nonzero(rows < L)[0]                           # rows i >= L stay 0
        if L == 0 or live.size == 0:
            continue
        for hi in range(h):
            S = (Q[bi, hi, rows[live]] @ K[bi, hi, :L].T) / np.sqrt(d)  # valid keys only
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            O[bi, hi, live] = P @ V[bi, hi, :L]
    return O
