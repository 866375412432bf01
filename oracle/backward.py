"""fp64 CPU oracle for the Linformer attention backward: the gradients of the
forward's output O with respect to Q, K, V, E and F, given dO.

TEST INFRASTRUCTURE ONLY (like oracle.py): only the tests, ``__graft_entry__``
and ``bench.py``'s CPU legs may import it; the CUDA library never does.

The forward is the definition in "Linformer(Self-Attention with Linear
Complexity) 요약 설명", section Model (Kbar = E.K, Vbar = F.V with E, F of shape
k x n; rows t >= L of K and V count as zero and query rows i >= L give O = 0,
padding paragraph) with the scaled dot product of the PaperWeekly survey,
section 2.1, and the sharing modes of the 中文验证版 page, section 方法适配.  The
pages use the method for training (the 요약 설명 page, section Experiments), so its
gradients are the chain rule through that definition, one step per line below,
with numpy matrix products as the only library primitive.  Pinned, independently of
these formulas, by finite differences of the C forward and by autograd.
"""
from __future__ import annotations

import numpy as np

PER_HEAD, KV, HEADWISE, LAYERWISE = 0, 1, 2, 3


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().float().cpu().numpy() if str(a.dtype) == "torch.bfloat16" else a.detach().cpu().numpy()
    return np.asarray(a, dtype=np.float64)


def linformer_bwd(Q, K, V, E, F, pad_lengths, dO, share_mode: int):
    """Returns dQ, dK, dV [b][h][n][d], dE (shaped like E) and dF (like F, or None
    when F is E: KV and LAYERWISE modes, whose dE holds both contributions)."""
    Q, K, V, E, dO = _f64(Q), _f64(K), _f64(V), _f64(E), _f64(dO)
    distinct = share_mode in (PER_HEAD, HEADWISE)
    per_head = share_mode in (PER_HEAD, KV)
    F = _f64(F) if distinct else None
    b, h, n, d = Q.shape
    pad = None if pad_lengths is None else np.asarray(_f64(pad_lengths)).astype(np.int64)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    dE = np.zeros_like(E)
    dF = np.zeros_like(F) if distinct else None
    scale = 1.0 / np.sqrt(d)
    for bi in range(b):
        L = n if pad is None else int(min(max(pad[bi], 0), n))
        for hi in range(h):
            Eh = E[hi] if per_head else E
            Fh = (F[hi] if per_head else F) if distinct else Eh
            Km = K[bi, hi].copy(); Km[L:] = 0.0          # rows t >= L count as zero
            Vm = V[bi, hi].copy(); Vm[L:] = 0.0
            Kb = Eh @ Km                                  # k x d
            Vb = Fh @ Vm
            S = (Q[bi, hi] @ Kb.T) * scale                # n x k
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            P[L:] = 0.0                                   # rows i >= L: O = 0, no gradient
            G = dO[bi, hi].copy(); G[L:] = 0.0
            dVb = P.T @ G                                 # O = P Vbar
            dP = G @ Vb.T
            dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))   # softmax, row by row
            dQ[bi, hi] = (dS @ Kb) * scale                # S = Q Kbar^T / sqrt(d)
            dKb = (dS.T @ Q[bi, hi]) * scale
            dK[bi, hi] = Eh.T @ dKb                        # Kbar = E Km
            dK[bi, hi, L:] = 0.0
            dV[bi, hi] = Fh.T @ dVb                        # Vbar = F Vm
            dV[bi, hi, L:] = 0.0
            gE = dKb @ Km.T
            gF = dVb @ Vm.T
            if distinct:
                (dE[hi] if per_head else dE)[...] += gE
                (dF[hi] if per_head else dF)[...] += gF
            else:                                          # F is E
                (dE[hi] if per_head else dE)[...] += gE + gF
    return dQ, dK, dV, dE, dF
