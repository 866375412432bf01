"""The backward oracle (oracle/backward.py) against what fixes it independently of
its formulas: central finite differences of the C forward oracle, autograd through
the forward written as plain PyTorch operations, and the k = n, E = F = I case,
where the method is softmax attention and its gradients are the textbook ones."""
import numpy as np
import pytest
import torch

from oracle import backward as bw
from oracle import oracle as orc
from rank_linear_complexity_gb300.workloads import F32, HEADWISE, KV, LAYERWISE, PER_HEAD
from tests.parity import case_inputs


def loss_and_weights(x, mode, W):
    O, _ = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], mode)
    return float((O * W).sum())


@pytest.mark.parametrize("mode", [PER_HEAD, KV, HEADWISE, LAYERWISE])
def test_finite_differences(mode):
    b, h, n, d, k = 2, 2, 24, 8, 6
    x = case_inputs(b, h, n, d, k, mode, F32, ragged=True, seed=3 + mode)
    x = {kk: (v.double() if v is not None and v.dtype.is_floating_point else v) for kk, v in x.items()}
    W = np.random.default_rng(mode).standard_normal((b, h, n, d))
    dQ, dK, dV, dE, dF = bw.linformer_bwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], W, mode)
    grads = {"Q": dQ, "K": dK, "V": dV, "E": dE}
    if dF is not None:
        grads["F"] = dF
    rng = np.random.default_rng(10 + mode)
    eps = 1e-5
    for name, g in grads.items():
        t = x[name]
        for _ in range(12):
            idx = tuple(int(rng.integers(s)) for s in t.shape)
            keep = t[idx].item()
            t[idx] = keep + eps
            up = loss_and_weights(x, mode, W)
            t[idx] = keep - eps
            dn = loss_and_weights(x, mode, W)
            t[idx] = keep
            fd = (up - dn) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


def forward_torch(Q, K, V, E, F, lengths, mode):
    """The forward as plain torch operations (autograd derives the gradients)."""
    b, h, n, d = Q.shape
    out = []
    for bi in range(b):
        L = n if lengths is None else int(lengths[bi])
        mask = (torch.arange(n) < L).double()[:, None]
        rows = []
        for hi in range(h):
            Eh = E[hi] if mode in (PER_HEAD, KV) else E
            Fh = Eh if mode in (KV, LAYERWISE) else (F[hi] if mode == PER_HEAD else F)
            Kb = Eh @ (K[bi, hi] * mask)
            Vb = Fh @ (V[bi, hi] * mask)
            P = torch.softmax(Q[bi, hi] @ Kb.T / d ** 0.5, dim=1)
            rows.append((P @ Vb) * mask)
        out.append(torch.stack(rows))
    return torch.stack(out)


def check_autograd(mode, oracle_bwd=None):
    oracle_bwd = oracle_bwd or bw.linformer_bwd
    b, h, n, d, k = 2, 3, 40, 16, 12
    x = case_inputs(b, h, n, d, k, mode, F32, ragged=True, seed=20 + mode)
    t = {kk: (v.double().requires_grad_(True) if v is not None and v.dtype.is_floating_point else v)
         for kk, v in x.items()}
    W = torch.randn(b, h, n, d, dtype=torch.float64, generator=torch.Generator().manual_seed(mode))
    (forward_torch(t["Q"], t["K"], t["V"], t["E"], t["F"], x["lengths"], mode) * W).sum().backward()
    dQ, dK, dV, dE, dF = oracle_bwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"],
                                    W.numpy(), mode)
    pairs = [(dQ, t["Q"]), (dK, t["K"]), (dV, t["V"]), (dE, t["E"])]
    if dF is not None:
        pairs.append((dF, t["F"]))
    for got, ref in pairs:
        assert np.abs(got - ref.grad.numpy()).max() <= 1e-10 * max(1.0, ref.grad.abs().max().item())


@pytest.mark.parametrize("mode", [PER_HEAD, KV, HEADWISE, LAYERWISE])
def test_autograd(mode):
    check_autograd(mode)


# Plausible mistakes, each planted in a copy of the oracle's source: every one must make
# the autograd pin fail in at least one sharing mode.  (Keeping dO's padded rows is not
# among them: P's padded rows are zero, so those rows reach no gradient.)
PLANTED = {
    "dQ without the 1/sqrt(d) scale": ("dQ[bi, hi] = (dS @ Kb) * scale", "dQ[bi, hi] = dS @ Kb"),
    "softmax backward without the row-sum term": (
        "dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))", "dS = P * dP"),
    "dVbar scaled by 1/sqrt(d) as well": ("dVb = P.T @ G", "dVb = (P.T @ G) * scale"),
    "padded dK rows not zeroed": ("dK[bi, hi, L:] = 0.0", "pass"),
    "F term dropped when F is E": ("(dE[hi] if per_head else dE)[...] += gE + gF",
                                   "(dE[hi] if per_head else dE)[...] += gE"),
    "shared E overwritten instead of summed": (
        "(dE[hi] if per_head else dE)[...] += gE\n", "(dE[hi] if per_head else dE)[...] = gE\n"),
}


@pytest.mark.parametrize("name", sorted(PLANTED))
def test_planted_mistakes_are_caught(name):
    import types
    old, new = PLANTED[name]
    src = open(bw.__file__).read()
    assert src.count(old) == 1, f"planting site not found: {old}"
    mod = types.ModuleType("planted_backward")
    exec(compile(src.replace(old, new), "planted_backward", "exec"), mod.__dict__)
    caught = 0
    for mode in (PER_HEAD, KV, HEADWISE, LAYERWISE):
        try:
            check_autograd(mode, mod.linformer_bwd)
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin fails with the mistake: {name}"


def test_identity_projection_is_attention_backward():
    n, d = 16, 8
    g = torch.Generator().manual_seed(4)
    Q, K, V, dO = (torch.randn(1, 1, n, d, dtype=torch.float64, generator=g) for _ in range(4))
    I = torch.eye(n, dtype=torch.float64)
    dQ, dK, dV, dE, _ = bw.linformer_bwd(Q, K, V, I, None, None, dO, LAYERWISE)
    # textbook softmax-attention gradients
    q, kk, v, go = Q[0, 0].numpy(), K[0, 0].numpy(), V[0, 0].numpy(), dO[0, 0].numpy()
    P = np.exp(q @ kk.T / np.sqrt(d)); P /= P.sum(1, keepdims=True)
    dv = P.T @ go
    dp = go @ v.T
    ds = P * (dp - (P * dp).sum(1, keepdims=True)) / np.sqrt(d)
    for got, ref in ((dQ[0, 0], ds @ kk), (dK[0, 0], ds.T @ q), (dV[0, 0], dv)):
        assert np.abs(got - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
