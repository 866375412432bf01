"""The fp32 forward (split projections, scores, row softmax and P.Vbar on the SIMT
product kernel) at the long-sequence sizes of the inference comparison: sampled rows
of sampled units against the fp64 oracle, which computes them row by row, at the fp32
bar (max|err| <= 1e-4 max|O_ref|); all outputs finite, padded rows zero."""
import numpy as np
import pytest
import torch

import rank_linear_complexity_gb300.linformer as lf
from oracle import oracle as orc
from rank_linear_complexity_gb300.workloads import F32, HEADWISE, LAYERWISE, make_inputs
from tests.parity import check, host64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.mark.parametrize("b,h,n,k,mode,ragged", [
    (1, 12, 65536, 128, LAYERWISE, False),
    (1, 12, 65536, 256, HEADWISE, False),
    (16, 12, 4096, 256, LAYERWISE, True),
])
def test_fp32_forward_long_sequences(b, h, n, k, mode, ragged):
    d = 64
    x = make_inputs(b, h, n, d, k, mode, F32, ragged=ragged, seed=n + k)
    g = {c: (v.to(DEV) if v is not None else None) for c, v in x.items()}
    O = lf.attention(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], mode)
    torch.cuda.synchronize()
    assert lf.linformer_debug_read_device_status() == 0
    assert torch.isfinite(O).all()
    rng = np.random.default_rng(n)
    for bi, hi in [(0, 0), (b - 1, h - 1), (b // 2, h // 3)]:
        L = n if x["lengths"] is None else int(x["lengths"][bi])
        rows = np.unique(np.r_[0, max(L - 1, 0), rng.integers(0, max(L, 1), 12)])
        ref, _, _ = orc.unit_rows(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], mode,
                                  bi, hi, rows)
        got = host64(O[bi, hi][torch.from_numpy(rows).to(DEV)])
        check(got, ref, F32, f"unit ({bi},{hi})")
        if L < n:
            assert not O[bi, hi, L:].any()
