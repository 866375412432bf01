"""The allocation-free entry point, linformer_attn_fwd_noalloc.

It exists for callers that may not allocate device memory when they run the
attention (fixed memory budgets, framework-owned allocations, allocator
callbacks, no stream-ordered pools): it takes its workspace from one fixed
device array in the library instead.  These tests call it through the C ABI and
compare it with linformer_attn_fwd, on two calls in a row so that the second call
starts from the array as the first one left it.  The file is named to be
collected last; it must also pass when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import rank_linear_complexity_gb300.linformer as lf
from rank_linear_complexity_gb300.workloads import BF16, BF16_F32OUT, HEADWISE, LAYERWISE, PER_HEAD
from tests.parity import case_inputs, check, host64, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

CASES = [
    # (b, h, n, d, k, share_mode, dtype, ragged)
    (4, 12, 2048, 64, 256, LAYERWISE, BF16, False),
    (2, 4, 1000, 64, 200, PER_HEAD, BF16, True),
    (1, 3, 8192, 64, 128, HEADWISE, BF16_F32OUT, False),
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}h{c[1]}n{c[2]}k{c[4]}m{c[5]}" for c in CASES])
def test_noalloc_matches_allocating_entry_point(case):
    b, h, n, d, k, mode, dtype, ragged = case
    x = case_inputs(b, h, n, d, k, mode, dtype, ragged=ragged, seed=41)
    g = to_device(x, DEV)
    out_dt = torch.float32 if dtype == BF16_F32OUT else torch.bfloat16
    ref = lf.attention(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], mode,
                       out_fp32=(dtype == BF16_F32OUT))
    torch.cuda.synchronize()
    for _ in range(2):
        O = torch.full((b, h, n, d), float("nan"), dtype=out_dt, device=DEV)
        st = lf.linformer_attn_fwd_noalloc(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], O,
                                           b, h, n, d, k, mode, dtype)
        assert st == 0, lf.status_string(st)
        torch.cuda.synchronize()
        assert lf.linformer_debug_read_device_status() == 0
        check(host64(O), host64(ref), dtype, f"noalloc vs linformer_attn_fwd {case}")


def test_noalloc_rejects_problems_larger_than_its_array():
    # 4096 units x k_pad 256 needs 512 MiB of images: refused before any launch.
    b, h, n, d, k = 512, 8, 64, 64, 256
    tiny = torch.empty(16, dtype=torch.bfloat16, device=DEV)
    st = lf.linformer_attn_fwd_noalloc(tiny, tiny, tiny, tiny, None, None, tiny, b, h, n, d, k,
                                       LAYERWISE, BF16)
    assert st == -2
    st = lf.linformer_attn_fwd_noalloc(tiny, tiny, tiny, tiny, None, None, tiny, 1, 1, 64, 32, 16,
                                       LAYERWISE, BF16)
    assert st == -3
