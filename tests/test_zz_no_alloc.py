"""The allocation-free entry point, linformer_attn_fwd_noalloc.

It exists for callers that may not allocate device memory when they run the
attention (fixed memory budgets, framework-owned allocations, allocator
callbacks, no stream-ordered pools): it takes its workspace from one fixed
device array in the library instead.  These tests call it through the C ABI and
compare it with the fp64 oracle and with linformer_attn_fwd, on two calls in a row
so that the second call starts from the array as the first one left it.  A further
test runs the entry point in a fresh process, before any allocating call of the
library, and checks that no device memory is taken while it runs.  The file is
named to be collected last; it must also pass when run alone in a fresh process.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import rank_linear_complexity_gb300.linformer as lf
from oracle import oracle as orc
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
    exact, _ = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], mode)
    for _ in range(2):
        O = torch.full((b, h, n, d), float("nan"), dtype=out_dt, device=DEV)
        st = lf.linformer_attn_fwd_noalloc(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], O,
                                           b, h, n, d, k, mode, dtype)
        assert st == 0, lf.status_string(st)
        torch.cuda.synchronize()
        assert lf.linformer_debug_read_device_status() == 0
        check(host64(O), exact, dtype, f"noalloc vs the oracle {case}")
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


_FRESH = textwrap.dedent("""
    import json, sys, torch
    sys.path.insert(0, {root!r})
    import rank_linear_complexity_gb300.linformer as lf
    from rank_linear_complexity_gb300.workloads import make_inputs
    b, h, n, d, k = 2, 6, 2048, 64, 256
    x = make_inputs(b, h, n, d, k, 3, 1, seed=5)
    g = {{kk: (v.cuda() if v is not None else None) for kk, v in x.items()}}
    O = torch.empty((b, h, n, d), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    call = lambda: lf.linformer_attn_fwd_noalloc(g["Q"], g["K"], g["V"], g["E"], None, None,
                                                 O, b, h, n, d, k, 3, 1)
    out = {{"first": call()}}  # first call on the device: looks up the array's address
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    out["second"] = call()
    torch.cuda.synchronize()
    out["free_delta"] = torch.cuda.mem_get_info()[0] - free0
    out["pool_peak"] = lf.linformer_pool_peak_bytes()
    out["status"] = lf.linformer_debug_read_device_status()
    # the allocating entry point in the same process does draw from the pool
    O2 = torch.empty_like(O)
    out["alloc_call"] = lf.linformer_attn_fwd(g["Q"], g["K"], g["V"], g["E"], None, None, O2,
                                              b, h, n, d, k, 3, 1)
    torch.cuda.synchronize()
    out["pool_peak_after_alloc_call"] = lf.linformer_pool_peak_bytes()
    out["same"] = bool(torch.equal(O, O2))
    print(json.dumps(out))
""")


def test_noalloc_takes_no_device_memory_in_a_fresh_process():
    """Run first in a new process: no pool allocation, and free device memory unchanged
    across the call (the allocating entry point, run afterwards, shows the measurement
    would see one)."""
    import json
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH.format(root=root)], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["first"] == 0 and out["second"] == 0 and out["status"] == 0, out
    assert out["pool_peak"] == 0, out
    assert out["free_delta"] == 0, out
    assert out["alloc_call"] == 0 and out["pool_peak_after_alloc_call"] > 0, out
    assert out["same"], out
