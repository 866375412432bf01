"""Device-side failure detection without a fault: a bounded wait on a barrier nothing
completes runs out after its limit (2 s), the kernel records the failure in the
device status word and exits, the host reads LINFORMER_ERR_DEVICE, and the same
context then runs a forward that matches the oracle."""
import time

import numpy as np
import pytest
import torch

import rank_linear_complexity_gb300.linformer as lf
from oracle import oracle as orc
from rank_linear_complexity_gb300.workloads import BF16, LAYERWISE, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ERR_DEVICE = -9


def test_bounded_wait_runs_out_and_the_context_survives():
    torch.cuda.set_device(DEV)
    assert lf.linformer_debug_read_device_status() == 0  # nothing pending from earlier tests
    t0 = time.perf_counter()
    assert lf.linformer_debug_wait_probe() == 0
    assert lf.linformer_debug_read_device_status() == ERR_DEVICE  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert 1.5 < elapsed < 60, elapsed
    assert lf.linformer_debug_read_device_status() == 0  # read and cleared

    x = make_inputs(2, 3, 320, 64, 128, LAYERWISE, BF16, seed=5)
    g = {c: (v.to(DEV) if v is not None else None) for c, v in x.items()}
    O = lf.attention(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], LAYERWISE)
    torch.cuda.synchronize()
    assert lf.linformer_debug_read_device_status() == 0
    ref, _ = orc.linformer_fwd(x["Q"], x["K"], x["V"], x["E"], x["F"], x["lengths"], LAYERWISE)
    err = np.abs(O.float().cpu().numpy() - ref)
    assert (err <= 2e-2 + 2.0 ** -8 * np.abs(ref)).all()
