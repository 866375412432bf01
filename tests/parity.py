"""Shared helpers for the GPU parity tests: tolerances and input plumbing.

Tolerances (the accuracy bar of the Linformer attention forward, per output dtype):
  * fp32 in / fp32 out:   max|err| <= 1e-4 * max|O_ref|.
  * bf16 in / fp32 out:   max|err| <= 2e-2, and relL1 = sum|err| / sum|O_ref| <= 1e-2.
  * bf16 in / bf16 out:   |err| <= 2e-2 + 2^-8 |O_ref| per element (2^-8 |O| is the
                          rounding of the bf16 result itself), and relL1 <= 1e-2.
The mean elementwise relative error is reported but not gated (it is unstable
where O is near zero).
"""
from __future__ import annotations

import numpy as np
import torch

from rank_linear_complexity_gb300.workloads import BF16, BF16_F32OUT, F32, make_inputs

ABS_TOL = 2e-2
REL_L1_TOL = 1e-2
BF16_OUT_REL = 2.0 ** -8
FP32_REL = 1e-4


def errors(got, ref) -> dict:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    denom = np.abs(ref).sum()
    return {
        "max_err": float(err.max()) if err.size else 0.0,
        "max_ref": float(np.abs(ref).max()) if ref.size else 0.0,
        "rel_l1": float(err.sum() / denom) if denom > 0 else float(err.sum()),
        "mean_rel": float(np.mean(err / np.maximum(np.abs(ref), 1e-6))) if err.size else 0.0,
        "finite": bool(np.isfinite(got).all()),
    }


def check(got, ref, dtype: int, what: str = "") -> dict:
    """Assert the per-dtype bar above; returns the error summary."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    e = errors(got, ref)
    assert e["finite"], f"{what}: non-finite output"
    if dtype == F32:
        bound = FP32_REL * max(e["max_ref"], 1e-30)
        assert e["max_err"] <= bound, f"{what}: max|err| {e['max_err']:.3e} > {bound:.3e} {e}"
        return e
    if dtype == BF16:
        ratio = np.abs(got - ref) / (ABS_TOL + BF16_OUT_REL * np.abs(ref))
        e["worst_ratio"] = float(ratio.max()) if ratio.size else 0.0
        assert e["worst_ratio"] <= 1.0, f"{what}: |err| over bound, {e}"
    else:
        e["worst_ratio"] = e["max_err"] / ABS_TOL
        assert e["max_err"] <= ABS_TOL, f"{what}: max|err| {e['max_err']:.3e} {e}"
    if e["max_ref"] > 0 and np.abs(ref).sum() > 0:
        assert e["rel_l1"] <= REL_L1_TOL, f"{what}: relL1 {e['rel_l1']:.3e} {e}"
    return e


def to_device(x: dict, dev) -> dict:
    return {k: (v.to(dev) if v is not None else None) for k, v in x.items()}


def host64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def case_inputs(b, h, n, d, k, share_mode, dtype, ragged=False, seed=0, lengths=None):
    x = make_inputs(b, h, n, d, k, share_mode, dtype, ragged=ragged, seed=seed)
    if lengths is not None:
        x["lengths"] = torch.tensor(lengths, dtype=torch.int32)
    return x
