"""Seeded synthetic inputs for the Linformer attention forward.

This module holds the workload table and the random-input recipe only: it does
none of the method's arithmetic.  Both the CUDA path's tests/benchmark and the
oracle's checks take their inputs from here.

Recipe (the pages benchmark on randomly generated inputs: "Linformer: Self-Attention
with Linear Complexity - 中文验证版", section 计算设置; "Linformer 요약 설명", section
Inference-time Efficiency Results):
  * Q, K, V ~ N(0, 1); E, F ~ N(0, 1/k) (the random-projection scale of the
    Johnson-Lindenstrauss argument in "Linformer 요약 설명", section Self-Attention
    is Low Rank);
  * drawn in fp32 from a CPU ``torch.Generator`` seeded with ``seed``, in the
    order Q, K, V, E, F, lengths, then cast to the workload's dtype;
  * ragged batches draw valid lengths uniformly from [n/4, n].
"""
from __future__ import annotations

import dataclasses

import torch

PER_HEAD, KV, HEADWISE, LAYERWISE = 0, 1, 2, 3
SHARE_NAMES = {PER_HEAD: "per_head", KV: "key_value", HEADWISE: "headwise",
               LAYERWISE: "layerwise"}
F32, BF16, BF16_F32OUT = 0, 1, 2


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    b: int
    h: int
    n: int
    d: int
    k: int
    share_mode: int
    dtype: int
    ragged: bool = False
    seed: int = 1234

    @property
    def units(self) -> int:
        return self.b * self.h

    @property
    def tokens(self) -> int:
        return self.b * self.h * self.n

    def describe(self) -> dict:
        return {"workload": self.name, "b": self.b, "h": self.h, "n": self.n, "d": self.d,
                "k": self.k, "share_mode": SHARE_NAMES[self.share_mode],
                "ragged": self.ragged}


# The five workloads of the method's evaluation: a small fp32 case, a RoBERTa-base
# shaped batch, the long-sequence n=4096/k=256 case, the n=65536 case and a
# ragged padded batch (shapes from the pages' inference table: n in {512, 4096,
# 65536}, k in {128, 256}; d = 64, h = 12 as in RoBERTa-base).
WORKLOADS = [
    Workload("fp32_b2h4_n512_k128_per_head", 2, 4, 512, 64, 128, PER_HEAD, F32, seed=1234),
    Workload("bf16_b32h12_n512_k128_key_value", 32, 12, 512, 64, 128, KV, BF16, seed=1235),
    Workload("bf16_b16h12_n4096_k256_layerwise", 16, 12, 4096, 64, 256, LAYERWISE, BF16,
             seed=1236),
    Workload("bf16_b1h12_n65536_k128_headwise", 1, 12, 65536, 64, 128, HEADWISE, BF16,
             seed=1237),
    Workload("bf16_b8h16_n16384_k256_per_head_ragged", 8, 16, 16384, 64, 256, PER_HEAD, BF16,
             ragged=True, seed=1238),
]
HEADLINE = WORKLOADS[2]


def torch_dtype(dtype: int) -> torch.dtype:
    return torch.float32 if dtype == F32 else torch.bfloat16


def out_dtype(dtype: int) -> torch.dtype:
    return torch.bfloat16 if dtype == BF16 else torch.float32


def projection_shape(share_mode: int, h: int, k: int, n: int) -> tuple:
    return (h, k, n) if share_mode in (PER_HEAD, KV) else (k, n)


def has_distinct_f(share_mode: int) -> bool:
    return share_mode in (PER_HEAD, HEADWISE)


def make_inputs(b: int, h: int, n: int, d: int, k: int, share_mode: int, dtype: int,
                ragged: bool = False, seed: int = 1234, lengths_range=None) -> dict:
    """Seeded inputs on the CPU: dict with Q, K, V, E, F (None if F = E), lengths."""
    g = torch.Generator().manual_seed(seed)
    td = torch_dtype(dtype)
    Q = torch.randn(b, h, n, d, generator=g, dtype=torch.float32).to(td)
    K = torch.randn(b, h, n, d, generator=g, dtype=torch.float32).to(td)
    V = torch.randn(b, h, n, d, generator=g, dtype=torch.float32).to(td)
    shp = projection_shape(share_mode, h, k, n)
    scale = 1.0 / (k ** 0.5)
    E = (torch.randn(*shp, generator=g, dtype=torch.float32) * scale).to(td)
    F = None
    if has_distinct_f(share_mode):
        F = (torch.randn(*shp, generator=g, dtype=torch.float32) * scale).to(td)
    lengths = None
    if ragged:
        lo, hi = lengths_range if lengths_range is not None else (max(0, n // 4), n)
        lengths = torch.randint(lo, hi + 1, (b,), generator=g, dtype=torch.int32)
    return {"Q": Q, "K": K, "V": V, "E": E, "F": F, "lengths": lengths}


def workload_inputs(w: Workload) -> dict:
    return make_inputs(w.b, w.h, w.n, w.d, w.k, w.share_mode, w.dtype, w.ragged, w.seed)


def output_gradient(b: int, h: int, n: int, d: int, seed: int = 4321) -> torch.Tensor:
    """Seeded upstream gradient dLoss/dO for the backward: N(0, 1), fp32, on the CPU."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn(b, h, n, d, generator=g, dtype=torch.float32)
