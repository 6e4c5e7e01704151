"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module only draws random numbers and rounds them to the storage dtype; it
holds none of the attention arithmetic.  Q, K and V are iid N(0, std^2) drawn
with numpy's PCG64 generator (bit-stable across platforms), rounded to bf16 or
fp16 by round-to-nearest-even, in the [batch, seq, heads, head_dim] layout.
Seeds are 20261202 + workload index; Q, K and V use independent streams.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

BASE_SEED = 20261202

_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    b: int
    sq: int
    skv: int
    hq: int
    hkv: int
    d: int
    dtype: str
    causal: bool
    std: float
    index: int
    q_pos_offset: int | None = None  # None: bottom-right alignment, skv - sq

    @property
    def torch_dtype(self):
        return _DTYPES[self.dtype]

    @property
    def offset(self) -> int:
        return self.skv - self.sq if self.q_pos_offset is None else self.q_pos_offset

    def visible_pairs_per_head(self) -> int:
        """Number of (query, key) pairs with key j visible to row i (integer count)."""
        if not self.causal:
            return self.sq * self.skv
        i = np.arange(self.sq, dtype=np.int64)
        lim = np.clip(i + self.offset + 1, 0, self.skv)
        return int(lim.sum())


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 1, 128, 128, 2, 2, 64, "bf16", False, 1.0, 0),
        Workload("causal_prefill", 4, 4096, 4096, 16, 16, 128, "bf16", True, 1.0, 1, 0),
        Workload("gqa_long", 1, 16384, 16384, 32, 8, 128, "bf16", True, 1.0, 2, 0),
        Workload("ragged_d64", 2, 5000, 5000, 16, 16, 64, "fp16", False, 2.0, 3),
        Workload("ragged_d256", 2, 5000, 5000, 16, 16, 256, "fp16", False, 2.0, 3),
        Workload("ragged_n5", 1, 5, 5, 1, 1, 64, "fp16", True, 2.0, 3, 0),
        Workload("decode", 8, 1, 32768, 32, 8, 128, "bf16", True, 1.0, 4, 32767),
    ]
}


def normal(shape, seed: int, stream: int, std: float = 1.0, dtype: torch.dtype = torch.bfloat16,
           chunk: int = 1 << 26) -> torch.Tensor:
    """iid N(0, std^2) rounded to `dtype`, on the CPU, deterministic in (seed, stream)."""
    n = int(np.prod(shape))
    gen = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))
    out = torch.empty(n, dtype=dtype)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = gen.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[s:e] = torch.from_numpy(x).to(dtype)
    return out.reshape(shape)


def make_qkv(w: Workload | str, seed_offset: int = 0):
    """(q, k, v) CPU tensors for a workload: q [b, sq, hq, d], k/v [b, skv, hkv, d]."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    seed = BASE_SEED + w.index + seed_offset
    q = normal((w.b, w.sq, w.hq, w.d), seed, 0, w.std, w.torch_dtype)
    k = normal((w.b, w.skv, w.hkv, w.d), seed, 1, w.std, w.torch_dtype)
    v = normal((w.b, w.skv, w.hkv, w.d), seed, 2, w.std, w.torch_dtype)
    return q, k, v


def make_custom(b, sq, skv, hq, hkv, d, dtype="bf16", std=1.0, seed=BASE_SEED + 100):
    dt = _DTYPES[dtype] if isinstance(dtype, str) else dtype
    q = normal((b, sq, hq, d), seed, 0, std, dt)
    k = normal((b, skv, hkv, d), seed, 1, std, dt)
    v = normal((b, skv, hkv, d), seed, 2, std, dt)
    return q, k, v
