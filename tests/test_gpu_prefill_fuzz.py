"""Seeded random shapes for the forward pass against the fp64 oracle, whole output:
query and key lengths that cut tiles anywhere (including no keys), grouped heads,
every head dimension, both 16-bit types, causal offsets, sliding windows and
softcap in random combinations, through the plain forward and the split-KV entry.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_parity, f64, gather

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from tiled_exact_attention_gb300 import fa_fwd, fa_fwd_splitkv, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300.inputs import make_custom  # noqa: E402

DEV = "cuda:0"


def _draw(i):
    rng = np.random.default_rng(8000 + i)
    g = int(rng.choice([1, 2, 4, 8]))
    hkv = int(rng.integers(1, 3))
    d = int(rng.choice([64, 128, 256]))
    b = int(rng.integers(1, 3))
    sq = int(rng.integers(1, 700))
    skv = int(rng.integers(0, 900))
    causal = bool(rng.integers(0, 2))
    off = int(rng.integers(-50, 600)) if causal and rng.integers(0, 2) else None
    window = None
    if rng.integers(0, 3) == 0:
        window = (int(rng.integers(-1, 300)), int(rng.integers(-1, 300)))
    softcap = float(rng.uniform(2.0, 20.0)) if rng.integers(0, 3) == 0 else 0.0
    dt = str(rng.choice(["bf16", "fp16"]))
    split = bool(rng.integers(0, 2))
    return b, sq, skv, g * hkv, hkv, d, dt, causal, off, window, softcap, split


@pytest.mark.parametrize("i", range(24))
def test_forward_random(i):
    b, sq, skv, hq, hkv, d, dt, causal, off, window, c, split = case = _draw(i)
    q, k, v = (t.to(DEV) for t in make_custom(b, sq, skv, hq, hkv, d, dt, seed=8100 + i))
    if split:
        o, lse = fa_fwd_splitkv(q, k, v, causal=causal, q_pos_offset=off, window=window, softcap=c, num_splits=3)
    else:
        o, lse = fa_fwd(q, k, v, causal=causal, q_pos_offset=off, window=window, softcap=c)
    assert fa_sync_status() == 0
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v), causal=causal, q_pos_offset=off,
                                    scale=1.0 / math.sqrt(d), rows=rows, window=window or (-1, -1), softcap=c)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, q.dtype, f"random forward {i}: {case}")
