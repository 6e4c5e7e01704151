"""GPU parity of fa_bwd (recompute-based backward pass) against the fp64 oracle.

The forward pass runs on the GPU (fa_fwd) to produce O and LSE as a training
step would; the oracle recomputes everything from Q, K, V and dO in fp64.
Tolerance: the kernels round P and dS to the storage type before the tensor-core
products and read O back in that type for D = rowsum(dO * O), so the error of a
gradient grows with the sums it is made of; it is checked against the size of the
reference tensor: max |dX - dX_ref| <= TOL_REL * max |dX_ref| per tensor.
"""
from __future__ import annotations

import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from parity_util import f64

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from tiled_exact_attention_gb300 import fa_bwd, fa_fwd, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300.inputs import make_custom, normal  # noqa: E402

DEV = "cuda:0"
TOL_REL = {torch.bfloat16: 1e-2, torch.float16: 2e-3}


def _seed(case) -> int:
    return 9000 + zlib.crc32(repr(case).encode()) % 100000


def _check(name, got, ref, dt, what):
    g = got.to(torch.float64).cpu().numpy()
    assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
    scale = max(np.abs(ref).max(), 1e-6)
    err = np.abs(g - ref).max()
    assert err <= TOL_REL[dt] * scale, f"{what}: {name} max|diff| {err:.3e} > {TOL_REL[dt]} * {scale:.3e}"
    return err / scale


CASES = [
    # b, sq, skv, hq, hkv, d, dtype, causal, offset, window
    (1, 128, 128, 2, 2, 64, "bf16", False, None, None),
    (1, 300, 300, 4, 2, 128, "bf16", True, None, None),
    (2, 257, 130, 2, 1, 128, "fp16", False, None, None),
    (1, 200, 400, 2, 2, 64, "bf16", True, None, None),
    (1, 513, 513, 2, 1, 128, "bf16", False, None, (100, 0)),
    (1, 300, 300, 2, 2, 128, "bf16", True, -40, None),
    (1, 1, 500, 4, 1, 128, "bf16", False, None, None),
    (1, 640, 640, 8, 2, 128, "bf16", True, None, None),
    (1, 100, 60, 2, 2, 64, "fp16", True, None, None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(str(x) for x in c))
def test_backward_matches_oracle(case):
    b, sq, skv, hq, hkv, d, dts, causal, off, window = case
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dts]
    seed = _seed(case)
    q, k, v = (t.to(DEV) for t in make_custom(b, sq, skv, hq, hkv, d, dts, std=1.0, seed=seed))
    do = normal((b, sq, hq, d), seed, 7, 1.0, dt).to(DEV)
    o, lse = fa_fwd(q, k, v, causal=causal, q_pos_offset=off, window=window)
    dq, dk, dv = fa_bwd(q, k, v, o, lse, do, causal=causal, q_pos_offset=off, window=window)
    assert fa_sync_status() == 0
    rq, rk, rv = oracle.attention_bwd(f64(q), f64(k), f64(v), f64(do), causal=causal, q_pos_offset=off,
                                      scale=1.0 / math.sqrt(d), window=window if window else (-1, -1))
    what = str(case)
    _check("dQ", dq, rq, dt, what)
    _check("dK", dk, rk, dt, what)
    _check("dV", dv, rv, dt, what)


def test_backward_deterministic():
    q, k, v = (t.to(DEV) for t in make_custom(1, 700, 700, 4, 2, 128, "bf16", seed=3))
    do = normal((1, 700, 4, 128), 3, 7, 1.0, torch.bfloat16).to(DEV)
    o, lse = fa_fwd(q, k, v, causal=True)
    g1 = fa_bwd(q, k, v, o, lse, do, causal=True)
    g2 = fa_bwd(q, k, v, o, lse, do, causal=True)
    assert fa_sync_status() == 0
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_backward_no_query_rows_gives_zero_key_gradients():
    q, k, v = (t.to(DEV) for t in make_custom(1, 4, 300, 2, 2, 64, "bf16", seed=4))
    do = normal((1, 4, 2, 64), 4, 7, 1.0, torch.bfloat16).to(DEV)
    o, lse = fa_fwd(q, k, v, causal=True, q_pos_offset=-10)  # every row sees no key
    dk = torch.full_like(k, 5.0)
    dv = torch.full_like(v, 5.0)
    dq, dk, dv = fa_bwd(q, k, v, o, lse, do, causal=True, q_pos_offset=-10, dk=dk, dv=dv)
    assert fa_sync_status() == 0
    assert torch.all(dq == 0) and torch.all(dk == 0) and torch.all(dv == 0)


FULL = [
    # b, sq, hq, hkv (d = 128, bf16, causal)
    (1, 4096, 4, 4),
    (1, 2048, 32, 8),   # the long GQA workload's head ratio: 32 query heads over 8 KV heads
]


@pytest.mark.parametrize("case", FULL, ids=lambda c: "-".join(str(x) for x in c))
def test_backward_long_sequences(case):
    """Causal backward on thousands of rows, every gradient entry against the oracle."""
    b, s, hq, hkv = case
    d, dt = 128, torch.bfloat16
    seed = _seed(case)
    q, k, v = (t.to(DEV) for t in make_custom(b, s, s, hq, hkv, d, "bf16", std=1.0, seed=seed))
    do = normal((b, s, hq, d), seed, 7, 1.0, dt).to(DEV)
    o, lse = fa_fwd(q, k, v, causal=True)
    dq, dk, dv = fa_bwd(q, k, v, o, lse, do, causal=True)
    assert fa_sync_status() == 0
    rq, rk, rv = oracle.attention_bwd(f64(q), f64(k), f64(v), f64(do), causal=True, scale=1.0 / math.sqrt(d))
    what = str(case)
    _check("dQ", dq, rq, dt, what)
    _check("dK", dk, rk, dt, what)
    _check("dV", dv, rv, dt, what)


def test_backward_benchmark_workload():
    """The backward benchmark's own inputs and launch (B=4, H=16, N=4096, d=128,
    causal, upstream gradient from the same seeded stream), every entry against
    the oracle."""
    from tiled_exact_attention_gb300.inputs import BASE_SEED, WORKLOADS, make_qkv

    w = WORKLOADS["causal_prefill"]
    q, k, v = (t.to(DEV) for t in make_qkv(w))
    do = normal(tuple(q.shape), BASE_SEED + w.index, 7, 1.0, q.dtype).to(DEV)
    o, lse = fa_fwd(q, k, v, causal=True, q_pos_offset=w.offset)
    from tiled_exact_attention_gb300 import fa_bwd_workspace_size

    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa_bwd_workspace_size(q, k, v, causal=True, q_pos_offset=w.offset), dtype=torch.uint8,
                     device=DEV)
    fa_bwd(q, k, v, o, lse, do, causal=True, q_pos_offset=w.offset, dq=dq, dk=dk, dv=dv, workspace=ws)
    assert fa_sync_status() == 0
    rq, rk, rv = oracle.attention_bwd(f64(q), f64(k), f64(v), f64(do), causal=True, q_pos_offset=w.offset,
                                      scale=1.0 / math.sqrt(w.d))
    _check("dQ", dq, rq, q.dtype, "benchmark workload")
    _check("dK", dk, rk, q.dtype, "benchmark workload")
    _check("dV", dv, rv, q.dtype, "benchmark workload")
