"""GPU checks of the decode kernel's fused merge: the last split of each head group
to finish merges every split's partials (one atomic counter per group in the
caller's workspace, zeroed by the call itself).  Covered: a workspace full of
garbage, one workspace reused across calls with different split counts and
shapes, many splits (the merge weights of 4 heads x 64 splits in shared memory),
and agreement with the unfused combine of the same partials.
"""
from __future__ import annotations

import math

import pytest
import torch

import oracle
from parity_util import assert_parity, f64, gather

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from tiled_exact_attention_gb300 import fa_fwd_splitkv, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300.api import fa_splitkv_workspace_size  # noqa: E402
from tiled_exact_attention_gb300.inputs import make_custom  # noqa: E402

DEV = "cuda:0"


def _compare(q, k, v, o, lse, what, off=None, causal=False):
    b, sq, hq, d = q.shape
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v), causal=causal, q_pos_offset=off,
                                    scale=1.0 / math.sqrt(d), rows=rows)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, q.dtype, what)


def test_garbage_workspace():
    q, k, v = (t.to(DEV) for t in make_custom(2, 1, 3000, 8, 2, 128, "bf16", seed=41))
    need = fa_splitkv_workspace_size(q, k, v, 6)
    work = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)  # counters start at -1, partials NaN
    o, lse = fa_fwd_splitkv(q, k, v, num_splits=6, workspace=work)
    assert fa_sync_status() == 0
    _compare(q, k, v, o, lse, "garbage workspace")


def test_workspace_reused_across_calls():
    shapes = [(2, 3000, 8, 2, 128, 6), (1, 777, 4, 4, 64, 3), (3, 5000, 8, 1, 128, 11), (2, 3000, 8, 2, 128, 1)]
    biggest = 0
    inputs = []
    for i, (b, skv, hq, hkv, d, ns) in enumerate(shapes):
        q, k, v = (t.to(DEV) for t in make_custom(b, 1, skv, hq, hkv, d, "bf16", seed=50 + i))
        inputs.append((q, k, v, ns))
        biggest = max(biggest, fa_splitkv_workspace_size(q, k, v, ns))
    work = torch.empty(biggest, dtype=torch.uint8, device=DEV)
    for rep in range(2):
        for q, k, v, ns in inputs:
            o, lse = fa_fwd_splitkv(q, k, v, num_splits=ns, workspace=work)
            assert fa_sync_status() == 0
            _compare(q, k, v, o, lse, f"reuse {rep} {tuple(q.shape)} ns={ns}")


def test_many_splits():
    q, k, v = (t.to(DEV) for t in make_custom(1, 1, 20000, 8, 2, 128, "bf16", seed=77))
    o, lse, used = fa_fwd_splitkv(q, k, v, num_splits=64, return_splits=True)
    assert fa_sync_status() == 0
    assert used == 64
    _compare(q, k, v, o, lse, "64 splits")


@pytest.mark.parametrize("ns", [2, 9])
def test_fused_merge_matches_results_of_one_split(ns):
    """Splitting changes only rounding: the fused merge of ns splits against a single split."""
    q, k, v = (t.to(DEV) for t in make_custom(2, 1, 4100, 16, 4, 128, "bf16", seed=90 + ns))
    o1, l1 = fa_fwd_splitkv(q, k, v, num_splits=1)
    o2, l2 = fa_fwd_splitkv(q, k, v, num_splits=ns)
    assert fa_sync_status() == 0
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-4
