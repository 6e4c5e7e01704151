"""GPU parity of single-query decoding with many query heads per KV head, against the
fp64 oracle.  With sq == 1 and g = hq / hkv >= 8 the split-KV entry views Q as g rows
of hkv heads, so the g query heads that share a KV head fill the rows of one
tensor-core tile ("ai-reference-codex: forward CUDA kernel", 7.4; "flash attention
V2 code walkthrough", the ngroups > 1 launch).  Covered: g = 8 ... 256 (one and two
128-row tiles, a ragged second tile), d = 64 / 128 / 256, both 16-bit types, ragged
key counts, one split (the kernel writes O itself), several and the default count,
a causal offset that hides keys (and one that hides all of them), no keys at all,
softcap, a strided Q and O, and the agreement of the default split count with a
single split.
"""
from __future__ import annotations

import math
import zlib

import pytest
import torch

import oracle
from parity_util import assert_parity, f64, gather

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from tiled_exact_attention_gb300 import fa_fwd_splitkv, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300.inputs import make_custom  # noqa: E402

DEV = "cuda:0"


def _seed(case) -> int:
    return 7100 + zlib.crc32(repr(case).encode()) % 100000


def _check(q, k, v, o, lse, causal, off, softcap, what):
    b, sq, hq, d = q.shape
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v), causal=causal, q_pos_offset=off,
                                    scale=1.0 / math.sqrt(d), rows=rows, softcap=softcap)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, q.dtype, what)


CASES = [
    # b, skv, hq, hkv, d, dtype, splits, causal, offset, softcap
    (2, 3000, 16, 2, 128, "bf16", 0, False, None, 0.0),
    (1, 5000, 32, 2, 64, "fp16", 3, False, None, 0.0),
    (3, 1000, 16, 1, 256, "bf16", 0, False, None, 0.0),
    (2, 700, 64, 1, 128, "bf16", 2, True, 300, 0.0),
    (1, 2000, 256, 1, 128, "bf16", 0, False, None, 0.0),
    (1, 1500, 192, 1, 64, "fp16", 4, False, None, 0.0),
    (2, 3001, 16, 2, 128, "bf16", 5, False, None, 5.0),
    (1, 129, 8, 1, 128, "bf16", 1, True, None, 0.0),
    (2, 200, 16, 2, 128, "bf16", 2, True, -3, 0.0),
    (1, 0, 16, 2, 128, "bf16", 0, False, None, 0.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(str(x) for x in c))
def test_head_rows_decode(case):
    b, skv, hq, hkv, d, dt, ns, causal, off, c = case
    q, k, v = (t.to(DEV) for t in make_custom(b, 1, skv, hq, hkv, d, dt, seed=_seed(case)))
    o, lse = fa_fwd_splitkv(q, k, v, causal=causal, q_pos_offset=off, num_splits=ns, softcap=c)
    assert fa_sync_status() == 0
    _check(q, k, v, o, lse, causal, off, c, f"head rows {case}")


@pytest.mark.parametrize("ns", [1, 3])
def test_head_rows_strided_q_and_o(ns):
    """Q and O with a head stride of 2d and a batch stride of 3 hq d: the view's
    row and head strides come from the caller's strides, not from d."""
    b, skv, hq, hkv, d = 2, 1100, 32, 4, 128
    q0, k, v = make_custom(b, 1, skv, hq, hkv, d, "bf16", seed=4242)
    qbig = torch.zeros((b, 3, hq, 2 * d), dtype=q0.dtype)
    qbig[:, 1, :, :d] = q0[:, 0]
    q = qbig.to(DEV)[:, 1:2, :, :d]
    obig = torch.full((b, 3, hq, 2 * d), float("nan"), dtype=q0.dtype, device=DEV)
    o = obig[:, 1:2, :, :d]
    lse = torch.empty((b, hq, 1), dtype=torch.float32, device=DEV)
    k, v = k.to(DEV), v.to(DEV)
    fa_fwd_splitkv(q, k, v, num_splits=ns, out=o, lse=lse)
    assert fa_sync_status() == 0
    _check(q, k, v, o, lse, False, None, 0.0, f"strided head rows, {ns} splits")
    assert torch.isnan(obig[:, 0]).all() and torch.isnan(obig[:, 2]).all() and torch.isnan(obig[..., d:]).all()


def test_head_rows_default_splits_match_one_split():
    q, k, v = (t.to(DEV) for t in make_custom(4, 1, 9000, 64, 8, 128, "bf16", seed=31))
    o1, l1 = fa_fwd_splitkv(q, k, v, num_splits=1)
    o2, l2, used = fa_fwd_splitkv(q, k, v, return_splits=True)
    assert fa_sync_status() == 0
    assert used >= 1
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-4
