"""GPU parity of fa_fwd_varlen (packed variable-length sequences) against the
fp64 oracle, run on each sequence on its own (the slices are plain indexing).

Rows of the packed tensors that no sequence owns (before cu_seqlens[0] and
after cu_seqlens[b]) hold a sentinel in the output, which must survive: the
last tile of a sequence must not write into the rows that follow it.
"""
from __future__ import annotations

import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_parity, f64

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from tiled_exact_attention_gb300 import fa_fwd, fa_fwd_varlen, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300._lib import FA_ERR_DEVICE_ARG  # noqa: E402
from tiled_exact_attention_gb300.inputs import normal  # noqa: E402

DEV = "cuda:0"
_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}
SENTINEL = 7.0


def _seed(case) -> int:
    return 7000 + zlib.crc32(repr(case).encode()) % 100000


def _packed(lens_q, lens_k, hq, hkv, d, dt, seed, lead=0, trail=0):
    """Packed Q/K/V with `lead` unowned rows before the first sequence and `trail` after the last."""
    tq = lead + sum(lens_q) + trail
    tk = lead + sum(lens_k) + trail
    q = normal((tq, hq, d), seed, 0, 1.0, dt)
    k = normal((tk, hkv, d), seed, 1, 1.0, dt)
    v = normal((tk, hkv, d), seed, 2, 1.0, dt)
    cu_q = (lead + np.concatenate([[0], np.cumsum(lens_q)])).astype(np.int32)
    cu_k = (lead + np.concatenate([[0], np.cumsum(lens_k)])).astype(np.int32)
    return q, k, v, cu_q, cu_k


def _check(q, k, v, cu_q, cu_k, o, lse, causal, window, dt, what):
    d = q.shape[2]
    for s in range(len(cu_q) - 1):
        q0, q1, k0, k1 = int(cu_q[s]), int(cu_q[s + 1]), int(cu_k[s]), int(cu_k[s + 1])
        if q1 == q0:
            continue
        o_ref, l_ref = oracle.attention(f64(q[q0:q1])[None], f64(k[k0:k1])[None], f64(v[k0:k1])[None],
                                        causal=causal, scale=1.0 / math.sqrt(d),
                                        window=window if window is not None else (-1, -1))
        # oracle rows are ordered (head, query); gather the GPU rows the same way
        og = o[q0:q1].permute(1, 0, 2).reshape(-1, d).to(torch.float64).cpu().numpy()
        lg = lse[:, q0:q1].reshape(-1).to(torch.float64).cpu().numpy()
        assert_parity(og, lg, o_ref, l_ref, dt, f"{what} seq {s}")
    # unowned rows keep the sentinel
    lo, hi = int(cu_q[0]), int(cu_q[-1])
    for rows in (slice(0, lo), slice(hi, o.shape[0])):
        assert torch.all(o[rows] == SENTINEL), f"{what}: rows outside every sequence were written"
        assert torch.all(lse[:, rows] == SENTINEL)


CASES = [
    # lens_q, lens_k, hq, hkv, d, dtype, causal, window, lead, trail
    ([1, 300, 0, 513], [1, 300, 50, 600], 4, 2, 128, "bf16", True, None, 0, 0),
    ([129, 1, 257], [5, 700, 0], 2, 2, 64, "fp16", False, None, 3, 40),
    ([200, 77], [100, 400], 2, 1, 128, "bf16", True, None, 0, 130),
    ([640, 5, 300], [640, 800, 300], 2, 2, 256, "bf16", True, (100, -1), 16, 1),
    ([384, 256, 130], [384, 256, 2000], 4, 4, 128, "fp16", False, (64, 64), 0, 0),
    ([1000], [1000], 2, 1, 128, "bf16", True, None, 0, 0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{len(c[0])}seq-d{c[4]}-{c[5]}-c{int(c[6])}-w{c[7]}")
def test_varlen_matches_oracle_per_sequence(case):
    lens_q, lens_k, hq, hkv, d, dts, causal, window, lead, trail = case
    dt = _DT[dts]
    q, k, v, cu_q, cu_k = _packed(lens_q, lens_k, hq, hkv, d, dt, _seed(case), lead, trail)
    o = torch.full(q.shape, SENTINEL, dtype=dt, device=DEV)
    lse = torch.full((hq, q.shape[0]), SENTINEL, dtype=torch.float32, device=DEV)
    fa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(cu_q).to(DEV), torch.from_numpy(cu_k).to(DEV),
                  causal=causal, window=window, out=o, lse=lse)
    assert fa_sync_status() == 0
    _check(q, k, v, cu_q, cu_k, o, lse, causal, window, dt, str(case))


def test_varlen_equal_lengths_match_dense_batch():
    """All sequences of one length: the packed call equals fa_fwd on the [b, s, h, d] batch."""
    b, s, hq, hkv, d = 3, 700, 4, 2, 128
    q = normal((b, s, hq, d), 5, 0, 1.0, torch.bfloat16).to(DEV)
    k = normal((b, s, hkv, d), 5, 1, 1.0, torch.bfloat16).to(DEV)
    v = normal((b, s, hkv, d), 5, 2, 1.0, torch.bfloat16).to(DEV)
    o_d, l_d = fa_fwd(q, k, v, causal=True)
    cu = torch.arange(0, (b + 1) * s, s, dtype=torch.int32, device=DEV)
    o_v, l_v = fa_fwd_varlen(q.reshape(b * s, hq, d), k.reshape(b * s, hkv, d), v.reshape(b * s, hkv, d), cu, cu,
                             causal=True)
    assert fa_sync_status() == 0
    assert torch.equal(o_v.reshape(b, s, hq, d), o_d)
    assert torch.equal(l_v.reshape(hq, b, s).permute(1, 0, 2), l_d)


@pytest.mark.parametrize("bad", ["past_total", "decreasing", "longer_than_max"])
def test_varlen_bad_offsets_are_reported_not_followed(bad):
    """Offsets the host cannot see are checked on the device: the bad sequence is
    skipped, FA_ERR_DEVICE_ARG is reported, the good one is still computed."""
    hq, hkv, d, dt = 2, 2, 128, torch.bfloat16
    q, k, v, cu_q, cu_k = _packed([100, 150], [100, 150], hq, hkv, d, dt, 11)
    max_q = 150
    if bad == "past_total":
        cu_q = np.array([0, 100, 400], dtype=np.int32)
    elif bad == "decreasing":
        cu_k = np.array([0, 100, 50], dtype=np.int32)
    else:
        max_q = 120
    o = torch.full(q.shape, SENTINEL, dtype=dt, device=DEV)
    lse = torch.full((hq, q.shape[0]), SENTINEL, dtype=torch.float32, device=DEV)
    fa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(cu_q).to(DEV), torch.from_numpy(cu_k).to(DEV),
                  max_seqlen_q=max_q, causal=True, out=o, lse=lse)
    assert fa_sync_status() == FA_ERR_DEVICE_ARG
    assert fa_sync_status() == 0  # the record is cleared
    # the first sequence is intact and correct
    o_ref, l_ref = oracle.attention(f64(q[:100])[None], f64(k[:100])[None], f64(v[:100])[None], causal=True)
    og = o[:100].permute(1, 0, 2).reshape(-1, d).to(torch.float64).cpu().numpy()
    lg = lse[:, :100].reshape(-1).to(torch.float64).cpu().numpy()
    assert_parity(og, lg, o_ref, l_ref, dt, bad)
    # the rejected sequence was not written
    assert torch.all(o[100:] == SENTINEL)
