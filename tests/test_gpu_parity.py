"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on
the same seeded inputs, element by element."""
from __future__ import annotations

import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_O, assert_parity, f64, gather, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from tiled_exact_attention_gb300 import (  # noqa: E402
    fa_fwd,
    fa_fwd_splitkv,
    fa_splitkv_combine,
    fa_splitkv_default_splits,
    fa_sync_status,
)
from tiled_exact_attention_gb300.inputs import WORKLOADS, make_custom, make_qkv  # noqa: E402

DEV = "cuda:0"


def _seed(case) -> int:
    return 1000 + zlib.crc32(repr(case).encode()) % 100000


def _cuda(*ts):
    return [t.to(DEV) for t in ts]


def _full_compare(q, k, v, causal, off, scale, o, lse, what):
    b, sq, hq, d = q.shape
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle_rows(q, k, v, causal=causal, q_pos_offset=off, scale=scale, rows=rows)
    og, lg = gather(o, lse, rows)
    return assert_parity(og, lg, o_ref, l_ref, q.dtype, what)


# ----------------------------------------------------------------------------- prefill


def test_tiny_config_full():
    w = WORKLOADS["tiny"]
    q, k, v = _cuda(*make_qkv(w))
    o, lse = fa_fwd(q, k, v, causal=w.causal)
    assert fa_sync_status() == 0
    _full_compare(q, k, v, w.causal, None, 1.0 / math.sqrt(w.d), o, lse, "tiny")


EDGE = [
    # b, sq, skv, hq, hkv, d, dtype, causal, offset
    (1, 1, 1, 1, 1, 64, "bf16", False, None),
    (1, 5, 5, 1, 1, 64, "fp16", True, None),
    (2, 63, 63, 2, 1, 64, "bf16", True, None),
    (1, 64, 65, 2, 2, 128, "bf16", False, None),
    (1, 65, 64, 4, 2, 128, "bf16", True, None),
    (1, 127, 129, 2, 2, 128, "fp16", True, None),
    (1, 128, 128, 2, 2, 128, "bf16", True, None),
    (1, 129, 257, 4, 1, 128, "bf16", True, None),
    (1, 255, 255, 2, 2, 64, "bf16", True, None),
    (2, 257, 130, 2, 2, 256, "fp16", False, None),
    (1, 200, 300, 2, 2, 256, "bf16", True, None),
    (1, 300, 300, 2, 1, 64, "fp16", True, -40),
    (1, 100, 400, 2, 2, 128, "bf16", True, 0),
    (1, 50, 80, 2, 2, 64, "bf16", True, 100),
    (1, 3, 0, 1, 1, 64, "bf16", False, None),
    (1, 520, 520, 8, 2, 128, "bf16", True, None),
    (1, 700, 650, 4, 4, 256, "fp16", True, None),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: "-".join(str(x) for x in c))
def test_edge_shapes_full(case):
    b, sq, skv, hq, hkv, d, dt, causal, off = case
    q, k, v = _cuda(*make_custom(b, sq, skv, hq, hkv, d, dt, std=1.0, seed=_seed(case)))
    o, lse = fa_fwd(q, k, v, causal=causal, q_pos_offset=off)
    assert fa_sync_status() == 0
    _full_compare(q, k, v, causal, off, 1.0 / math.sqrt(d), o, lse, str(case))


def test_ragged_n5_tile_case():
    w = WORKLOADS["ragged_n5"]
    q, k, v = _cuda(*make_qkv(w))
    o, lse = fa_fwd(q, k, v, causal=True, q_pos_offset=w.offset)
    assert fa_sync_status() == 0
    _full_compare(q, k, v, True, w.offset, 1.0 / math.sqrt(w.d), o, lse, "ragged_n5")


@pytest.mark.parametrize("name", ["causal_prefill", "ragged_d64", "ragged_d256"])
def test_full_size_every_row(name):
    """Every row of the causal-prefill and ragged-tail workloads at their full size,
    in the launch configuration the benchmark times (persistent grid, default
    tiles), against the oracle: a tile-schedule mistake that touches only a few
    (batch, head, row-block) items of the persistent scheduler cannot hide."""
    w = WORKLOADS[name]
    qc, kc, vc = make_qkv(w)
    q, k, v = _cuda(qc, kc, vc)
    o, lse = fa_fwd(q, k, v, causal=w.causal, q_pos_offset=w.offset if w.causal else None)
    assert fa_sync_status() == 0
    rows = oracle.all_rows(w.b, w.hq, w.sq)
    o_ref, l_ref = oracle_rows(qc, kc, vc, causal=w.causal, q_pos_offset=w.offset, scale=1.0 / math.sqrt(w.d),
                               rows=rows)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, qc.dtype, name)


def test_gqa_long_whole_heads():
    """The long GQA workload (B=1, Hq=32, Hkv=8, N=16384): four whole query heads
    (two sharing KV head 0, one in the middle, the last), the first 256 rows of
    every head (the row groups the longest-first schedule runs last), and a
    random sample over all heads."""
    w = WORKLOADS["gqa_long"]
    qc, kc, vc = make_qkv(w)
    q, k, v = _cuda(qc, kc, vc)
    o, lse = fa_fwd(q, k, v, causal=True, q_pos_offset=w.offset)
    assert fa_sync_status() == 0
    rows = {tuple(r) for r in sample_rows(w.b, w.hq, w.sq, n_random=256, seed=w.index)}
    for h in (0, 1, 13, w.hq - 1):
        rows.update((0, h, i) for i in range(w.sq))
    for h in range(w.hq):
        rows.update((0, h, i) for i in range(256))
    rows = np.array(sorted(rows), dtype=np.int64)
    o_ref, l_ref = oracle_rows(qc, kc, vc, causal=True, q_pos_offset=w.offset, scale=1.0 / math.sqrt(w.d),
                               rows=rows)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, qc.dtype, "gqa_long")
    # a property that holds for every row: every row sees at least its own key
    assert torch.isfinite(o).all()
    assert torch.isfinite(lse).all()


def test_permuted_layout_matches_contiguous():
    """Q/K/V stored [b, h, s, d] and passed as [b, s, h, d] views (non-default strides)."""
    q, k, v = _cuda(*make_custom(2, 300, 300, 4, 2, 128, "bf16", seed=77))
    qp = q.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    kp = k.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    vp = v.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    o1, l1 = fa_fwd(q, k, v, causal=True)
    o2, l2 = fa_fwd(qp, kp, vp, causal=True)
    assert fa_sync_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_output_only_16_byte_aligned(d):
    """An output whose base and row stride are 16- but not 32-byte aligned takes the
    16-byte store path; same result as a contiguous output."""
    b, s, h = 1, 300, 2
    q, k, v = _cuda(*make_custom(b, s, s, h, h, d, "bf16", seed=79))
    o1, l1 = fa_fwd(q, k, v, causal=True)
    row = h * d + 8  # elements: a multiple of 8 but not of 16
    buf = torch.full((b * s * row + 8,), 3.0, dtype=torch.bfloat16, device=DEV)
    o2 = buf[8:].as_strided((b, s, h, d), (s * row, row, d, 1))
    assert o2.data_ptr() % 32 == 16
    fa_fwd(q, k, v, causal=True, out=o2)
    assert fa_sync_status() == 0
    assert torch.equal(o1, o2)
    # the 8 padding elements of each row are untouched
    pad = buf[8:].view(b * s, row)[:, h * d:]
    assert torch.all(pad == 3.0)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("dts", ["bf16", "fp16"])
def test_output_with_gaps_between_heads_rows_and_batches(d, dts):
    """O written into a larger buffer with gaps after every head, row and batch
    (the tile stores address O through its strides; a 333-row sequence leaves
    store tiles partly past its end): equal to the contiguous result, and no
    element outside O is touched."""
    b, s, h = 2, 333, 3
    q, k, v = _cuda(*make_custom(b, s, s, h, h, d, dts, seed=81 + d))
    o1, l1 = fa_fwd(q, k, v, causal=True)
    sh, sr = d + 8, h * (d + 8) + 16
    sb = s * sr + 64
    buf = torch.full((b * sb,), 7.0, dtype=q.dtype, device=DEV)
    o2 = buf.as_strided((b, s, h, d), (sb, sr, sh, 1))
    fa_fwd(q, k, v, causal=True, out=o2)
    assert fa_sync_status() == 0
    assert torch.equal(o1, o2)
    mask = torch.ones_like(buf, dtype=torch.bool)
    mask.as_strided((b, s, h, d), (sb, sr, sh, 1)).fill_(False)
    assert torch.all(buf[mask] == 7.0)


def test_deterministic():
    q, k, v = _cuda(*make_custom(1, 640, 640, 4, 4, 128, "bf16", seed=5))
    o1, l1 = fa_fwd(q, k, v, causal=True)
    o2, l2 = fa_fwd(q, k, v, causal=True)
    assert fa_sync_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ----------------------------------------------------------------------------- split-KV


def test_decode_config_full():
    w = WORKLOADS["decode"]
    qc, kc, vc = make_qkv(w)
    q, k, v = _cuda(qc, kc, vc)
    o, lse, ns = fa_fwd_splitkv(q, k, v, causal=True, q_pos_offset=w.offset, return_splits=True)
    assert fa_sync_status() == 0
    assert ns == fa_splitkv_default_splits(q, k, v, causal=True, q_pos_offset=w.offset) and ns >= 1
    rows = oracle.all_rows(w.b, w.hq, w.sq)
    o_ref, l_ref = oracle_rows(qc, kc, vc, causal=True, q_pos_offset=w.offset, scale=1.0 / math.sqrt(w.d),
                               rows=rows)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, qc.dtype, "decode")


SPLIT_CASES = [
    # b, sq, skv, hq, hkv, d, dtype, causal, offset, splits
    (2, 1, 1000, 8, 2, 128, "bf16", True, 999, 1),
    (2, 1, 1000, 8, 2, 128, "bf16", True, 999, 3),
    (2, 1, 1000, 8, 2, 128, "bf16", True, 500, 7),
    (1, 1, 777, 8, 1, 64, "fp16", False, None, 5),
    (1, 1, 300, 2, 2, 256, "bf16", True, 299, 2),
    (3, 1, 129, 3, 1, 128, "bf16", False, None, 2),
    (1, 1, 200, 4, 4, 128, "bf16", True, -5, 3),
    (1, 40, 600, 4, 2, 128, "bf16", True, None, 3),
    (1, 40, 600, 4, 2, 128, "bf16", True, None, 1),
    (2, 1, 900, 16, 2, 128, "bf16", True, 600, 1),
    (2, 130, 300, 2, 2, 64, "fp16", False, None, 2),
    (1, 200, 256, 2, 1, 256, "bf16", True, None, 4),
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: "-".join(str(x) for x in c))
def test_splitkv_explicit_splits(case):
    b, sq, skv, hq, hkv, d, dt, causal, off, ns = case
    q, k, v = _cuda(*make_custom(b, sq, skv, hq, hkv, d, dt, seed=_seed(case)))
    o, lse, used = fa_fwd_splitkv(q, k, v, causal=causal, q_pos_offset=off, num_splits=ns, return_splits=True)
    assert fa_sync_status() == 0
    assert 1 <= used <= ns
    _full_compare(q, k, v, causal, off, 1.0 / math.sqrt(d), o, lse, str(case))
    # split-KV and the plain forward agree within rounding
    o2, l2 = fa_fwd(q, k, v, causal=causal, q_pos_offset=off)
    assert fa_sync_status() == 0
    fin = torch.isfinite(l2)
    assert torch.equal(fin, torch.isfinite(lse))
    assert (o.float() - o2.float()).abs().max().item() <= 2 * TOL_O[q.dtype]


def test_combine_crafted_partials():
    rng = np.random.default_rng(42)
    ns, b, hq, sq, d = 5, 2, 3, 4, 128
    op = rng.standard_normal((ns, b, hq, sq, d)).astype(np.float32)
    lp = (rng.standard_normal((ns, b, hq, sq)) * 3).astype(np.float32)
    lp[:, 0, 0, 0] = -np.inf           # a row no split contributes to
    lp[1:, 1, 2, 3] = -np.inf          # a row only split 0 contributes to
    op[1:, 1, 2, 3] = 0.0
    lp[2, 0, 1, :] = -np.inf           # one empty split for some rows
    op[2, 0, 1, :] = 0.0
    out = torch.empty((b, sq, hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((b, hq, sq), dtype=torch.float32, device=DEV)
    fa_splitkv_combine(torch.from_numpy(op).to(DEV), torch.from_numpy(lp).to(DEV), out, lse)
    assert fa_sync_status() == 0
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle.combine(op.astype(np.float64)[:, rows[:, 0], rows[:, 1], rows[:, 2]],
                                  lp.astype(np.float64)[:, rows[:, 0], rows[:, 1], rows[:, 2]])
    og, lg = gather(out, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, torch.bfloat16, "combine")


# ----------------------------------------------------------------------------- status path


def test_wait_timeout_is_reported_and_context_survives():
    from tiled_exact_attention_gb300 import fa_selftest_wait_timeout

    assert fa_sync_status() == 0
    fa_selftest_wait_timeout()
    assert fa_sync_status() == 4  # FA_ERR_TIMEOUT
    assert fa_sync_status() == 0  # cleared
    q, k, v = _cuda(*make_custom(1, 130, 130, 2, 2, 64, "bf16", seed=3))
    o, lse = fa_fwd(q, k, v)
    assert fa_sync_status() == 0
    _full_compare(q, k, v, False, None, 1 / 8.0, o, lse, "after timeout")
