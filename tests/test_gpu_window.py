"""GPU parity of the sliding-window (local) mask against the fp64 oracle.

Query i sees keys [i + offset - left, i + offset + right] ("flash attention V2
code walkthrough", Is_local), -1 leaving a side open; with causal set as well
the right edge is at most the diagonal.  Covered: the prefill kernel (whole
output compared), the split-KV path, the decode kernel (sq == 1) and the
KV-cache decode with a left window.
"""
from __future__ import annotations

import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_parity, f64, gather

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from tiled_exact_attention_gb300 import fa_fwd, fa_fwd_kvcache, fa_fwd_splitkv, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300.inputs import make_custom, normal  # noqa: E402

DEV = "cuda:0"
_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def _seed(case) -> int:
    return 5000 + zlib.crc32(repr(case).encode()) % 100000


def _compare_all(q, k, v, causal, off, window, o, lse, what):
    b, sq, hq, d = q.shape
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v), causal=causal, q_pos_offset=off,
                                    scale=1.0 / math.sqrt(d), rows=rows, window=window)
    og, lg = gather(o, lse, rows)
    return assert_parity(og, lg, o_ref, l_ref, q.dtype, what)


WINDOWS = [
    # b, sq, skv, hq, hkv, d, dtype, causal, offset, (left, right)
    (1, 300, 300, 2, 1, 128, "bf16", False, None, (64, 0)),
    (1, 513, 513, 4, 2, 128, "bf16", False, None, (100, 100)),
    (2, 257, 400, 2, 2, 64, "fp16", False, None, (0, 0)),
    (1, 700, 700, 2, 2, 256, "bf16", True, None, (200, 50)),
    (1, 129, 1000, 2, 1, 128, "bf16", False, None, (-1, 30)),
    (1, 400, 400, 2, 2, 128, "fp16", False, None, (130, -1)),
    (1, 300, 300, 2, 2, 64, "bf16", False, -200, (50, 20)),
    (1, 200, 100, 2, 2, 128, "bf16", False, 50, (10, 10)),
    (1, 260, 260, 2, 2, 128, "bf16", False, None, (5000, 5000)),
    (1, 1030, 1030, 2, 1, 128, "bf16", False, None, (255, 0)),
    (1, 640, 640, 2, 2, 256, "fp16", False, None, (63, 64)),
]


@pytest.mark.parametrize("case", WINDOWS, ids=lambda c: "-".join(str(x) for x in c))
def test_prefill_window_full(case):
    b, sq, skv, hq, hkv, d, dt, causal, off, window = case
    q, k, v = (t.to(DEV) for t in make_custom(b, sq, skv, hq, hkv, d, dt, std=1.0, seed=_seed(case)))
    o, lse = fa_fwd(q, k, v, causal=causal, q_pos_offset=off, window=window)
    assert fa_sync_status() == 0
    _compare_all(q, k, v, causal, off, window, o, lse, str(case))


@pytest.mark.parametrize("case", [WINDOWS[1], WINDOWS[3], WINDOWS[6], WINDOWS[9]],
                         ids=lambda c: "-".join(str(x) for x in c))
@pytest.mark.parametrize("splits", [2, 5])
def test_splitkv_window_full(case, splits):
    b, sq, skv, hq, hkv, d, dt, causal, off, window = case
    q, k, v = (t.to(DEV) for t in make_custom(b, sq, skv, hq, hkv, d, dt, std=1.0, seed=_seed(case)))
    o, lse = fa_fwd_splitkv(q, k, v, causal=causal, q_pos_offset=off, window=window, num_splits=splits)
    assert fa_sync_status() == 0
    _compare_all(q, k, v, causal, off, window, o, lse, f"split{splits} {case}")


def test_window_open_right_zero_equals_causal_bitwise():
    q, k, v = (t.to(DEV) for t in make_custom(1, 777, 777, 4, 2, 128, "bf16", seed=31))
    o1, l1 = fa_fwd(q, k, v, causal=True)
    o2, l2 = fa_fwd(q, k, v, window=(-1, 0))
    assert fa_sync_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


DECODE = [
    # b, skv, hq, hkv, d, dtype, (left, right), splits
    (2, 5000, 8, 2, 128, "bf16", (1000, 0), 0),
    (2, 5000, 8, 2, 128, "bf16", (1000, 0), 4),
    (3, 3000, 4, 4, 64, "fp16", (300, -1), 0),
    (1, 2000, 8, 1, 256, "bf16", (0, 0), 0),
    (2, 700, 8, 2, 128, "bf16", (63, 0), 3),
    # g = 16: a window keeps the CUDA-core decode kernel; one wider than the keys is
    # dropped and the heads-as-rows tile takes the call
    (2, 3000, 32, 2, 128, "bf16", (500, 0), 0),
    (1, 1000, 16, 2, 128, "bf16", (5000, 0), 0),
]


@pytest.mark.parametrize("case", DECODE, ids=lambda c: "-".join(str(x) for x in c))
def test_decode_window(case):
    b, skv, hq, hkv, d, dt, window, ns = case
    q, k, v = (t.to(DEV) for t in make_custom(b, 1, skv, hq, hkv, d, dt, std=1.0, seed=_seed(case)))
    o, lse = fa_fwd_splitkv(q, k, v, window=window, num_splits=ns)
    assert fa_sync_status() == 0
    _compare_all(q, k, v, False, None, window, o, lse, f"decode {case}")


def test_kvcache_paged_window_skips_old_keys():
    """Paged cache with a left window: every key before the window is NaN in the
    pool, so a read of one would show up in the result."""
    b, hq, hkv, d, ps, wl = 3, 8, 2, 128, 64, 200
    lens = [150, 1000, 2345]
    dt = torch.bfloat16
    seed = 90210
    q = normal((b, hq, d), seed, 1, 1.0, dt)
    ks = [normal((n, hkv, d), seed, 10 + 2 * i, 1.0, dt) for i, n in enumerate(lens)]
    vs = [normal((n, hkv, d), seed, 11 + 2 * i, 1.0, dt) for i, n in enumerate(lens)]
    pages_per = [math.ceil(n / ps) for n in lens]
    num_pages = sum(pages_per) + 2
    perm = np.random.default_rng(seed).permutation(num_pages)
    k_pool = torch.full((num_pages, ps, hkv, d), float("nan"), dtype=dt)
    v_pool = torch.full((num_pages, ps, hkv, d), float("nan"), dtype=dt)
    table = np.zeros((b, max(pages_per)), dtype=np.int32)
    nxt = 0
    for i, n in enumerate(lens):
        start = max(0, n - 1 - wl)
        for pg in range(pages_per[i]):
            page = int(perm[nxt])
            nxt += 1
            table[i, pg] = page
            lo, hi = pg * ps, min(n, (pg + 1) * ps)
            for src, pool in ((ks[i], k_pool), (vs[i], v_pool)):
                pool[page, : hi - lo] = src[lo:hi]
                if lo < start:  # keys before the window: NaN
                    pool[page, : min(hi, start) - lo] = float("nan")
    o, lse = fa_fwd_kvcache(q.to(DEV), k_pool.to(DEV), v_pool.to(DEV), block_table=torch.from_numpy(table).to(DEV),
                            seqlens_k=torch.tensor(lens, dtype=torch.int32, device=DEV), window_left=wl)
    assert fa_sync_status() == 0
    o_ref = np.zeros((b, hq, d))
    l_ref = np.zeros((b, hq))
    for i, n in enumerate(lens):
        oi, li = oracle.attention(f64(q[i])[None, None], f64(ks[i])[None], f64(vs[i])[None], causal=False,
                                  q_pos_offset=n - 1, window=(wl, -1))
        o_ref[i], l_ref[i] = oi, li
    assert_parity(o.to(torch.float64).cpu().numpy().reshape(-1, d), lse.cpu().double().numpy().reshape(-1),
                  o_ref.reshape(-1, d), l_ref.reshape(-1), dt, "paged window")


def test_kvcache_packed_window():
    b, hq, hkv, d, wl = 3, 4, 1, 64, 100
    lens = [50, 101, 900]
    dt = torch.float16
    seed = 4711
    q = normal((b, hq, d), seed, 1, 1.0, dt)
    ks = [normal((n, hkv, d), seed, 10 + 2 * i, 1.0, dt) for i, n in enumerate(lens)]
    vs = [normal((n, hkv, d), seed, 11 + 2 * i, 1.0, dt) for i, n in enumerate(lens)]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, lse = fa_fwd_kvcache(q.to(DEV), torch.cat(ks).to(DEV), torch.cat(vs).to(DEV),
                            cu_seqlens_k=torch.from_numpy(cu).to(DEV), window_left=wl, num_splits=2)
    assert fa_sync_status() == 0
    o_ref = np.zeros((b, hq, d))
    l_ref = np.zeros((b, hq))
    for i, n in enumerate(lens):
        oi, li = oracle.attention(f64(q[i])[None, None], f64(ks[i])[None], f64(vs[i])[None], causal=False,
                                  q_pos_offset=n - 1, window=(wl, -1))
        o_ref[i], l_ref[i] = oi, li
    assert_parity(o.to(torch.float64).cpu().numpy().reshape(-1, d), lse.cpu().double().numpy().reshape(-1),
                  o_ref.reshape(-1, d), l_ref.reshape(-1), dt, "packed window")
