"""Seeded random shapes for single-query decoding against the fp64 oracle: the
split-KV entry and the KV-cache entry (paged and packed), with group sizes that
are not powers of two (g = 12, 24, 40) next to the usual ones, every head
dimension, both 16-bit types, causal offsets, split counts and page sizes drawn
from a fixed seed.  Group sizes of 8 and more take the heads-as-rows tile, the
others the CUDA-core decode kernel; both must agree with the oracle.
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

from tiled_exact_attention_gb300 import fa_fwd_kvcache, fa_fwd_splitkv, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300.inputs import make_custom, normal  # noqa: E402

DEV = "cuda:0"
_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}
GROUPS = [1, 2, 4, 8, 12, 16, 24, 40, 64, 128]


def _draw_splitkv(i):
    rng = np.random.default_rng(9000 + i)
    g = int(rng.choice(GROUPS))
    hkv = int(rng.integers(1, 4))
    d = int(rng.choice([64, 128, 256]))
    b = int(rng.integers(1, 4))
    skv = int(rng.integers(0, 3000))
    causal = bool(rng.integers(0, 2))
    off = int(rng.integers(-5, skv + 5)) if causal and skv > 0 else None
    ns = int(rng.choice([0, 0, 1, 2, 5]))
    dt = str(rng.choice(["bf16", "fp16"]))
    return b, skv, g * hkv, hkv, d, dt, causal, off, ns


@pytest.mark.parametrize("i", range(24))
def test_splitkv_decode_random(i):
    b, skv, hq, hkv, d, dt, causal, off, ns = _draw_splitkv(i)
    q, k, v = (t.to(DEV) for t in make_custom(b, 1, skv, hq, hkv, d, dt, seed=9100 + i))
    o, lse = fa_fwd_splitkv(q, k, v, causal=causal, q_pos_offset=off, num_splits=ns)
    assert fa_sync_status() == 0
    rows = oracle.all_rows(b, hq, 1)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v), causal=causal, q_pos_offset=off,
                                    scale=1.0 / math.sqrt(d), rows=rows)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, q.dtype, f"random split-KV decode {i}: {(b, skv, hq, hkv, d, dt, causal, off, ns)}")


@pytest.mark.parametrize("i", range(16))
def test_kvcache_decode_random(i):
    rng = np.random.default_rng(9500 + i)
    g = int(rng.choice(GROUPS))
    hkv = int(rng.integers(1, 3))
    hq = g * hkv
    d = int(rng.choice([64, 128, 256]))
    b = int(rng.integers(1, 4))
    lens = [int(x) for x in rng.integers(0, 2500, size=b)]
    paged = bool(rng.integers(0, 2))
    ps = int(rng.choice([64, 128, 192, 256]))
    ns = int(rng.choice([0, 1, 3]))
    dt = _DT[str(rng.choice(["bf16", "fp16"]))]
    seed = 9600 + i
    q = normal((b, hq, d), seed, 1, 1.0, dt)
    ks = [normal((n, hkv, d), seed, 10 + 2 * j, 1.0, dt) for j, n in enumerate(lens)]
    vs = [normal((n, hkv, d), seed, 11 + 2 * j, 1.0, dt) for j, n in enumerate(lens)]
    if paged:
        pages_per = [math.ceil(n / ps) for n in lens]
        num_pages = sum(pages_per) + 2
        perm = rng.permutation(num_pages)
        k_pool = torch.full((num_pages, ps, hkv, d), float("nan"), dtype=dt)
        v_pool = torch.full((num_pages, ps, hkv, d), float("nan"), dtype=dt)
        table = np.zeros((b, max(1, max(pages_per))), dtype=np.int32)
        nxt = 0
        for j, n in enumerate(lens):
            for pg in range(pages_per[j]):
                page = int(perm[nxt])
                nxt += 1
                table[j, pg] = page
                lo, hi = pg * ps, min(n, (pg + 1) * ps)
                k_pool[page, : hi - lo] = ks[j][lo:hi]
                v_pool[page, : hi - lo] = vs[j][lo:hi]
        o, lse = fa_fwd_kvcache(q.to(DEV), k_pool.to(DEV), v_pool.to(DEV), block_table=torch.from_numpy(table).to(DEV),
                                seqlens_k=torch.tensor(lens, dtype=torch.int32, device=DEV), num_splits=ns)
    else:
        tail = torch.full((40, hkv, d), float("nan"), dtype=dt)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        o, lse = fa_fwd_kvcache(q.to(DEV), torch.cat(ks + [tail]).to(DEV), torch.cat(vs + [tail]).to(DEV),
                                cu_seqlens_k=torch.from_numpy(cu).to(DEV), num_splits=ns)
    assert fa_sync_status() == 0
    o_ref = np.zeros((b, hq, d))
    l_ref = np.zeros((b, hq))
    for j, n in enumerate(lens):
        oj, lj = oracle.attention(f64(q[j])[None, None], f64(ks[j])[None], f64(vs[j])[None], causal=False)
        o_ref[j], l_ref[j] = oj, lj
    assert_parity(o.to(torch.float64).cpu().numpy().reshape(-1, d), lse.cpu().double().numpy().reshape(-1),
                  o_ref.reshape(-1, d), l_ref.reshape(-1), dt,
                  f"random KV cache {i}: b={b} hq={hq} hkv={hkv} d={d} paged={paged} ps={ps} lens={lens} ns={ns}")
