"""GPU parity of the softcap variant (every scaled score s capped to c * tanh(s / c),
the reading of the walkthrough's Is_softcap flag) against the fp64 oracle: the
prefill kernel (whole output), the split-KV path (prefill and decode kernels),
the KV-cache decode (paged and packed), packed variable-length sequences and
the backward pass.  Q and K have std 2, so that scaled scores reach well past the
caps used (|s| up to ~12 against c = 3 and c = 8): the cap changes the result; V
keeps std 1 (the 16-bit tolerances scale with |V|).
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

from tiled_exact_attention_gb300 import (  # noqa: E402
    fa_bwd, fa_fwd, fa_fwd_kvcache, fa_fwd_splitkv, fa_fwd_varlen, fa_sync_status)
from tiled_exact_attention_gb300.inputs import make_custom, normal  # noqa: E402

DEV = "cuda:0"
_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}
STD = 2.0


def _qkv(b, sq, skv, hq, hkv, d, dt, seed):
    q, k, v = make_custom(b, sq, skv, hq, hkv, d, dt, std=STD, seed=seed)
    return q.to(DEV), k.to(DEV), (v / STD).to(DEV)  # (halving is exact in bf16 / fp16)


def _seed(case) -> int:
    return 3100 + zlib.crc32(repr(case).encode()) % 100000


def _compare_all(q, k, v, causal, off, window, c, o, lse, what):
    b, sq, hq, d = q.shape
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v), causal=causal, q_pos_offset=off,
                                    scale=1.0 / math.sqrt(d), rows=rows, window=window or (-1, -1), softcap=c)
    og, lg = gather(o, lse, rows)
    return assert_parity(og, lg, o_ref, l_ref, q.dtype, what)


PREFILL = [
    # b, sq, skv, hq, hkv, d, dtype, causal, offset, window, softcap
    (1, 300, 300, 2, 1, 128, "bf16", True, None, None, 3.0),
    (2, 257, 400, 4, 2, 64, "fp16", False, None, None, 8.0),
    (1, 700, 700, 2, 2, 256, "bf16", True, None, None, 8.0),
    (1, 513, 513, 2, 2, 128, "bf16", False, None, (100, 100), 3.0),
    (1, 129, 1000, 2, 1, 128, "fp16", True, 500, None, 50.0),
]


@pytest.mark.parametrize("case", PREFILL, ids=lambda c: "-".join(str(x) for x in c))
def test_prefill_softcap(case):
    b, sq, skv, hq, hkv, d, dt, causal, off, window, c = case
    q, k, v = _qkv(b, sq, skv, hq, hkv, d, dt, _seed(case))
    o, lse = fa_fwd(q, k, v, causal=causal, q_pos_offset=off, window=window, softcap=c)
    assert fa_sync_status() == 0
    _compare_all(q, k, v, causal, off, window, c, o, lse, str(case))


def test_softcap_changes_the_result():
    """The same call without the cap differs by far more than the tolerance (the cap is live)."""
    q, k, v = _qkv(1, 256, 256, 2, 2, 128, "bf16", 12)
    o1, l1 = fa_fwd(q, k, v, causal=True, softcap=3.0)
    o2, l2 = fa_fwd(q, k, v, causal=True)
    assert fa_sync_status() == 0
    assert (l1 - l2).abs().max().item() > 1.0


@pytest.mark.parametrize("case", [PREFILL[0], PREFILL[3]], ids=lambda c: "-".join(str(x) for x in c))
@pytest.mark.parametrize("splits", [3])
def test_splitkv_prefill_softcap(case, splits):
    b, sq, skv, hq, hkv, d, dt, causal, off, window, c = case
    q, k, v = _qkv(b, sq, skv, hq, hkv, d, dt, _seed(case))
    o, lse = fa_fwd_splitkv(q, k, v, causal=causal, q_pos_offset=off, window=window, num_splits=splits, softcap=c)
    assert fa_sync_status() == 0
    _compare_all(q, k, v, causal, off, window, c, o, lse, f"split{splits} {case}")


DECODE = [
    # b, skv, hq, hkv, d, dtype, splits, softcap
    (2, 5000, 8, 2, 128, "bf16", 0, 3.0),
    (3, 3000, 4, 4, 64, "fp16", 4, 8.0),
    (1, 2000, 8, 1, 256, "bf16", 0, 30.0),
]


@pytest.mark.parametrize("case", DECODE, ids=lambda c: "-".join(str(x) for x in c))
def test_decode_softcap(case):
    b, skv, hq, hkv, d, dt, ns, c = case
    q, k, v = _qkv(b, 1, skv, hq, hkv, d, dt, _seed(case))
    o, lse = fa_fwd_splitkv(q, k, v, num_splits=ns, softcap=c)
    assert fa_sync_status() == 0
    _compare_all(q, k, v, False, None, None, c, o, lse, f"decode {case}")


@pytest.mark.parametrize("hq", [8, 32])
@pytest.mark.parametrize("paged", [True, False])
def test_kvcache_softcap(paged, hq):
    b, hkv, d, ps, c = 3, 2, 128, 128, 5.0
    lens = [1, 700, 2345]
    dt = torch.bfloat16
    seed = 2718 + int(paged) + hq
    q = normal((b, hq, d), seed, 1, STD, dt)
    ks = [normal((n, hkv, d), seed, 10 + 2 * i, STD, dt) for i, n in enumerate(lens)]
    vs = [normal((n, hkv, d), seed, 11 + 2 * i, 1.0, dt) for i, n in enumerate(lens)]
    if paged:
        pages_per = [math.ceil(n / ps) for n in lens]
        num_pages = sum(pages_per) + 1
        perm = np.random.default_rng(seed).permutation(num_pages)
        k_pool = torch.full((num_pages, ps, hkv, d), float("nan"), dtype=dt)
        v_pool = torch.full((num_pages, ps, hkv, d), float("nan"), dtype=dt)
        table = np.zeros((b, max(pages_per)), dtype=np.int32)
        nxt = 0
        for i, n in enumerate(lens):
            for pg in range(pages_per[i]):
                page = int(perm[nxt])
                nxt += 1
                table[i, pg] = page
                lo, hi = pg * ps, min(n, (pg + 1) * ps)
                k_pool[page, : hi - lo] = ks[i][lo:hi]
                v_pool[page, : hi - lo] = vs[i][lo:hi]
        o, lse = fa_fwd_kvcache(q.to(DEV), k_pool.to(DEV), v_pool.to(DEV),
                                block_table=torch.from_numpy(table).to(DEV),
                                seqlens_k=torch.tensor(lens, dtype=torch.int32, device=DEV), softcap=c)
    else:
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        o, lse = fa_fwd_kvcache(q.to(DEV), torch.cat(ks).to(DEV), torch.cat(vs).to(DEV),
                                cu_seqlens_k=torch.from_numpy(cu).to(DEV), num_splits=2, softcap=c)
    assert fa_sync_status() == 0
    o_ref = np.zeros((b, hq, d))
    l_ref = np.zeros((b, hq))
    for i, n in enumerate(lens):
        oi, li = oracle.attention(f64(q[i])[None, None], f64(ks[i])[None], f64(vs[i])[None], causal=False,
                                  softcap=c)
        o_ref[i], l_ref[i] = oi, li
    assert_parity(o.to(torch.float64).cpu().numpy().reshape(-1, d), lse.cpu().double().numpy().reshape(-1),
                  o_ref.reshape(-1, d), l_ref.reshape(-1), dt, f"kvcache softcap paged={paged} hq={hq}")


def test_varlen_softcap():
    lens_q, lens_k, hq, hkv, d, c = [1, 300, 200], [1, 300, 700], 4, 2, 128, 4.0
    dt = torch.bfloat16
    seed = 99
    q = normal((sum(lens_q), hq, d), seed, 0, STD, dt)
    k = normal((sum(lens_k), hkv, d), seed, 1, STD, dt)
    v = normal((sum(lens_k), hkv, d), seed, 2, 1.0, dt)
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    o, lse = fa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(cu_q).to(DEV),
                           torch.from_numpy(cu_k).to(DEV), causal=True, softcap=c)
    assert fa_sync_status() == 0
    for s in range(len(lens_q)):
        q0, q1, k0, k1 = int(cu_q[s]), int(cu_q[s + 1]), int(cu_k[s]), int(cu_k[s + 1])
        o_ref, l_ref = oracle.attention(f64(q[q0:q1])[None], f64(k[k0:k1])[None], f64(v[k0:k1])[None],
                                        causal=True, scale=1.0 / math.sqrt(d), softcap=c)
        og = o[q0:q1].permute(1, 0, 2).reshape(-1, d).to(torch.float64).cpu().numpy()
        lg = lse[:, q0:q1].reshape(-1).to(torch.float64).cpu().numpy()
        assert_parity(og, lg, o_ref, l_ref, dt, f"varlen softcap seq {s}")


BWD = [
    # b, sq, skv, hq, hkv, d, dtype, causal, softcap
    (1, 300, 300, 4, 2, 128, "bf16", True, 3.0),
    (2, 257, 130, 2, 1, 128, "fp16", False, 8.0),
    (1, 200, 400, 2, 2, 64, "bf16", True, 5.0),
]
TOL_REL = {torch.bfloat16: 1e-2, torch.float16: 2e-3}


@pytest.mark.parametrize("case", BWD, ids=lambda c: "-".join(str(x) for x in c))
def test_backward_softcap(case):
    b, sq, skv, hq, hkv, d, dts, causal, c = case
    dt = _DT[dts]
    seed = _seed(case)
    q, k, v = _qkv(b, sq, skv, hq, hkv, d, dts, seed)
    do = normal((b, sq, hq, d), seed, 7, 1.0, dt).to(DEV)
    o, lse = fa_fwd(q, k, v, causal=causal, softcap=c)
    dq, dk, dv = fa_bwd(q, k, v, o, lse, do, causal=causal, softcap=c)
    assert fa_sync_status() == 0
    refs = oracle.attention_bwd(f64(q), f64(k), f64(v), f64(do), causal=causal, scale=1.0 / math.sqrt(d),
                                softcap=c)
    for name, got, ref in (("dQ", dq, refs[0]), ("dK", dk, refs[1]), ("dV", dv, refs[2])):
        g = got.to(torch.float64).cpu().numpy()
        scale = max(np.abs(ref).max(), 1e-6)
        err = np.abs(g - ref).max()
        assert err <= TOL_REL[dt] * scale, f"{case}: {name} max|diff| {err:.3e} > {TOL_REL[dt]} * {scale:.3e}"
