"""GPU parity of fa_fwd_kvcache (split-KV decode over a paged or packed KV cache).

The oracle runs on each sequence's keys gathered into a contiguous buffer (the
gather is plain indexing); the cache slots no sequence owns are filled with NaN,
so any read of a row past a sequence's end would show up in the result.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from tiled_exact_attention_gb300 import fa_fwd_kvcache, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300.inputs import normal  # noqa: E402

DEV = "cuda:0"
_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def _sequences(lens, hkv, d, dt, seed):
    ks = [normal((n, hkv, d), seed, 10 + 2 * i, 1.0, dt) for i, n in enumerate(lens)]
    vs = [normal((n, hkv, d), seed, 11 + 2 * i, 1.0, dt) for i, n in enumerate(lens)]
    return ks, vs


def _oracle(q, ks, vs):
    """Per sequence: the query sees all of its keys (position len - 1)."""
    b, hq, d = q.shape
    o = np.zeros((b, hq, d))
    lse = np.zeros((b, hq))
    for i in range(b):
        qi = q[i].to(torch.float64).numpy()[None, None]           # [1, 1, hq, d]
        ki = ks[i].to(torch.float64).numpy()[None]                # [1, len, hkv, d]
        vi = vs[i].to(torch.float64).numpy()[None]
        oi, li = oracle.attention(qi, ki, vi, causal=False)
        o[i], lse[i] = oi, li
    return o, lse


def _check(o_gpu, lse_gpu, o_ref, lse_ref, dt, what):
    og = o_gpu.to(torch.float64).cpu().numpy().reshape(-1, o_gpu.shape[-1])
    lg = lse_gpu.to(torch.float64).cpu().numpy().reshape(-1)
    assert_parity(og, lg, o_ref.reshape(-1, o_ref.shape[-1]), lse_ref.reshape(-1), dt, what)


PAGED = [
    # b, hq, hkv, d, dtype, page_size, lens, splits
    (3, 8, 2, 128, "bf16", 64, [1, 777, 5000], 0),
    (3, 8, 2, 128, "bf16", 256, [300, 0, 4100], 3),
    (2, 32, 8, 128, "bf16", 128, [2049, 6000], 1),
    (4, 4, 4, 64, "fp16", 128, [129, 64, 1000, 7], 0),
    (2, 8, 1, 256, "bf16", 64, [500, 1500], 2),
    # pages smaller than the 128-key block, or not a multiple of it: a block is
    # loaded as 64-row boxes from different pages
    (2, 8, 2, 128, "bf16", 192, [1000, 385], 0),
    (3, 4, 2, 64, "fp16", 64, [300, 129, 64], 2),
    (2, 8, 2, 128, "bf16", 320, [641, 1279], 3),
    # g = hq / hkv >= 8: the heads of a KV head are the rows of one tensor-core
    # tile (one and two 128-row tiles; 64-row boxes from different pages)
    (3, 16, 2, 128, "bf16", 64, [1, 777, 5000], 0),
    (3, 32, 2, 128, "fp16", 256, [300, 0, 4100], 3),
    (2, 64, 8, 128, "bf16", 128, [2049, 6000], 1),
    (2, 16, 1, 64, "bf16", 192, [1000, 385], 0),
    (2, 128, 1, 128, "bf16", 320, [641, 1279], 3),
    (1, 256, 1, 128, "bf16", 128, [3000], 0),
    (2, 16, 2, 256, "fp16", 128, [700, 2], 2),
]


@pytest.mark.parametrize("case", PAGED, ids=lambda c: "-".join(str(x) for x in c[:6]) + f"-{len(c[6])}seq-s{c[7]}")
def test_paged_cache(case):
    b, hq, hkv, d, dts, ps, lens, ns = case
    dt = _DT[dts]
    seed = 4242 + b * 7 + ps
    q = normal((b, hq, d), seed, 1, 1.0, dt)
    ks, vs = _sequences(lens, hkv, d, dt, seed)
    pages_per = [math.ceil(n / ps) for n in lens]
    num_pages = sum(pages_per) + 5
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_pages)
    k_pool = torch.full((num_pages, ps, hkv, d), float("nan"), dtype=dt)
    v_pool = torch.full((num_pages, ps, hkv, d), float("nan"), dtype=dt)
    width = max(1, max(pages_per))
    table = np.zeros((b, width), dtype=np.int32)
    nxt = 0
    for i, n in enumerate(lens):
        for pg in range(pages_per[i]):
            page = int(perm[nxt])
            nxt += 1
            table[i, pg] = page
            lo, hi = pg * ps, min(n, (pg + 1) * ps)
            k_pool[page, : hi - lo] = ks[i][lo:hi]
            v_pool[page, : hi - lo] = vs[i][lo:hi]
    o, lse, used = fa_fwd_kvcache(q.to(DEV), k_pool.to(DEV), v_pool.to(DEV),
                                  block_table=torch.from_numpy(table).to(DEV),
                                  seqlens_k=torch.tensor(lens, dtype=torch.int32, device=DEV),
                                  num_splits=ns, return_splits=True)
    assert fa_sync_status() == 0
    assert used >= 1
    o_ref, l_ref = _oracle(q, ks, vs)
    _check(o, lse, o_ref, l_ref, dt, f"paged {case}")


PACKED = [
    # b, hq, hkv, d, dtype, lens, splits
    (4, 8, 2, 128, "bf16", [5, 1000, 0, 1995], 0),
    (3, 16, 4, 128, "fp16", [4096, 63, 65], 4),
    (2, 4, 1, 64, "bf16", [1, 300], 1),
    (4, 16, 2, 128, "bf16", [5, 1000, 0, 1995], 0),
    (2, 64, 4, 64, "fp16", [4096, 63], 4),
    (2, 8, 1, 128, "bf16", [130, 1], 1),
]


@pytest.mark.parametrize("case", PACKED, ids=lambda c: "-".join(str(x) for x in c[:5]) + f"-{len(c[5])}seq-s{c[6]}")
def test_packed_varlen(case):
    b, hq, hkv, d, dts, lens, ns = case
    dt = _DT[dts]
    seed = 777 + b
    q = normal((b, hq, d), seed, 1, 1.0, dt)
    ks, vs = _sequences(lens, hkv, d, dt, seed)
    tail = torch.full((70, hkv, d), float("nan"), dtype=dt)  # rows past the last sequence
    k = torch.cat(ks + [tail])
    v = torch.cat(vs + [tail])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, lse = fa_fwd_kvcache(q.to(DEV), k.to(DEV), v.to(DEV), cu_seqlens_k=torch.from_numpy(cu).to(DEV),
                            num_splits=ns)
    assert fa_sync_status() == 0
    o_ref, l_ref = _oracle(q, ks, vs)
    _check(o, lse, o_ref, l_ref, dt, f"packed {case}")


def test_paged_matches_contiguous_decode():
    """All sequences of equal length: the paged path agrees with fa_fwd_splitkv on the same keys."""
    from tiled_exact_attention_gb300 import fa_fwd_splitkv

    b, hq, hkv, d, n, ps = 2, 8, 2, 128, 3000, 256
    dt = torch.bfloat16
    q = normal((b, 1, hq, d), 99, 1, 1.0, dt).to(DEV)
    k = normal((b, n, hkv, d), 99, 2, 1.0, dt).to(DEV)
    v = normal((b, n, hkv, d), 99, 3, 1.0, dt).to(DEV)
    o_ref, l_ref = fa_fwd_splitkv(q, k, v, causal=True, q_pos_offset=n - 1, num_splits=5)
    npg = math.ceil(n / ps)
    k_pool = torch.zeros((b * npg, ps, hkv, d), dtype=dt, device=DEV)
    v_pool = torch.zeros_like(k_pool)
    table = torch.arange(b * npg, dtype=torch.int32, device=DEV).reshape(b, npg).flip(1).contiguous()
    for i in range(b):
        for pg in range(npg):
            lo, hi = pg * ps, min(n, (pg + 1) * ps)
            k_pool[table[i, pg].item(), : hi - lo] = k[i, lo:hi]
            v_pool[table[i, pg].item(), : hi - lo] = v[i, lo:hi]
    o, lse = fa_fwd_kvcache(q[:, 0], k_pool, v_pool, block_table=table,
                            seqlens_k=torch.full((b,), n, dtype=torch.int32, device=DEV), num_splits=5)
    assert fa_sync_status() == 0
    assert (o.float() - o_ref[:, 0].float()).abs().max().item() <= 2e-2
    assert (lse - l_ref[:, :, 0]).abs().max().item() <= 1e-3



@pytest.mark.parametrize("hq,ns", [(8, 1), (8, 3), (16, 1), (16, 3)])
def test_paged_length_past_its_table_row_is_rejected_on_the_device(hq, ns):
    """A sequence length that needs more pages than its block-table row holds is
    caught by the kernels before any table read: the sequence is skipped,
    FA_ERR_DEVICE_ARG is reported, the other sequences are still computed.  (The
    table is a view into a taller allocation, so even an unchecked read past the
    row would stay inside memory the test owns.)"""
    from tiled_exact_attention_gb300._lib import FA_ERR_DEVICE_ARG

    b, hkv, d, ps, dt = 3, 2, 128, 128, torch.bfloat16
    lens = [700, 300, 500]
    width = 6  # pages per table row: 768 keys at most
    seed = 515 + hq
    q = normal((b, hq, d), seed, 1, 1.0, dt)
    ks, vs = _sequences(lens, hkv, d, dt, seed)
    num_pages = b * width + 8
    k_pool = torch.zeros((num_pages, ps, hkv, d), dtype=dt)
    v_pool = torch.zeros((num_pages, ps, hkv, d), dtype=dt)
    table_alloc = np.zeros((b + 4, width), dtype=np.int32)
    for i, n in enumerate(lens):
        for pg in range(math.ceil(n / ps)):
            page = i * width + pg
            table_alloc[i, pg] = page
            lo, hi = pg * ps, min(n, (pg + 1) * ps)
            k_pool[page, : hi - lo] = ks[i][lo:hi]
            v_pool[page, : hi - lo] = vs[i][lo:hi]
    table = torch.from_numpy(table_alloc).to(DEV)[:b]
    seqlens = torch.tensor([lens[0], width * ps + 1, lens[2]], dtype=torch.int32, device=DEV)
    assert fa_sync_status() == 0
    o, lse = fa_fwd_kvcache(q.to(DEV), k_pool.to(DEV), v_pool.to(DEV), block_table=table, seqlens_k=seqlens,
                            max_seqlen_k=max(lens), num_splits=ns)
    assert fa_sync_status() == FA_ERR_DEVICE_ARG
    assert fa_sync_status() == 0  # reported once, then cleared
    o_ref, l_ref = _oracle(q, ks, vs)
    keep = [0, 2]
    _check(o[keep], lse[keep], o_ref[keep], l_ref[keep], dt, f"paged, bad length, hq={hq} ns={ns}")


@pytest.mark.parametrize("hq", [8, 16])
def test_packed_offsets_past_the_rows_are_rejected_on_the_device(hq):
    """Packed keys whose prefix sums run past the declared rows: the sequence is
    skipped and FA_ERR_DEVICE_ARG reported; the others are still computed.  (The
    declared rows are a view of a longer tensor.)"""
    from tiled_exact_attention_gb300._lib import FA_ERR_DEVICE_ARG

    hkv, d, dt = 2, 128, torch.bfloat16
    lens = [400, 300, 1000]
    seed = 616 + hq
    q = normal((3, hq, d), seed, 1, 1.0, dt)
    ks, vs = _sequences(lens, hkv, d, dt, seed)
    k = torch.cat(ks).to(DEV)
    v = torch.cat(vs).to(DEV)
    declared = lens[0] + lens[1] + 200  # the last sequence runs 800 rows past the declared end
    cu = torch.tensor([0, lens[0], lens[0] + lens[1], sum(lens)], dtype=torch.int32, device=DEV)
    assert fa_sync_status() == 0
    o, lse = fa_fwd_kvcache(q.to(DEV), k[:declared], v[:declared], cu_seqlens_k=cu, max_seqlen_k=max(lens),
                            num_splits=2)
    assert fa_sync_status() == FA_ERR_DEVICE_ARG
    assert fa_sync_status() == 0
    o_ref, l_ref = _oracle(q, ks, vs)
    keep = [0, 1]
    _check(o[keep], lse[keep], o_ref[keep], l_ref[keep], dt, f"packed, bad offsets, hq={hq}")
