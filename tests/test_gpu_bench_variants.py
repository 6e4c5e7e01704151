"""GPU parity of the benchmark's variant lines at their full sizes, on the very
inputs and calls bench.py times: the sliding window (1024, 0) and the softcap 30
on the causal prefill workload (B=4, H=16, N=4096, d=128), the 16 packed causal
sequences (lengths 256-4096), and the split-KV decode with 8 query heads per KV
head (B=8, Hq=64, Hkv=8, KV=32768, the heads-as-rows tensor-core path).  Each is
compared with the fp64 oracle on whole heads or sequences and on a row sample
that includes the tile edges.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_parity, f64, gather, sample_rows

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from tiled_exact_attention_gb300 import fa_fwd, fa_fwd_splitkv, fa_fwd_varlen, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300.inputs import BASE_SEED, WORKLOADS, make_custom, make_qkv, normal  # noqa: E402

DEV = "cuda:0"


def _rows(w):
    rows = {tuple(r) for r in sample_rows(w.b, w.hq, w.sq, n_random=256, seed=w.index)}
    rows.update((w.b - 1, w.hq // 2, i) for i in range(w.sq))
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("variant", ["window", "softcap"])
def test_prefill_variant_full_size(variant):
    w = WORKLOADS["causal_prefill"]
    qc, kc, vc = make_qkv(w)
    q, k, v = (t.to(DEV) for t in (qc, kc, vc))
    window = (1024, 0) if variant == "window" else None
    c = 30.0 if variant == "softcap" else 0.0
    o, lse = fa_fwd(q, k, v, causal=True, window=window, softcap=c)
    assert fa_sync_status() == 0
    rows = _rows(w)
    o_ref, l_ref = oracle.attention(f64(qc), f64(kc), f64(vc), causal=True, scale=1.0 / math.sqrt(w.d), rows=rows,
                                    window=window or (-1, -1), softcap=c)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, qc.dtype, variant)


def test_packed_sequences_full_size():
    rng = np.random.default_rng(BASE_SEED + 60)
    lens = rng.integers(256, 4097, size=16).astype(np.int64)
    total = int(lens.sum())
    hq, d = 16, 128
    qc = normal((total, hq, d), BASE_SEED + 60, 0)
    kc = normal((total, hq, d), BASE_SEED + 60, 1)
    vc = normal((total, hq, d), BASE_SEED + 60, 2)
    cu_np = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cu = torch.from_numpy(cu_np).to(DEV)
    o, lse = fa_fwd_varlen(qc.to(DEV), kc.to(DEV), vc.to(DEV), cu, cu, max_seqlen_q=int(lens.max()), causal=True)
    assert fa_sync_status() == 0
    sample = np.random.default_rng(7)
    for s in range(len(lens)):
        q0, q1 = int(cu_np[s]), int(cu_np[s + 1])
        n = q1 - q0
        if s in (0, len(lens) - 1):
            rows = oracle.all_rows(1, hq, n)
        else:
            idx = {0, 1, n - 1, n - 2} | {int(x) for x in sample.integers(0, n, size=24)}
            rows = np.array([(0, h, i) for h in (0, hq - 1) for i in sorted(idx)], dtype=np.int64)
        seq = (lambda t: f64(t[q0:q1])[None])
        o_ref, l_ref = oracle.attention(seq(qc), seq(kc), seq(vc), causal=True, scale=1.0 / math.sqrt(d), rows=rows)
        og = o[q0:q1].to(torch.float64).cpu().numpy()[rows[:, 2], rows[:, 1]]
        lg = lse[:, q0:q1].to(torch.float64).cpu().numpy()[rows[:, 1], rows[:, 2]]
        assert_parity(og, lg, o_ref, l_ref, qc.dtype, f"packed sequence {s} (length {n})")


def test_heads_as_rows_decode_full_size():
    b, skv, hq, hkv, d = 8, 32768, 64, 8, 128
    qc, kc, vc = make_custom(b, 1, skv, hq, hkv, d, "bf16", seed=BASE_SEED + 70)
    o, lse = fa_fwd_splitkv(qc.to(DEV), kc.to(DEV), vc.to(DEV))
    assert fa_sync_status() == 0
    rows = oracle.all_rows(b, hq, 1)
    o_ref, l_ref = oracle.attention(f64(qc), f64(kc), f64(vc), causal=False, scale=1.0 / math.sqrt(d), rows=rows)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, qc.dtype, "heads-as-rows decode")


@pytest.mark.parametrize("shape", [(1, 32, 8, 128), (8, 32, 8, 64)], ids=["decode_b1", "decode_d64"])
def test_small_and_d64_decode_full_size(shape):
    """The decode_b1 and decode_d64 lines: KV = 32768, query at the last position; every row."""
    b, hq, hkv, d = shape
    skv = 32768
    qc, kc, vc = make_custom(b, 1, skv, hq, hkv, d, "bf16", seed=BASE_SEED + 80)
    o, lse = fa_fwd_splitkv(qc.to(DEV), kc.to(DEV), vc.to(DEV), causal=True, q_pos_offset=skv - 1)
    assert fa_sync_status() == 0
    rows = oracle.all_rows(b, hq, 1)
    o_ref, l_ref = oracle.attention(f64(qc), f64(kc), f64(vc), causal=True, q_pos_offset=skv - 1,
                                    scale=1.0 / math.sqrt(d), rows=rows)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, qc.dtype, f"decode {shape}")


def test_paged_decode_full_size():
    """The decode_paged line: B=8, Hq=32, Hkv=8, d=128, 256-key pages in a shuffled
    order, lengths 16384-49152; every row, each sequence's pages gathered back for the oracle."""
    from tiled_exact_attention_gb300 import fa_fwd_kvcache

    b, hq, hkv, d, ps = 8, 32, 8, 128, 256
    rng = np.random.default_rng(BASE_SEED + 50)
    lens = rng.integers(16384, 49153, size=b).astype(np.int32)
    pages_per = [int((n + ps - 1) // ps) for n in lens]
    num_pages = sum(pages_per)
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.zeros((b, max(pages_per)), dtype=np.int32)
    nxt = 0
    for i, npg in enumerate(pages_per):
        table[i, :npg] = perm[nxt:nxt + npg]
        nxt += npg
    qc = normal((b, hq, d), BASE_SEED + 50, 0)
    kc = normal((num_pages, ps, hkv, d), BASE_SEED + 50, 1)
    vc = normal((num_pages, ps, hkv, d), BASE_SEED + 50, 2)
    o, lse = fa_fwd_kvcache(qc.to(DEV), kc.to(DEV), vc.to(DEV), block_table=torch.from_numpy(table).to(DEV),
                            seqlens_k=torch.from_numpy(lens).to(DEV), max_seqlen_k=int(lens.max()))
    assert fa_sync_status() == 0
    for i in range(b):
        n, pages = int(lens[i]), table[i, :pages_per[i]]
        ks = kc[torch.from_numpy(pages).long()].reshape(-1, hkv, d)[:n][None]
        vs = vc[torch.from_numpy(pages).long()].reshape(-1, hkv, d)[:n][None]
        rows = oracle.all_rows(1, hq, 1)
        o_ref, l_ref = oracle.attention(f64(qc[i][None, None]), f64(ks), f64(vs), scale=1.0 / math.sqrt(d), rows=rows)
        og = o[i].to(torch.float64).cpu().numpy()
        lg = lse[i].to(torch.float64).cpu().numpy()
        assert_parity(og, lg, o_ref, l_ref, qc.dtype, f"paged sequence {i} (length {n})")
