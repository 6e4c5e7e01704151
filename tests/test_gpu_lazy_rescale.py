"""GPU parity where the running row maximum climbs across key blocks.

The online softmax ("hs-black: FlashAttention 1/2/3", section "Online softmax:
merge while reading") rescales the carried numerator and denominator by
alpha = exp(m - m') whenever the maximum moves.  The tensor-core kernel moves its
reference maximum only when a block's maximum exceeds it by more than 8 log2
units (exact in real arithmetic: the numerator and the denominator share the
reference), so the rounding path depends on where each block's maximum falls
relative to that threshold.  These inputs are built so that, in the order the
kernel visits the key blocks (the highest block first), every row's block
maximum climbs by a chosen amount g per block: just under, at and just over 8
log2 units, half and twice that, more than 100 natural units (150 log2 units and
beyond), and falling maxima.  The results must match the oracle element by element like
any other input.

Construction: q_i = (u_i, 0, ..., 0) and K's first column holds c = t for one
key of the block visited t-th (t = 0, 1, ...) and c = t - delta (delta in
[0.05, 2]) for its other keys; every other entry of K is 0.  Row i's score for
that key is then scale * u_i * t, so in log2 units its block maximum grows by
g_i = log2(e) * scale * u_i per block.  The increments realised after rounding
the inputs to 16 bits are recomputed here from the stored values and checked to
straddle the threshold as intended.
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

from tiled_exact_attention_gb300 import fa_fwd, fa_fwd_splitkv, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300.inputs import normal  # noqa: E402

DEV = "cuda:0"
LOG2E = 1.0 / math.log(2.0)

# per-row increments of the block maximum, log2 units
G_SPECIAL = [7.9, 8.1, 7.95, 8.05, 8.0, 3.9, 4.1, 16.0, 150.0, 200.0, 1000.0, -7.9, -8.1, -150.0, 0.0, 0.25]


def _key_block(d: int) -> int:
    # keys per block of the tensor-core forward kernel (128 for d <= 128, 64 for d = 256)
    return 128 if d <= 128 else 64


def _build(d, rows_g, nblk, tail, dt, seed, hq=2, hkv=1):
    """Q [1, sq, hq, d] with row i of head h carrying u = rows_g[h][i] / (log2 e * scale); K, V [1, skv, hkv, d]."""
    bn = _key_block(d)
    skv = nblk * bn - tail
    scale = 1.0 / math.sqrt(d)
    sq = len(rows_g[0])
    q = torch.zeros((1, sq, hq, d), dtype=torch.float32)
    for h in range(hq):
        q[0, :, h, 0] = torch.tensor(rows_g[h], dtype=torch.float32) / (LOG2E * scale)
    rng = np.random.default_rng(seed)
    kcol = np.empty(skv, dtype=np.float64)
    for n in range(nblk):
        t = nblk - 1 - n  # visit position of block n
        lo, hi = n * bn, min((n + 1) * bn, skv)
        kcol[lo:hi] = t - rng.uniform(0.05, 2.0, size=hi - lo)
        kcol[lo] = t  # the block's first key is always inside the sequence
    k = torch.zeros((1, skv, hkv, d), dtype=torch.float32)
    k[0, :, :, 0] = torch.from_numpy(kcol).float()[:, None]
    v = normal((1, skv, hkv, d), seed, 2, 1.0, torch.float32)
    return q.to(dt), k.to(dt), v.to(dt), scale


def _realised_increments(q, k, d, nblk):
    """Per (row, head): the block maxima in log2 units, in visit order, from the stored inputs."""
    bn = _key_block(d)
    scale = 1.0 / math.sqrt(d)
    s = np.einsum("ihd,jd->ihj", f64(q)[0], f64(k)[0, :, 0, :]) * scale * LOG2E
    mx = np.stack([s[:, :, n * bn:(n + 1) * bn].max(axis=2) for n in range(nblk - 1, -1, -1)], axis=2)
    return np.diff(mx, axis=2)


def _rows_g(sq, head):
    base = np.array(G_SPECIAL, dtype=np.float64)
    fill = np.linspace(7.5, 8.5, sq - len(base)) if head == 0 else np.linspace(-1.0, 20.0, sq - len(base))
    g = np.concatenate([base, fill])
    return g if head == 0 else g[::-1].copy()


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("dts", ["bf16", "fp16"])
@pytest.mark.parametrize("tail", [0, 37])
def test_forward_rising_block_maxima(d, dts, tail):
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dts]
    sq, nblk = 256, 6
    rows_g = [_rows_g(sq, 0), _rows_g(sq, 1)]
    q, k, v, scale = _build(d, rows_g, nblk, tail, dt, seed=4100 + d + tail)
    inc = _realised_increments(q, k, d, nblk)
    # the stored inputs do straddle the threshold: increments just under and just over 8
    assert ((inc > 7.8) & (inc < 8.0)).any() and ((inc > 8.0) & (inc < 8.2)).any()
    assert (inc > 100.0 * LOG2E - 1e-3).any() and (inc < -8.0).any()
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse = fa_fwd(q, k, v, causal=False, scale=scale)
    assert fa_sync_status() == 0
    rows = oracle.all_rows(1, 2, sq)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v), causal=False, scale=scale, rows=rows)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, dt, f"d={d} {dts} tail={tail}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [2, 3])
def test_split_mode_rising_block_maxima(d, splits):
    """The same rows through the split-KV path (sq > 1: the forward kernel in
    split mode, each split starting its own running maximum, then the merge)."""
    sq, nblk = 256, 6
    rows_g = [_rows_g(sq, 0), _rows_g(sq, 1)]
    q, k, v, scale = _build(d, rows_g, nblk, 0, torch.bfloat16, seed=4200 + d)
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse, used = fa_fwd_splitkv(q, k, v, causal=False, scale=scale, num_splits=splits, return_splits=True)
    assert fa_sync_status() == 0 and used == splits
    rows = oracle.all_rows(1, 2, sq)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v), causal=False, scale=scale, rows=rows)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, torch.bfloat16, f"split d={d} ns={splits}")


@pytest.mark.parametrize("g_heads", [4, 8, 16])
def test_decode_rising_block_maxima(g_heads):
    """One query row per head (decode): each query head carries its own increment;
    with 8 or more heads per KV head they are the rows of one tensor-core tile."""
    d, nblk, hkv = 128, 12, 2
    hq = g_heads * hkv
    g = np.array((G_SPECIAL * 2)[:hq], dtype=np.float64)
    bn = _key_block(d)
    skv = nblk * bn
    scale = 1.0 / math.sqrt(d)
    rng = np.random.default_rng(4300 + g_heads)
    q = torch.zeros((2, 1, hq, d), dtype=torch.float32)
    q[:, 0, :, 0] = torch.from_numpy(g / (LOG2E * scale)).float()[None, :]
    kcol = np.empty(skv)
    for n in range(nblk):
        t = nblk - 1 - n
        kcol[n * bn:(n + 1) * bn] = t - rng.uniform(0.05, 2.0, size=bn)
        kcol[n * bn] = t
    k = torch.zeros((2, skv, hkv, d), dtype=torch.float32)
    k[:, :, :, 0] = torch.from_numpy(kcol).float()[None, :, None]
    v = normal((2, skv, hkv, d), 4300 + g_heads, 2, 1.0, torch.float32)
    q, k, v = (t.to(torch.bfloat16).to(DEV) for t in (q, k, v))
    for ns in (1, 3):
        o, lse = fa_fwd_splitkv(q, k, v, causal=True, q_pos_offset=skv - 1, scale=scale, num_splits=ns)
        assert fa_sync_status() == 0
        rows = oracle.all_rows(2, hq, 1)
        o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v), causal=True, q_pos_offset=skv - 1, scale=scale,
                                        rows=rows)
        og, lg = gather(o, lse, rows)
        assert_parity(og, lg, o_ref, l_ref, torch.bfloat16, f"decode g={g_heads} ns={ns}")
