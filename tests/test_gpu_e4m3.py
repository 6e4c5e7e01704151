"""GPU checks of the 8-bit (e4m3) forward path.

* The quantiser against oracle/e4m3.py, code for code (both sides form
  x * (1 / descale) in fp32 and round to nearest even).
* The e4m3 forward pass against the fp64 oracle run on the dequantised inputs
  (codes * descales).  What the kernel adds beyond that is the rounding of each
  probability to e4m3 before the P V product, and the rounding of O to bf16.
  Per element (row i, column c) the check is the bound that rounding allows:

    |O_ic - O_ref,ic| <= 2^-4 * sum_j P_ij |V_jc|              (normal e4m3 codes)
                       + 2^-10 * Pmax_i * sum_{j visible} |V_jc| (subnormal codes)
                       + 2^-8 * |O_ref,ic| + 1e-6             (bf16 O, fp32 sums)

  The kernel forms p_j = 2^(x_j - m_ref) with a reference maximum m_ref no
  larger than the row's maximum, so its largest p is at least 1 and its row sum
  l is at least 1 / Pmax_i, Pmax_i = exp(m_i - LSE_i) the largest probability of
  the row.  A normal e4m3 code (p >= 2^-6) is off by at most 2^-4 of p; a
  subnormal one by at most 2^-10.  Every term is computed by the oracle: the
  first from the oracle with |V| in place of V, the sum of |V| over the visible
  keys from the oracle at scale 0 (uniform weights 1 / n_i, LSE = ln n_i), and
  an upper bound of m_i from the oracle at 1000 times the scale
  (LSE_1000 / 1000 >= m_i).  LSE is formed from fp32 scores and sums and keeps
  the 1e-3 bound.  A case with V shifted away from zero makes |O| far larger
  than the bound, so a V scale applied twice or not at all cannot pass.
"""
from __future__ import annotations

import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from oracle import e4m3
from parity_util import e4m3_rounding_bound

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from tiled_exact_attention_gb300 import fa_fwd_e4m3, fa_quantize_e4m3, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300.inputs import make_custom, normal  # noqa: E402

DEV = "cuda:0"


def _f32(t):
    return t.detach().cpu().to(torch.float32).numpy()


@pytest.mark.parametrize("shape,dts,per_head,transpose", [
    ((2, 300, 3, 128), "bf16", False, False),
    ((1, 257, 2, 64), "fp16", False, False),
    ((2, 300, 3, 128), "bf16", True, True),
    ((1, 129, 4, 128), "fp16", True, True),
    ((1, 300, 2, 256), "bf16", False, False),
    ((2, 200, 2, 256), "fp16", True, True),
    ((1, 140, 3, 64), "bf16", True, True),
])
def test_quantizer_matches_reference_code_for_code(shape, dts, per_head, transpose):
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dts]
    x = normal(shape, 321, 0, 2.0, dt)
    x[0, :, 0, :5] *= 300.0          # outliers in one head
    x[-1, 128:256, -1, :] = 0.0      # an all-zero block
    x[0, :, 1, :] *= 1e-4            # small values, some in the subnormal range after scaling
    codes, ds = fa_quantize_e4m3(x.to(DEV), per_head=per_head, transpose=transpose)
    assert fa_sync_status() == 0
    ref_codes, ref_ds = e4m3.quantize_blocks(_f32(x), per_head=per_head)
    assert np.array_equal(ds.cpu().numpy(), ref_ds)
    got = codes.cpu().numpy()
    if transpose:
        got = got[..., : shape[1]].transpose(0, 3, 1, 2)  # [b, h, d, s] -> [b, s, h, d]
    assert np.array_equal(got, ref_codes)


CASES = [
    # b, sq, skv, hq, hkv, d, causal, offset, window, V mean
    (1, 513, 513, 2, 2, 128, True, None, None, 0.0),
    (2, 300, 700, 4, 2, 128, False, None, None, 0.0),
    (1, 640, 640, 8, 2, 128, True, None, None, 0.0),
    (1, 400, 400, 2, 1, 128, False, None, (100, 20), 0.0),
    (1, 200, 100, 2, 2, 128, True, 50, None, 0.0),
    (2, 300, 700, 4, 2, 128, False, None, None, 1.5),
    (1, 640, 640, 4, 4, 128, True, None, None, -2.0),
    (1, 513, 513, 2, 2, 64, True, None, None, 0.0),
    (2, 300, 700, 4, 2, 64, False, None, None, 1.5),
    (1, 400, 400, 2, 1, 64, False, None, (100, 20), 0.0),
    (1, 640, 640, 8, 2, 64, True, None, None, -2.0),
    (1, 513, 513, 2, 2, 256, True, None, None, 0.0),
    (2, 300, 700, 4, 2, 256, False, None, None, 1.5),
    (1, 400, 400, 2, 1, 256, False, None, (100, 20), 0.0),
    (1, 200, 100, 2, 2, 256, True, 50, None, -2.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(str(x) for x in c))
def test_e4m3_forward_matches_oracle_on_dequantised_inputs(case):
    b, sq, skv, hq, hkv, d, causal, off, window, vmean = case
    q, k, v = make_custom(b, sq, skv, hq, hkv, d, "bf16", std=1.0, seed=zlib.crc32(repr(case).encode()) % 100000)
    if vmean:
        v = (v.float() + vmean).to(torch.bfloat16)
    (q8, qd), (k8, kd), (vt8, vd) = (fa_quantize_e4m3(q.to(DEV)), fa_quantize_e4m3(k.to(DEV)),
                                     fa_quantize_e4m3(v.to(DEV), per_head=True, transpose=True))
    o, lse = fa_fwd_e4m3(q8, qd, k8, kd, vt8, vd, causal=causal, q_pos_offset=off, window=window)
    assert fa_sync_status() == 0
    qx = e4m3.dequantize_blocks(q8.cpu().numpy(), qd.cpu().numpy())
    kx = e4m3.dequantize_blocks(k8.cpu().numpy(), kd.cpu().numpy())
    v8 = vt8.cpu().numpy()[..., :skv].transpose(0, 3, 1, 2)
    vx = e4m3.dequantize_blocks(v8, vd.cpu().numpy(), per_head=True)
    scale = 1.0 / math.sqrt(d)
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle.attention(qx, kx, vx, causal=causal, q_pos_offset=off, scale=scale,
                                    rows=rows, window=window if window else (-1, -1))
    og = o.to(torch.float64).cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]]
    lg = lse.to(torch.float64).cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    masked = np.isneginf(l_ref)
    assert np.all(np.isneginf(lg[masked])) and np.all(og[masked] == 0.0)
    vis = ~masked
    tol = e4m3_rounding_bound(qx, kx, vx, causal, off, window, o_ref, l_ref, rows, scale)
    err = np.abs(og - o_ref)
    worst = np.unravel_index(np.argmax(err[vis] - tol[vis]), err[vis].shape)
    assert np.all(err[vis] <= tol[vis]), (
        f"O off by {err[vis][worst]:.3e} where rounding allows {tol[vis][worst]:.3e}")
    dl = np.abs(lg[vis] - l_ref[vis]).max()
    assert dl <= 1e-3, f"LSE max|diff| {dl:.3e}"
    if vmean:
        # the bound is tight enough to see a V scale applied twice (O doubled) or not at all
        assert np.mean(np.abs(o_ref[vis]) > tol[vis]) > 0.9


def _draw_e4m3(i):
    rng = np.random.default_rng(9100 + i)
    d = int(rng.choice([64, 128, 256]))
    g = int(rng.choice([1, 2, 4]))
    hkv = int(rng.integers(1, 3))
    b = int(rng.integers(1, 3))
    sq = int(rng.integers(1, 600))
    skv = int(rng.integers(1, 800))
    causal = bool(rng.integers(0, 2))
    off = int(rng.integers(-40, 500)) if causal and rng.integers(0, 2) else None
    window = (int(rng.integers(-1, 250)), int(rng.integers(-1, 250))) if rng.integers(0, 3) == 0 else None
    vmean = float(rng.choice([0.0, 0.0, 1.5, -2.0]))
    return b, sq, skv, g * hkv, hkv, d, causal, off, window, vmean


@pytest.mark.parametrize("i", range(12))
def test_e4m3_forward_random(i):
    """Seeded random shapes (every head dimension, lengths cutting tiles anywhere,
    groups, offsets, windows, shifted V) against the same per-element bound."""
    b, sq, skv, hq, hkv, d, causal, off, window, vmean = case = _draw_e4m3(i)
    q, k, v = make_custom(b, sq, skv, hq, hkv, d, "bf16", std=1.0, seed=9200 + i)
    if vmean:
        v = (v.float() + vmean).to(torch.bfloat16)
    (q8, qd), (k8, kd), (vt8, vd) = (fa_quantize_e4m3(q.to(DEV)), fa_quantize_e4m3(k.to(DEV)),
                                     fa_quantize_e4m3(v.to(DEV), per_head=True, transpose=True))
    o, lse = fa_fwd_e4m3(q8, qd, k8, kd, vt8, vd, causal=causal, q_pos_offset=off, window=window)
    assert fa_sync_status() == 0
    qx = e4m3.dequantize_blocks(q8.cpu().numpy(), qd.cpu().numpy())
    kx = e4m3.dequantize_blocks(k8.cpu().numpy(), kd.cpu().numpy())
    vx = e4m3.dequantize_blocks(vt8.cpu().numpy()[..., :skv].transpose(0, 3, 1, 2), vd.cpu().numpy(), per_head=True)
    scale = 1.0 / math.sqrt(d)
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle.attention(qx, kx, vx, causal=causal, q_pos_offset=off, scale=scale, rows=rows,
                                    window=window if window else (-1, -1))
    og = o.to(torch.float64).cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]]
    lg = lse.to(torch.float64).cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    masked = np.isneginf(l_ref)
    assert np.all(np.isneginf(lg[masked])) and np.all(og[masked] == 0.0), case
    vis = ~masked
    tol = e4m3_rounding_bound(qx, kx, vx, causal, off, window, o_ref, l_ref, rows, scale)
    assert np.all(np.abs(og - o_ref)[vis] <= tol[vis]), case
    if vis.any():
        assert np.abs(lg[vis] - l_ref[vis]).max() <= 1e-3, case


@pytest.mark.parametrize("name", ["causal_prefill", "ragged_d64", "ragged_d256"])
def test_e4m3_full_size_on_the_benchmark_inputs(name):
    """The 8-bit forward at the benchmark's full sizes, on its own inputs quantised
    the way its e4m3 lines quantise them and in the same launch: one whole head of
    the last batch and a random sample of rows (with the edge rows) against the
    per-element bound."""
    from tiled_exact_attention_gb300 import quantize_qkv_e4m3
    from tiled_exact_attention_gb300.inputs import WORKLOADS, make_qkv
    from parity_util import sample_rows

    w = WORKLOADS[name]
    qc, kc, vc = make_qkv(w)
    (q8, qd), (k8, kd), (vt8, vd) = quantize_qkv_e4m3(qc.to(DEV), kc.to(DEV), vc.to(DEV))
    off = w.offset if w.causal else None
    o, lse = fa_fwd_e4m3(q8, qd, k8, kd, vt8, vd, causal=w.causal, q_pos_offset=off)
    assert fa_sync_status() == 0
    qx = e4m3.dequantize_blocks(q8.cpu().numpy(), qd.cpu().numpy())
    kx = e4m3.dequantize_blocks(k8.cpu().numpy(), kd.cpu().numpy())
    vx = e4m3.dequantize_blocks(vt8.cpu().numpy()[..., :w.skv].transpose(0, 3, 1, 2), vd.cpu().numpy(),
                                per_head=True)
    rows = {tuple(r) for r in sample_rows(w.b, w.hq, w.sq, n_random=512, seed=w.index)}
    rows.update((w.b - 1, w.hq - 1, i) for i in range(w.sq))
    rows = np.array(sorted(rows), dtype=np.int64)
    scale = 1.0 / math.sqrt(w.d)
    o_ref, l_ref = oracle.attention(qx, kx, vx, causal=w.causal, q_pos_offset=off, scale=scale, rows=rows)
    og = o.to(torch.float64).cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]]
    lg = lse.to(torch.float64).cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    masked = np.isneginf(l_ref)
    assert np.all(np.isneginf(lg[masked])) and np.all(og[masked] == 0.0)
    vis = ~masked
    tol = e4m3_rounding_bound(qx, kx, vx, w.causal, off, None, o_ref, l_ref, rows, scale)
    err = np.abs(og - o_ref)
    assert np.all(err[vis] <= tol[vis]), f"{name}: O off by {np.max(err[vis] - tol[vis]):.3e} beyond the bound"
    assert np.abs(lg[vis] - l_ref[vis]).max() <= 1e-3, name
