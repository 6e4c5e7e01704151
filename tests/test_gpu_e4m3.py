"""GPU checks of the 8-bit (e4m3) forward path.

* The quantiser against oracle/e4m3.py, code for code (both sides form
  x * (1 / descale) in fp32 and round to nearest even).
* The e4m3 forward pass against the fp64 oracle run on the dequantised inputs
  (codes * descales).  What the kernel adds beyond that is the rounding of P to
  e4m3 before the P V product: each probability carries a relative error of at
  most 2^-4, so |O - O_ref| <= 2^-4 * max|V| (+ the bf16 rounding of O); LSE is
  formed from fp32 scores and sums and keeps the 1e-3 bound.
"""
from __future__ import annotations

import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from oracle import e4m3

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
    # b, sq, skv, hq, hkv, causal, offset, window
    (1, 513, 513, 2, 2, True, None, None),
    (2, 300, 700, 4, 2, False, None, None),
    (1, 640, 640, 8, 2, True, None, None),
    (1, 400, 400, 2, 1, False, None, (100, 20)),
    (1, 200, 100, 2, 2, True, 50, None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(str(x) for x in c))
def test_e4m3_forward_matches_oracle_on_dequantised_inputs(case):
    b, sq, skv, hq, hkv, causal, off, window = case
    d = 128
    q, k, v = make_custom(b, sq, skv, hq, hkv, d, "bf16", std=1.0, seed=zlib.crc32(repr(case).encode()) % 100000)
    (q8, qd), (k8, kd), (vt8, vd) = (fa_quantize_e4m3(q.to(DEV)), fa_quantize_e4m3(k.to(DEV)),
                                     fa_quantize_e4m3(v.to(DEV), per_head=True, transpose=True))
    o, lse = fa_fwd_e4m3(q8, qd, k8, kd, vt8, vd, causal=causal, q_pos_offset=off, window=window)
    assert fa_sync_status() == 0
    qx = e4m3.dequantize_blocks(q8.cpu().numpy(), qd.cpu().numpy())
    kx = e4m3.dequantize_blocks(k8.cpu().numpy(), kd.cpu().numpy())
    v8 = vt8.cpu().numpy()[..., :skv].transpose(0, 3, 1, 2)
    vx = e4m3.dequantize_blocks(v8, vd.cpu().numpy(), per_head=True)
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle.attention(qx, kx, vx, causal=causal, q_pos_offset=off, scale=1.0 / math.sqrt(d),
                                    rows=rows, window=window if window else (-1, -1))
    og = o.to(torch.float64).cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]]
    lg = lse.to(torch.float64).cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    masked = np.isneginf(l_ref)
    assert np.all(np.isneginf(lg[masked])) and np.all(og[masked] == 0.0)
    vis = ~masked
    tol_o = 2.0 ** -4 * np.abs(vx).max() + 1e-2
    do = np.abs(og[vis] - o_ref[vis]).max()
    dl = np.abs(lg[vis] - l_ref[vis]).max()
    assert do <= tol_o, f"O max|diff| {do:.3e} > {tol_o:.3e}"
    assert dl <= 1e-3, f"LSE max|diff| {dl:.3e}"
