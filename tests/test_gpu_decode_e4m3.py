"""GPU parity of fa_fwd_splitkv_e4m3 (split-KV decode over e4m3 keys and values).

K is quantised with one scale per 128-key block and V with one scale per
(batch, head), as fa_quantize_e4m3 does; the oracle runs on the dequantised
values (codes times scales, exact in fp64) with the 16-bit query.  The kernel
widens the codes exactly and keeps every product and sum in fp32, so the
16-bit tolerances of the other parity tests apply: O max |diff| 1e-2 (bf16) or
4e-3 (fp16), LSE 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import e4m3
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from tiled_exact_attention_gb300 import fa_fwd_splitkv_e4m3, fa_quantize_e4m3, fa_sync_status  # noqa: E402
from tiled_exact_attention_gb300.inputs import normal  # noqa: E402

DEV = "cuda:0"
_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}

CASES = [
    # b, skv, hq, hkv, d, dtype, splits, std
    (2, 1000, 8, 2, 128, "bf16", 0, 1.0),
    (2, 1000, 8, 2, 128, "bf16", 3, 1.0),
    (1, 777, 8, 1, 64, "fp16", 0, 2.0),
    (3, 129, 3, 1, 128, "bf16", 2, 1.0),
    (1, 300, 16, 2, 64, "bf16", 5, 1.0),
    (2, 4096, 32, 8, 128, "fp16", 0, 1.0),
    (1, 5000, 4, 4, 128, "fp16", 7, 2.0),   # peaky rows (std 2), |O| up to ~10
    (8, 32768, 32, 8, 128, "bf16", 0, 1.0),   # the split-KV decode workload's shape
]


def _quantised(b, skv, hq, hkv, d, dts, seed, std):
    dt = _DT[dts]
    q = normal((b, hq, d), seed, 0, std, dt)
    k = normal((b, skv, hkv, d), seed, 1, std, dt)
    v = normal((b, skv, hkv, d), seed, 2, std, dt)
    k8, kd = fa_quantize_e4m3(k.to(DEV))
    v8, vd = fa_quantize_e4m3(v.to(DEV), per_head=True)
    return q, k8, kd, v8, vd


def _reference(q, k8, kd, v8, vd, scale):
    kx = e4m3.dequantize_blocks(k8.cpu().numpy(), kd.cpu().numpy())
    vx = e4m3.dequantize_blocks(v8.cpu().numpy(), vd.cpu().numpy(), per_head=True)
    qx = q.to(torch.float64).numpy()[:, None]  # [b, 1, hq, d]
    return oracle.attention(qx, kx, vx, causal=False, scale=scale)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(str(x) for x in c))
def test_decode_e4m3_matches_oracle_on_dequantised_kv(case):
    b, skv, hq, hkv, d, dts, ns, std = case
    q, k8, kd, v8, vd = _quantised(b, skv, hq, hkv, d, dts, 6000 + skv + d, std)
    o, lse, used = fa_fwd_splitkv_e4m3(q.to(DEV), k8, kd, v8, vd, num_splits=ns, return_splits=True)
    assert fa_sync_status() == 0
    assert used >= 1 and (ns == 0 or used == min(ns, math.ceil(skv / 128)))
    o_ref, l_ref = _reference(q, k8, kd, v8, vd, 1.0 / math.sqrt(d))
    og = o.to(torch.float64).cpu().numpy().reshape(-1, d)
    lg = lse.to(torch.float64).cpu().numpy().reshape(-1)
    assert_parity(og, lg, o_ref, l_ref, _DT[dts], str(case))


def test_decode_e4m3_no_keys():
    """skv = 0: every row sees no key, O = 0 and LSE = -inf."""
    q = normal((2, 4, 128), 7, 0, 1.0, torch.bfloat16).to(DEV)
    k8 = torch.zeros((2, 0, 2, 128), dtype=torch.uint8, device=DEV)
    kd = torch.zeros((2, 2, 0), dtype=torch.float32, device=DEV)
    vd = torch.zeros((2, 2), dtype=torch.float32, device=DEV)
    o, lse = fa_fwd_splitkv_e4m3(q, k8, kd, k8.clone(), vd)
    assert fa_sync_status() == 0
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_decode_e4m3_matches_16bit_decode_within_quantisation():
    """The same problem through the 16-bit split-KV decode: the two differ by the
    e4m3 rounding of K and V only (a loose sanity bound, not a parity check)."""
    from tiled_exact_attention_gb300 import fa_fwd_splitkv

    b, skv, hq, hkv, d = 2, 3000, 8, 2, 128
    q, k, v = (normal(s, 77, i, 1.0, torch.bfloat16).to(DEV)
               for i, s in enumerate(((b, hq, d), (b, skv, hkv, d), (b, skv, hkv, d))))
    k8, kd = fa_quantize_e4m3(k)
    v8, vd = fa_quantize_e4m3(v, per_head=True)
    o8, l8 = fa_fwd_splitkv_e4m3(q, k8, kd, v8, vd)
    o16, l16 = fa_fwd_splitkv(q[:, None], k, v, causal=True, q_pos_offset=skv - 1)
    assert fa_sync_status() == 0
    assert (o8.float() - o16[:, 0].float()).abs().max().item() < 0.1
    assert (l8 - l16[:, :, 0]).abs().max().item() < 0.1
