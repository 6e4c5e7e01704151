"""Pins of the oracle's softcap (logit capping) to facts outside itself.

Reading of "flash attention V2 code walkthrough", template flag Is_softcap (tanh
softly limits the logits when softcap > 0; no formula is printed): every scaled
score s becomes c * tanh(s / c).  The pins: a two-key case whose capped scores are
exact (tanh((ln 3) / 2) = 1/2), the limit c -> inf (the cap vanishes like s^3 / (3 c^2)),
the bound |s'| < c on the LSE, the tiled recurrence against the direct definition,
and torch's autograd through its own tanh and softmax for the backward pass.  The
last tests plant the two plausible mistakes (cap before the scale; the cap's
derivative dropped) and check that the pins catch them.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _two_keys(scale):
    # q = 1 (d = 1); raw dot products 0 and 2 ln 3; with scale 1/2 the scaled scores are
    # 0 and ln 3, capped (c = 2) to 2 tanh(0) = 0 and 2 tanh((ln 3) / 2) = 2 * (1/2) = 1
    q = np.ones((1, 1, 1, 1))
    k = np.array([0.0, 2.0 * math.log(3.0)]).reshape(1, 2, 1, 1) / (2.0 * scale)
    v = np.array([1.0, 3.0]).reshape(1, 2, 1, 1)
    return q, k, v


def test_two_keys_closed_form(oracle_mod):
    q, k, v = _two_keys(0.5)
    o, lse = oracle_mod.attention(q, k, v, scale=0.5, softcap=2.0)
    e = math.e
    assert abs(o[0, 0] - (1.0 + 3.0 * e) / (1.0 + e)) < 1e-14
    assert abs(lse[0] - math.log(1.0 + e)) < 1e-14


def test_cap_before_scale_is_caught(oracle_mod):
    q, k, v = _two_keys(0.5)
    o, _ = oracle_mod.attention(q, k, v, scale=0.5, softcap=2.0, mutation=oracle_mod.MUT_CAP_BEFORE_SCALE)
    e = math.e
    assert abs(o[0, 0] - (1.0 + 3.0 * e) / (1.0 + e)) > 1e-3


def test_large_cap_vanishes_like_inverse_square(oracle_mod):
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal(s) for s in ((1, 6, 2, 8), (1, 9, 2, 8), (1, 9, 2, 8)))
    o0, l0 = oracle_mod.attention(q, k, v, causal=True)
    diffs = []
    for c in (40.0, 80.0, 160.0):
        o, l = oracle_mod.attention(q, k, v, causal=True, softcap=c)
        diffs.append(np.abs(o - o0).max() + np.abs(l - l0).max())
    assert diffs[0] > 1e-8  # a tanh cap (a clamp at +-c would change nothing here)
    for a, b in zip(diffs, diffs[1:]):
        assert 3.5 < a / b < 4.5  # c * tanh(s / c) = s - s^3 / (3 c^2) + ...
    o, l = oracle_mod.attention(q, k, v, causal=True, softcap=1e7)
    assert np.abs(o - o0).max() < 1e-12 and np.abs(l - l0).max() < 1e-12


def test_lse_bounded_by_the_cap(oracle_mod):
    rng = np.random.default_rng(5)
    n = 17
    q = rng.standard_normal((1, 4, 1, 16)) * 30.0
    k = rng.standard_normal((1, n, 1, 16)) * 30.0
    v = rng.standard_normal((1, n, 1, 16))
    c = 3.0
    o, lse = oracle_mod.attention(q, k, v, scale=1.0, softcap=c)
    assert np.all(lse <= c + math.log(n) + 1e-12) and np.all(lse >= -c + math.log(n) - 1e-12)
    o_plain, lse_plain = oracle_mod.attention(q, k, v, scale=1.0)
    assert np.abs(lse_plain).max() > 100.0  # the same scores uncapped are far outside the bound


@pytest.mark.parametrize("tile,splits,causal,window", [(1, 1, True, (-1, -1)), (3, 2, False, (-1, -1)),
                                                        (4, 3, True, (2, -1)), (8, 1, False, (3, 1))])
def test_tiled_matches_direct(oracle_mod, tile, splits, causal, window):
    rng = np.random.default_rng(tile * 10 + splits)
    q, k, v = (rng.standard_normal(s) * 2.0 for s in ((2, 9, 4, 8), (2, 11, 2, 8), (2, 11, 2, 8)))
    o, lse = oracle_mod.attention(q, k, v, causal=causal, window=window, softcap=1.5)
    ot, lt = oracle_mod.attention_tiled(q, k, v, tile=tile, num_splits=splits, causal=causal, window=window,
                                        softcap=1.5)
    fin = np.isfinite(lse)
    assert np.array_equal(fin, np.isfinite(lt))
    np.testing.assert_allclose(ot, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lt[fin], lse[fin], rtol=0, atol=1e-12)


def _torch_grads(q, k, v, do, scale, c, band):
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    g = qt.shape[2] // kt.shape[2]
    kk = kt.repeat_interleave(g, dim=2)
    vv = vt.repeat_interleave(g, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", qt, kk) * scale
    s = c * torch.tanh(s / c)
    s = s.masked_fill(~torch.from_numpy(band), float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = torch.einsum("bhij,bjhd->bihd", p, vv)
    (o * torch.from_numpy(do)).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("causal,off,c", [(False, 0, 2.0), (True, 0, 0.7), (True, 3, 5.0)])
def test_backward_matches_autograd(oracle_mod, causal, off, c):
    rng = np.random.default_rng(int(c * 10) + off)
    b, sq, skv, hq, hkv, d = 2, 6, 9, 4, 2, 8
    q, k, v, do = (rng.standard_normal(s) * 1.5 for s in ((b, sq, hq, d), (b, skv, hkv, d), (b, skv, hkv, d),
                                                          (b, sq, hq, d)))
    i = np.arange(sq)[:, None]
    j = np.arange(skv)[None, :]
    band = (j <= i + off) if causal else np.ones((sq, skv), dtype=bool)
    sc = 1.0 / math.sqrt(d)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, do, causal=causal, q_pos_offset=off, scale=sc, softcap=c)
    tq, tk, tv = _torch_grads(q, k, v, do, sc, c, band)
    np.testing.assert_allclose(dq, tq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tv, rtol=0, atol=1e-11)
    # the same pin catches a dropped derivative of the cap
    mq, mk, _ = oracle_mod.attention_bwd(q, k, v, do, causal=causal, q_pos_offset=off, scale=sc, softcap=c,
                                         mutation=oracle_mod.MUT_CAP_NO_DERIV)
    assert np.abs(mq - tq).max() > 1e-4 and np.abs(mk - tk).max() > 1e-4
