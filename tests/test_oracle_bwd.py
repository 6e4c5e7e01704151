"""Pins of the fp64 backward oracle to facts outside itself: the worked example and
exercise of the "hs-black" page, torch's autograd through its own softmax (fp64),
central differences of the oracle's forward pass, and the zero-sum identities of
the page ("a convenient self-check": every row of dS sums to zero).  The last test
plants mistakes in the oracle and checks that the pins catch them."""
import math

import numpy as np
import pytest
import torch

from golden_io import read_kv

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _scalar(scores, values, dout):
    n = len(scores)
    q = np.ones((1, 1, 1, 1))
    k = np.asarray(scores, dtype=np.float64).reshape(1, n, 1, 1)
    v = np.asarray(values, dtype=np.float64).reshape(1, n, 1, 1)
    do = np.full((1, 1, 1, 1), float(dout))
    return q, k, v, do


def test_worked_example_one_query_two_keys(oracle_mod):
    g = read_kv("two_key_example.txt")
    q, k, v, do = _scalar(g["k"], g["v"], g["dO"])
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, do, scale=1.0)
    # with q = 1 and scale 1, dK_j = dS_j q = dS_j: the printed dS
    np.testing.assert_allclose(dk.ravel(), g["printed_dS"], rtol=0, atol=1e-14)
    # dV = P dO with the printed P
    np.testing.assert_allclose(dv.ravel(), np.array(g["printed_P"]) * g["dO"], rtol=0, atol=1e-14)
    # dQ = sum_j dS_j k_j
    assert abs(dq.ravel()[0] - float(np.dot(g["printed_dS"], g["k"]))) < 1e-14
    # D = dO * O (printed 10): dS_j = P_j (dO v_j - D)
    p = np.array(g["printed_P"])
    np.testing.assert_allclose(p * (g["dO"] * np.array(g["v"]) - g["printed_D"]), g["printed_dS"], atol=1e-14)


def test_exercise_two(oracle_mod):
    g = read_kv("backward_exercise2.txt")
    q, k, v, do = _scalar(np.log(g["P"]), g["v"], g["dO"])
    o, _ = oracle_mod.attention(q, k, v, scale=1.0)
    assert abs(o[0, 0] - g["answer_O"]) < 1e-13
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, do, scale=1.0)
    np.testing.assert_allclose(dk.ravel(), g["answer_dS"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv.ravel(), g["answer_dV"], rtol=0, atol=1e-13)
    assert abs(dk.sum()) < 1e-13  # the self-check


def _torch_grads(q, k, v, do, scale, band):
    """fp64 attention through torch's own softmax and autograd ([b, s, h, d] layout)."""
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    g = qt.shape[2] // kt.shape[2]
    kk = kt.repeat_interleave(g, dim=2)
    vv = vt.repeat_interleave(g, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", qt, kk) * scale
    s = s.masked_fill(~torch.from_numpy(band), float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = torch.einsum("bhij,bjhd->bihd", p, vv)
    (o * torch.from_numpy(do)).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def _band(sq, skv, causal, off, wl, wr):
    i = np.arange(sq)[:, None]
    j = np.arange(skv)[None, :]
    m = np.ones((sq, skv), dtype=bool)
    if causal:
        m &= j <= i + off
    if wl >= 0:
        m &= j >= i + off - wl
    if wr >= 0:
        m &= j <= i + off + wr
    return m


AUTOGRAD_CASES = [
    # b, sq, skv, hq, hkv, d, causal, off, (wl, wr), scale
    (2, 7, 7, 2, 2, 8, False, 0, (-1, -1), None),
    (1, 9, 9, 4, 2, 16, True, 0, (-1, -1), None),
    (2, 5, 11, 3, 1, 5, False, 6, (-1, -1), 0.3),
    (1, 12, 12, 2, 1, 8, False, 0, (3, 2), None),
    (1, 6, 10, 4, 4, 4, True, 4, (2, -1), 1.7),
]


@pytest.mark.parametrize("case", AUTOGRAD_CASES)
def test_matches_autograd(oracle_mod, case):
    b, sq, skv, hq, hkv, d, causal, off, win, scale = case
    rng = np.random.default_rng(sum(case[:6]) + 101)
    q = rng.standard_normal((b, sq, hq, d))
    k = rng.standard_normal((b, skv, hkv, d))
    v = rng.standard_normal((b, skv, hkv, d))
    do = rng.standard_normal((b, sq, hq, d))
    sc = 1.0 / math.sqrt(d) if scale is None else scale
    band = _band(sq, skv, causal, off, *win)
    assert band.any(axis=1).all()  # (rows with no key are covered separately)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, do, causal=causal, q_pos_offset=off, scale=sc, window=win)
    tq, tk, tv = _torch_grads(q, k, v, do, sc, band)
    np.testing.assert_allclose(dq, tq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tv, rtol=0, atol=1e-11)


def test_central_differences(oracle_mod):
    """Every gradient entry of a tiny causal GQA problem against a central difference
    of L = sum(dO * O) computed with the oracle's forward pass."""
    rng = np.random.default_rng(7)
    b, sq, skv, hq, hkv, d = 1, 3, 4, 2, 1, 3
    q = rng.standard_normal((b, sq, hq, d))
    k = rng.standard_normal((b, skv, hkv, d))
    v = rng.standard_normal((b, skv, hkv, d))
    do = rng.standard_normal((b, sq, hq, d))

    def loss(q_, k_, v_):
        o, _ = oracle_mod.attention(q_, k_, v_, causal=True)
        rows = oracle_mod.all_rows(b, hq, sq)
        return float((o * do[rows[:, 0], rows[:, 2], rows[:, 1]]).sum())

    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, do, causal=True)
    h = 1e-5
    for x, gx in ((q, dq), (k, dk), (v, dv)):
        for idx in np.ndindex(x.shape):
            xp = x.copy()
            xm = x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            num = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(num - gx[idx]) < 1e-8, (idx, num, gx[idx])


def test_zero_sum_identities(oracle_mod):
    """Rows of dS sum to zero, so sum_j dK_j = 0 for every (batch, kv head); and
    sum_j dV_j = sum over rows that see a key of dO_i."""
    rng = np.random.default_rng(9)
    b, sq, skv, hq, hkv, d = 2, 10, 13, 4, 2, 6
    q, do = rng.standard_normal((2, b, sq, hq, d))
    k, v = rng.standard_normal((2, b, skv, hkv, d))
    for causal, off, win in ((False, 3, (-1, -1)), (True, -2, (-1, -1)), (False, 3, (2, 1))):
        dq, dk, dv = oracle_mod.attention_bwd(q, k, v, do, causal=causal, q_pos_offset=off, window=win)
        np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
        band = _band(sq, skv, causal, off, *win)
        sees = band.any(axis=1)
        expect = do[:, sees].reshape(b, -1, hkv, hq // hkv, d).sum(axis=(1, 3))
        np.testing.assert_allclose(dv.sum(axis=1), expect, atol=1e-12)


def test_rows_without_keys_contribute_nothing(oracle_mod):
    rng = np.random.default_rng(13)
    q, do = rng.standard_normal((2, 1, 6, 2, 4))
    k, v = rng.standard_normal((2, 1, 5, 1, 4))
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, do, causal=True, q_pos_offset=-3)
    assert np.all(dq[:, :3] == 0.0)  # rows 0..2 see no key
    dq2, dk2, dv2 = oracle_mod.attention_bwd(q[:, 3:], k, v, do[:, 3:], causal=True, q_pos_offset=0)
    np.testing.assert_allclose(dk, dk2, atol=1e-14)
    np.testing.assert_allclose(dv, dv2, atol=1e-14)
    # no keys at all
    z = oracle_mod.attention_bwd(q, k[:, :0], v[:, :0], do)
    assert np.all(z[0] == 0.0) and z[1].size == 0


@pytest.mark.parametrize("mutation", ["MUT_BWD_NO_D", "MUT_BWD_NO_SCALE", "MUT_BWD_DK_FROM_P"])
def test_planted_backward_mistakes_are_caught(oracle_mod, mutation):
    mut = getattr(oracle_mod, mutation)
    caught = []
    g = read_kv("two_key_example.txt")
    q, k, v, do = _scalar(g["k"], g["v"], g["dO"])
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, do, scale=1.0, mutation=mut)
    caught.append(not np.allclose(dk.ravel(), g["printed_dS"], atol=1e-12))
    b, sq, skv, hq, hkv, d, causal, off, win, scale = AUTOGRAD_CASES[1]
    rng = np.random.default_rng(1)
    q = rng.standard_normal((b, sq, hq, d))
    k = rng.standard_normal((b, skv, hkv, d))
    v = rng.standard_normal((b, skv, hkv, d))
    do = rng.standard_normal((b, sq, hq, d))
    sc = 1.0 / math.sqrt(d)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, do, causal=causal, q_pos_offset=off, scale=sc, mutation=mut)
    tq, tk, tv = _torch_grads(q, k, v, do, sc, _band(sq, skv, causal, off, *win))
    caught.append(not (np.allclose(dq, tq, atol=1e-9) and np.allclose(dk, tk, atol=1e-9)))
    assert any(caught)
