"""Pins of the fp64 oracle to facts outside itself.

Each test checks the oracle against something the pages print, a closed form,
an invariant, or an independent library routine, so that a plausible mistake
(a dropped term, a wrong sign or index, a transposed operand) fails at least
one of them.  The mutation tests at the end plant such mistakes in the oracle
and check that they are caught.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from golden_io import read_kv, read_mask_pictures

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _qkv(rng, b, sq, skv, hq, hkv, d, std=1.0):
    q = rng.standard_normal((b, sq, hq, d)) * std
    k = rng.standard_normal((b, skv, hkv, d)) * std
    v = rng.standard_normal((b, skv, hkv, d)) * std
    return q, k, v


def _scalar_problem(scores, values):
    """d = 1 problem whose scaled scores (scale = 1) are `scores`."""
    n = len(scores)
    q = np.ones((1, 1, 1, 1))
    k = np.asarray(scores, dtype=np.float64).reshape(1, n, 1, 1)
    v = np.asarray(values, dtype=np.float64).reshape(1, n, 1, 1)
    return q, k, v


# ---------------------------------------------------------------- worked examples


def test_online_merge_worked_example(oracle_mod):
    g = read_kv("online_merge_example.txt")
    scores = list(g["block1_scores"]) + list(g["block2_scores"])
    values = list(g["block1_values"]) + list(g["block2_values"])
    q, k, v = _scalar_problem(scores, values)
    tol = 0.5 * 10 ** (-int(g["printed_digits"]))
    o, lse = oracle_mod.attention(q, k, v, scale=1.0)
    assert abs(o[0, 0] - g["printed_O"]) <= tol
    # LSE is the logsumexp of the scores (library routine).
    assert abs(lse[0] - scipy.special.logsumexp(scores)) < 1e-14
    # The page's own two-block merge, and every other tiling, land on the same value.
    for tile in (1, 2, 3, 4):
        ot, lt = oracle_mod.attention_tiled(q, k, v, scale=1.0, tile=tile)
        assert abs(ot[0, 0] - o[0, 0]) < 1e-13
        assert abs(lt[0] - lse[0]) < 1e-13


def test_two_key_worked_example(oracle_mod):
    g = read_kv("two_key_example.txt")
    # O with v = [2, 6]
    q, k, v = _scalar_problem(g["k"], g["v"])
    o, lse = oracle_mod.attention(q, k, v)  # d = 1, default scale 1/sqrt(1)
    assert abs(o[0, 0] - g["printed_O"]) < 1e-14
    assert abs(lse[0] - math.log(4.0)) < 1e-14  # ln(1 + 3)
    # P itself: use one-hot values so that O = P.
    q2 = np.array([1.0, 0.0]).reshape(1, 1, 1, 2)
    k2 = np.array([[g["k"][0], 0.0], [g["k"][1], 0.0]]).reshape(1, 2, 1, 2)
    v2 = np.eye(2).reshape(1, 2, 1, 2)
    p, _ = oracle_mod.attention(q2, k2, v2, scale=1.0)
    np.testing.assert_allclose(p[0], g["printed_P"], atol=1e-15)


def test_combine_exercise_split_blocks(oracle_mod):
    """Exercise 1 of the hs-black page: block A has s = 0, v = 10; block B has s = ln 3, v = 2.
    Weights are e^0 : e^ln3 = 1 : 3, so O = (10 + 3*2) / 4 = 4; averaging the two local
    outputs would give 6 (answer worked by hand)."""
    o, lse = oracle_mod.combine(np.array([[[10.0]], [[2.0]]]), np.array([[0.0], [math.log(3.0)]]))
    assert abs(o[0, 0] - 4.0) < 1e-14
    assert abs(lse[0] - math.log(4.0)) < 1e-14
    assert abs(o[0, 0] - 6.0) > 1.0
    # the same numbers through the split model
    q, k, v = _scalar_problem([0.0, math.log(3.0)], [10.0, 2.0])
    ot, lt = oracle_mod.attention_tiled(q, k, v, scale=1.0, tile=1, num_splits=2)
    assert abs(ot[0, 0] - 4.0) < 1e-14 and abs(lt[0] - math.log(4.0)) < 1e-14


def test_combine_all_empty_and_single(oracle_mod):
    o, lse = oracle_mod.combine(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(o == 0.0) and np.all(np.isneginf(lse))
    rng = np.random.default_rng(5)
    op = rng.standard_normal((1, 3, 4))
    lp = rng.standard_normal((1, 3))
    o, lse = oracle_mod.combine(op, lp)
    np.testing.assert_allclose(o, op[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, lp[0], rtol=0, atol=1e-15)


# ---------------------------------------------------------------- masks


def _visibility_from_outputs(oracle_mod, sq, skv, causal=True, off=None, mutation=0):
    """Recover which keys each row sees: equal scores (K = 0) and one-hot values
    make O[i] = indicator(visible) / count."""
    q = np.ones((1, sq, 1, skv))
    k = np.zeros((1, skv, 1, skv))
    v = np.eye(skv).reshape(1, skv, 1, skv)
    o, lse = oracle_mod.attention(q, k, v, causal=causal, q_pos_offset=off, mutation=mutation)
    return (o > 0).astype(int), o, lse


@pytest.mark.parametrize("case", read_mask_pictures())
def test_causal_mask_pictures(oracle_mod, case):
    sq, skv, rows = case
    vis, o, lse = _visibility_from_outputs(oracle_mod, sq, skv)
    assert vis.tolist() == rows
    for i, row in enumerate(rows):
        n = sum(row)
        if n == 0:  # fully masked row: exactly 0 and -inf
            assert np.all(o[i] == 0.0) and np.isneginf(lse[i])
        else:
            np.testing.assert_allclose(o[i][np.array(row) == 1], 1.0 / n, rtol=0, atol=1e-15)
            assert abs(lse[i] - math.log(n)) < 1e-14


def test_tail_tile_example(oracle_mod):
    g = read_kv("tail_tile_example.txt")
    n, tile, row = int(g["N"]), int(g["tile"]), int(g["row"])
    second = [j for j in range(tile, 2 * tile) if oracle_mod.visible(row, j, n, True, 0)]
    assert second == [int(g["valid_keys_in_second_block"])]
    rng = np.random.default_rng(11)
    q, k, v = _qkv(rng, 1, n, n, 1, 1, 3)
    o, lse = oracle_mod.attention(q, k, v, causal=True)
    ot, lt = oracle_mod.attention_tiled(q, k, v, tile=tile, causal=True)
    np.testing.assert_allclose(ot, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lt, lse, rtol=0, atol=1e-12)


def test_fully_masked_rows_negative_offset(oracle_mod):
    rng = np.random.default_rng(3)
    q, k, v = _qkv(rng, 2, 6, 5, 2, 1, 4)
    o, lse = oracle_mod.attention(q, k, v, causal=True, q_pos_offset=-3)
    rows = oracle_mod.all_rows(2, 2, 6)
    masked = rows[:, 2] + (-3) < 0
    assert np.all(o[masked] == 0.0) and np.all(np.isneginf(lse[masked]))
    assert np.all(np.isfinite(lse[~masked]))
    # skv = 0: every row is fully masked
    o0, l0 = oracle_mod.attention(q, k[:, :0], v[:, :0])
    assert np.all(o0 == 0.0) and np.all(np.isneginf(l0))


# ---------------------------------------------------------------- library routines


def _sdpa_reference(q, k, v, causal, scale):
    """torch's fp64 CPU attention with its own log-sum-exp output ([b, s, h, d] layout in/out)."""
    qt = torch.from_numpy(q).permute(0, 2, 1, 3).contiguous()
    kt = torch.from_numpy(k).permute(0, 2, 1, 3).contiguous()
    vt = torch.from_numpy(v).permute(0, 2, 1, 3).contiguous()
    g = qt.shape[1] // kt.shape[1]
    kt = kt.repeat_interleave(g, dim=1)
    vt = vt.repeat_interleave(g, dim=1)
    out, lse = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(qt, kt, vt, 0.0, causal,
                                                                           attn_mask=None, scale=scale)[:2]
    return out.permute(0, 2, 1, 3).numpy(), lse.numpy()  # o [b, s, h, d], lse [b, h, s]


SDPA_CASES = [
    # b, sq, skv, hq, hkv, d, causal
    (2, 7, 7, 2, 2, 8, False),
    (1, 9, 9, 4, 2, 16, True),
    (2, 5, 11, 3, 3, 5, False),
    (1, 33, 33, 4, 1, 64, True),
    (1, 17, 40, 2, 1, 32, False),
]


@pytest.mark.parametrize("case", SDPA_CASES)
def test_matches_library_attention(oracle_mod, case):
    b, sq, skv, hq, hkv, d, causal = case
    rng = np.random.default_rng(sum(case[:6]))
    q, k, v = _qkv(rng, b, sq, skv, hq, hkv, d, std=1.5)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle_mod.attention(q, k, v, causal=causal, q_pos_offset=0 if causal else None)
    ro, rl = _sdpa_reference(q, k, v, causal, scale)
    rows = oracle_mod.all_rows(b, hq, sq)
    np.testing.assert_allclose(o, ro[rows[:, 0], rows[:, 2], rows[:, 1]], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl[rows[:, 0], rows[:, 1], rows[:, 2]], rtol=0, atol=1e-12)


def test_d1_is_softmax_weighted_mean(oracle_mod):
    rng = np.random.default_rng(7)
    s = rng.standard_normal(13) * 3
    vals = rng.standard_normal(13)
    q, k, v = _scalar_problem(s, vals)
    o, lse = oracle_mod.attention(q, k, v, scale=1.0)
    assert abs(o[0, 0] - scipy.special.softmax(s) @ vals) < 1e-14
    assert abs(lse[0] - scipy.special.logsumexp(s)) < 1e-14


# ---------------------------------------------------------------- invariants


def test_key_shift_invariance(oracle_mod):
    """Adding one vector u to every key shifts row i's scores by scale*(q_i . u): O is
    unchanged and LSE moves by exactly that amount (softmax is shift-invariant)."""
    rng = np.random.default_rng(21)
    b, sq, skv, hq, hkv, d = 2, 6, 9, 4, 2, 8
    q, k, v = _qkv(rng, b, sq, skv, hq, hkv, d)
    u = rng.standard_normal(d)
    scale = 0.37
    o, lse = oracle_mod.attention(q, k, v, causal=True, scale=scale)
    o2, lse2 = oracle_mod.attention(q, k + u, v, causal=True, scale=scale)
    rows = oracle_mod.all_rows(b, hq, sq)
    shift = scale * (q[rows[:, 0], rows[:, 2], rows[:, 1]] @ u)
    finite = np.isfinite(lse)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2[finite], lse[finite] + shift[finite], rtol=0, atol=1e-12)


def test_value_scaling(oracle_mod):
    rng = np.random.default_rng(22)
    q, k, v = _qkv(rng, 1, 5, 8, 2, 2, 4)
    o, lse = oracle_mod.attention(q, k, v)
    o2, lse2 = oracle_mod.attention(q, k, 3.5 * v)
    np.testing.assert_allclose(o2, 3.5 * o, rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(lse2, lse)


# ---------------------------------------------------------------- tiled model vs definition


@pytest.mark.parametrize("causal", [False, True])
def test_tiled_matches_direct_small(oracle_mod, causal):
    rng = np.random.default_rng(100 + causal)
    for n in range(1, 10):
        q, k, v = _qkv(rng, 1, n, n, 2, 1, 3, std=2.0)
        o, lse = oracle_mod.attention(q, k, v, causal=causal)
        for tile in (1, 2, 3, 4, 8):
            for ns in (1, 2, 3):
                ot, lt = oracle_mod.attention_tiled(q, k, v, tile=tile, num_splits=ns, causal=causal)
                np.testing.assert_allclose(ot, o, rtol=0, atol=1e-12)
                np.testing.assert_allclose(lt, lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("off", [-4, -1, 0, 3, 50])
def test_tiled_matches_direct_offsets(oracle_mod, off):
    rng = np.random.default_rng(200 + off)
    q, k, v = _qkv(rng, 2, 7, 10, 4, 2, 5)
    o, lse = oracle_mod.attention(q, k, v, causal=True, q_pos_offset=off)
    for tile in (1, 3, 4):
        ot, lt = oracle_mod.attention_tiled(q, k, v, tile=tile, num_splits=2, causal=True, q_pos_offset=off)
        np.testing.assert_allclose(ot, o, rtol=0, atol=1e-12)
        np.testing.assert_array_equal(np.isneginf(lt), np.isneginf(lse))
        fin = np.isfinite(lse)
        np.testing.assert_allclose(lt[fin], lse[fin], rtol=0, atol=1e-12)


def test_empty_split_marker(oracle_mod):
    """A split whose key range this row cannot see yields (0, -inf) and leaves the merge unchanged."""
    rng = np.random.default_rng(9)
    q, k, v = _qkv(rng, 1, 2, 12, 1, 1, 4)
    o, lse, op, lp = oracle_mod.attention_tiled(q, k, v, tile=2, num_splits=3, causal=True, q_pos_offset=0,
                                                return_partials=True)
    # row 0 sees key 0 only, row 1 keys 0..1 -> splits 1 and 2 are empty for both rows
    assert np.all(op[1:] == 0.0) and np.all(np.isneginf(lp[1:]))
    od, ld = oracle_mod.attention(q, k, v, causal=True, q_pos_offset=0)
    np.testing.assert_allclose(o, od, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, ld, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- split heuristic


def test_split_heuristic_page_example(oracle_mod):
    g = read_kv("split_heuristic.txt")
    units, slots = int(g["units"]), int(g["slots"])
    nd = int(g["printed_digits"])
    assert round(oracle_mod.split_efficiency(units, slots, 2), nd) == g["efficiency_2"]
    assert round(oracle_mod.split_efficiency(units, slots, 3), nd) == g["efficiency_3"]
    assert oracle_mod.num_splits(units, slots, nblk=1024) == int(g["chosen_splits"])


def test_split_heuristic_bounds(oracle_mod):
    assert oracle_mod.num_splits(10, 100, nblk=1) == 1
    assert oracle_mod.num_splits(1, 4, nblk=8, max_splits=128) == 4
    assert oracle_mod.num_splits(400, 100, nblk=64) == 1
    for units in (1, 7, 48, 64, 300):
        s = oracle_mod.num_splits(units, 152, nblk=512)
        best = max(oracle_mod.split_efficiency(units, 152, t) for t in range(1, 129))
        assert oracle_mod.split_efficiency(units, 152, s) >= 0.85 * best
        assert all(oracle_mod.split_efficiency(units, 152, t) < 0.85 * best for t in range(1, s))


# ---------------------------------------------------------------- sliding window


def _band_reference(q, k, v, off, wl, wr, scale, causal=False):
    """torch's fp64 CPU attention with a band mask from tril/triu of a ones matrix (library routines)."""
    sq, skv = q.shape[1], k.shape[1]
    band = torch.ones(sq, skv, dtype=torch.bool)
    if wr >= 0:
        band = band.tril(off + wr)
    if wl >= 0:
        band = band.triu(off - wl)
    if causal:
        band = band & torch.ones(sq, skv, dtype=torch.bool).tril(off)
    add = torch.zeros(sq, skv, dtype=torch.float64).masked_fill(~band, float("-inf"))
    qt = torch.from_numpy(q).permute(0, 2, 1, 3).contiguous()
    kt = torch.from_numpy(k).permute(0, 2, 1, 3).contiguous()
    vt = torch.from_numpy(v).permute(0, 2, 1, 3).contiguous()
    g = qt.shape[1] // kt.shape[1]
    kt, vt = kt.repeat_interleave(g, dim=1), vt.repeat_interleave(g, dim=1)
    out, lse = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(qt, kt, vt, 0.0, False, attn_mask=add,
                                                                           scale=scale)[:2]
    return out.permute(0, 2, 1, 3).numpy(), lse.numpy(), band.numpy()


WINDOW_CASES = [
    # b, sq, skv, hq, hkv, d, off, wl, wr, causal
    (1, 9, 9, 2, 1, 8, 0, 3, 0, False),
    (2, 7, 12, 2, 2, 16, 5, 2, 4, False),
    (1, 10, 10, 4, 2, 8, 0, 4, -1, True),
    (1, 6, 20, 2, 2, 8, 14, -1, 3, False),
    (1, 11, 11, 2, 1, 8, 0, 0, 0, False),
]


@pytest.mark.parametrize("case", WINDOW_CASES)
def test_window_matches_library_band_mask(oracle_mod, case):
    b, sq, skv, hq, hkv, d, off, wl, wr, causal = case
    rng = np.random.default_rng(sum(case[:6]) + 17)
    q, k, v = _qkv(rng, b, sq, skv, hq, hkv, d, std=1.3)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle_mod.attention(q, k, v, causal=causal, q_pos_offset=off, window=(wl, wr))
    ro, rl, band = _band_reference(q, k, v, off, wl, wr, scale, causal)
    rows = oracle_mod.all_rows(b, hq, sq)
    np.testing.assert_allclose(o, ro[rows[:, 0], rows[:, 2], rows[:, 1]], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl[rows[:, 0], rows[:, 1], rows[:, 2]], rtol=0, atol=1e-12)
    for i in range(sq):
        for j in range(skv):
            assert oracle_mod.visible(i, j, skv, causal, off, window=(wl, wr)) == bool(band[i, j])
    for tile in (1, 3, 4):
        ot, lt = oracle_mod.attention_tiled(q, k, v, tile=tile, num_splits=2, causal=causal, q_pos_offset=off,
                                            window=(wl, wr))
        np.testing.assert_allclose(ot, o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lt, lse, rtol=0, atol=1e-12)


def test_window_right_zero_is_causal(oracle_mod):
    """The page's causal flag is the window (unbounded, 0): same visibility everywhere."""
    for (sq, skv) in ((2, 5), (5, 2), (7, 7)):
        off = skv - sq
        for i in range(sq):
            for j in range(skv):
                assert oracle_mod.visible(i, j, skv, True, off) == oracle_mod.visible(i, j, skv, False, off,
                                                                                      window=(-1, 0))


# ---------------------------------------------------------------- planted mistakes


def _pins_pass(oracle_mod, mutation) -> bool:
    """Run the pins above against a mutated oracle; True iff all still pass."""
    try:
        g = read_kv("online_merge_example.txt")
        q, k, v = _scalar_problem(list(g["block1_scores"]) + list(g["block2_scores"]),
                                  list(g["block1_values"]) + list(g["block2_values"]))
        for tile in (1, 2, 4):
            ot, _ = oracle_mod.attention_tiled(q, k, v, scale=1.0, tile=tile, mutation=mutation)
            assert abs(ot[0, 0] - g["printed_O"]) <= 5e-4
        for sq, skv, rows in read_mask_pictures():
            vis, _, _ = _visibility_from_outputs(oracle_mod, sq, skv, mutation=mutation)
            assert vis.tolist() == rows
        for case in SDPA_CASES:
            b, sq, skv, hq, hkv, d, causal = case
            rng = np.random.default_rng(sum(case[:6]))
            q, k, v = _qkv(rng, b, sq, skv, hq, hkv, d, std=1.5)
            o, lse = oracle_mod.attention(q, k, v, causal=causal, q_pos_offset=0 if causal else None,
                                          mutation=mutation)
            ro, rl = _sdpa_reference(q, k, v, causal, 1.0 / math.sqrt(d))
            rows = oracle_mod.all_rows(b, hq, sq)
            np.testing.assert_allclose(o, ro[rows[:, 0], rows[:, 2], rows[:, 1]], rtol=0, atol=1e-12)
    except AssertionError:
        return False
    return True


def test_pins_pass_for_correct_oracle(oracle_mod):
    assert _pins_pass(oracle_mod, 0)


@pytest.mark.parametrize("mutation", ["MUT_NO_ALPHA_ON_O", "MUT_NO_ALPHA_ON_L", "MUT_NO_SCALE",
                                      "MUT_STRICT_CAUSAL"])
def test_planted_mistakes_are_caught(oracle_mod, mutation):
    assert not _pins_pass(oracle_mod, getattr(oracle_mod, mutation))
