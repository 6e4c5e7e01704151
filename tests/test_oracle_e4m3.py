"""Pins of the e4m3 reference (oracle/e4m3.py) to the published format: known codes,
round trips of every finite code, ties to even, saturation, and the block scales."""
import numpy as np
import pytest

from oracle import e4m3


def test_known_codes():
    known = {0x00: 0.0, 0x38: 1.0, 0xB8: -1.0, 0x40: 2.0, 0x30: 0.5, 0x7E: 448.0, 0xFE: -448.0,
             0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x3C: 1.5}
    for code, val in known.items():
        assert e4m3.decode(np.array([code], dtype=np.uint8))[0] == val, hex(code)
    assert np.isnan(e4m3.decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(e4m3.encode(e4m3.decode(codes).astype(np.float32)), codes)  # 0x80 is -0
    # the sign survives rounding to zero
    assert e4m3.encode(np.array([-0.0], dtype=np.float32))[0] == 0x80
    assert e4m3.encode(np.array([-1e-9], dtype=np.float32))[0] == 0x80


def test_ties_to_even_and_saturation():
    assert e4m3.encode(np.float32(1.0625)) == 0x38       # between 1.0 (m=0) and 1.125 (m=1)
    assert e4m3.encode(np.float32(1.1875)) == 0x3A       # between 1.125 (m=1) and 1.25 (m=2)
    assert e4m3.encode(np.float32(1.0626)) == 0x39
    assert e4m3.encode(np.float32(500.0)) == 0x7E
    assert e4m3.encode(np.float32(-1e6)) == 0xFE
    assert e4m3.encode(np.float32(2.0 ** -10)) == 0x00   # half of the smallest subnormal: tie to even (zero)
    assert e4m3.encode(np.float32(3 * 2.0 ** -11)) == 0x01  # 0.75 * 2^-9: nearest subnormal is 2^-9
    assert e4m3.encode(np.float32(3 * 2.0 ** -10)) == 0x02  # 1.5 * 2^-9: tie between 0x01 and 0x02, even wins


def test_block_scales_and_bounds():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((2, 300, 3, 64)) * np.array([1.0, 100.0, 1e-3])[None, None, :, None]).astype(np.float32)
    x[1, 128:256, 2, :] = 0.0  # an all-zero block
    codes, ds = e4m3.quantize_blocks(x)
    assert ds.shape == (2, 3, 3)
    assert ds[1, 2, 1] == 1.0
    amax = np.abs(x[0, :128, 1, :]).max()
    assert ds[0, 1, 0] == np.float32(amax) / np.float32(448)
    xd = e4m3.dequantize_blocks(codes, ds)
    # relative error of a normal-range e4m3 value is at most 2^-4
    big = np.abs(x) > 2.0 ** -6 * np.repeat(ds, 128, axis=2)[:, :, :300].transpose(0, 2, 1)[..., None]
    assert np.all(np.abs(xd - x)[big] <= 2.0 ** -4 * np.abs(x)[big] * 1.0000001)
    # the largest value of every block maps to 448 exactly
    assert np.abs(e4m3.decode(codes[0, :128, 1, :])).max() == 448.0
    codes_h, ds_h = e4m3.quantize_blocks(x, per_head=True)
    assert ds_h.shape == (2, 3)
    np.testing.assert_allclose(e4m3.dequantize_blocks(codes_h, ds_h, per_head=True), x,
                               atol=float(np.abs(x).max()) / 16)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_block_scales_at_every_head_width(d):
    """One scale per 128 rows of one (batch, head), whatever the head width."""
    rng = np.random.default_rng(d)
    x = (rng.standard_normal((1, 257, 2, d)) * 3.0).astype(np.float32)
    codes, ds = e4m3.quantize_blocks(x)
    assert codes.shape == x.shape and ds.shape == (1, 2, 3)
    for h in range(2):
        for k, (r0, r1) in enumerate(((0, 128), (128, 256), (256, 257))):
            assert ds[0, h, k] == np.float32(np.abs(x[0, r0:r1, h, :]).max()) / np.float32(448)
            assert np.abs(e4m3.decode(codes[0, r0:r1, h, :])).max() == 448.0


def _model_e4m3_forward(qx, kx, vx, scale, causal, off, window):
    """A step-by-step fp64 model of what rounding P to e4m3 does in the 8-bit forward pass:
    per row, key blocks of 128 from the highest, the reference maximum moved only when a
    block's maximum exceeds it by more than 8 log2 units, p = 2^(x - m_ref) rounded to e4m3
    for the P V product, l summed from the unrounded p, O = o / l rounded to bf16."""
    import torch

    b, sq, hq, d = qx.shape
    skv, hkv = kx.shape[1], kx.shape[2]
    g = hq // hkv
    wl, wr = window
    out = np.zeros((b * hq * sq, d))
    r = 0
    for bi in range(b):
        for h in range(hq):
            for i in range(sq):
                x = kx[bi, :, h // g, :] @ qx[bi, i, h, :] * scale / np.log(2.0)
                j = np.arange(skv)
                vis = np.ones(skv, dtype=bool)
                if causal:
                    vis &= j <= i + off
                if wl >= 0:
                    vis &= j >= i + off - wl
                if wr >= 0:
                    vis &= j <= i + off + wr
                x = np.where(vis, x, -np.inf)
                m_ref, l, o = -np.inf, 0.0, np.zeros(d)
                for n in range((skv + 127) // 128 - 1, -1, -1):
                    blk = x[n * 128:(n + 1) * 128]
                    bm = blk.max()
                    if bm > m_ref + 8:
                        alpha = 2.0 ** (m_ref - bm) if np.isfinite(m_ref) else 0.0
                        o, l, m_ref = o * alpha, l * alpha, bm
                    if not np.isfinite(m_ref):
                        continue
                    p = 2.0 ** (blk - m_ref)
                    pr = e4m3.decode(e4m3.encode(p.astype(np.float32)))
                    l += p.sum()
                    o += pr @ vx[bi, n * 128:n * 128 + len(blk), h // g, :]
                if l > 0:
                    out[r] = torch.tensor(o / l).to(torch.bfloat16).double().numpy()
                r += 1
    return out


@pytest.mark.parametrize("d,causal,window,vmean", [
    (64, True, None, 0.0), (128, False, (60, 10), 0.0), (256, True, None, 1.5), (64, False, None, -2.0),
])
def test_rounding_bound_holds_for_a_model_of_p_rounding(d, causal, window, vmean):
    """The tolerance of the GPU e4m3 check (parity_util.e4m3_rounding_bound, every term from
    the oracle) bounds the model above on causal, windowed and shifted-V inputs at every head
    width, and stays tight enough that a doubled O would fail it on shifted-V inputs."""
    from parity_util import e4m3_rounding_bound

    import oracle

    rng = np.random.default_rng(d + (7 if causal else 0))
    b, sq, skv, hq, hkv = 1, 150, 300, 2, 1
    x = lambda *shape: rng.standard_normal(shape).astype(np.float32)  # noqa: E731
    q, k, v = x(b, sq, hq, d), x(b, skv, hkv, d), x(b, skv, hkv, d) + np.float32(vmean)
    qx = e4m3.dequantize_blocks(*e4m3.quantize_blocks(q))
    kx = e4m3.dequantize_blocks(*e4m3.quantize_blocks(k))
    vc, vd = e4m3.quantize_blocks(v, per_head=True)
    vx = e4m3.dequantize_blocks(vc, vd, per_head=True)
    scale = 1.0 / np.sqrt(d)
    off = skv - sq
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle.attention(qx, kx, vx, causal=causal, q_pos_offset=off, scale=scale, rows=rows,
                                    window=window if window else (-1, -1))
    tol = e4m3_rounding_bound(qx, kx, vx, causal, off, window, o_ref, l_ref, rows, scale)
    model = _model_e4m3_forward(qx, kx, vx, scale, causal, off, window if window else (-1, -1))
    vis = ~np.isneginf(l_ref)
    assert np.all(np.abs(model[vis] - o_ref[vis]) <= tol[vis])
    if vmean:
        assert np.mean(np.abs(o_ref[vis]) > tol[vis]) > 0.9
