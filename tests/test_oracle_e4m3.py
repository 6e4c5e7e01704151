"""Pins of the e4m3 reference (oracle/e4m3.py) to the published format: known codes,
round trips of every finite code, ties to even, saturation, and the block scales."""
import numpy as np

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
