"""Pins for the oracle's INT8 quantiser (CPU only).

The page gives x_q = round(x / scale) + zero_point and x = (x_q - zero_point) *
scale ("cs336 lecture 10" notes, Quantization). The readings taken (per
(token, kv_head) row; range widened to contain 0; scale = (max - min) / 255;
zero_point = -128 - round(min / scale); round half to even) are pinned here by
hand-worked rows, exact end points and the round-trip error bound.
"""
import numpy as np
import pytest

import oracle


def test_hand_worked_row_with_unit_scale():
    # min -1, max 254 -> scale = 255/255 = 1 exactly; zp = -128 - round(-1) = -127
    x = np.array([-1.0, 0.0, 2.5, 3.5, -0.5, 254.0, 0.5, 1.5], np.float32)
    codes, scale, zp = oracle.quantize_row(x)
    assert scale == 1.0 and zp == -127
    # round half to even: 2.5 -> 2, 3.5 -> 4, -0.5 -> -0, 0.5 -> 0, 1.5 -> 2
    assert codes.tolist() == [-128, -127, -125, -123, -127, 127, -127, -125]


def test_hand_worked_row_all_positive():
    # min is widened to 0, max 51 -> scale 0.2 (fp32), zp = -128
    x = np.array([0.0, 51.0, 25.5, 10.0], np.float32)
    codes, scale, zp = oracle.quantize_row(x)
    assert scale == np.float32(51.0) / np.float32(255.0)
    assert zp == -128
    assert codes[0] == -128 and codes[1] == 127
    # 25.5 / 0.2 = 127.5 (fp32 quotient), half to even -> 128 - 128 = 0
    q = np.float32(25.5) / np.float32(scale)
    assert codes[2] == int(np.rint(q)) - 128


def test_all_negative_and_zero_rows():
    codes, scale, zp = oracle.quantize_row(np.array([-2.0, -1.0, 0.0], np.float32))
    assert zp == 127 and codes.tolist()[0] == -128 and codes.tolist()[2] == 127
    codes, scale, zp = oracle.quantize_row(np.zeros(16, np.float32))
    assert scale == 1.0 and zp == -128 and (codes == -128).all()


@pytest.mark.parametrize("seed", range(5))
def test_end_points_zero_and_round_trip_bound(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        d = int(rng.choice([64, 128]))
        x = (rng.standard_normal(d) * rng.choice([1e-3, 1.0, 50.0])).astype(np.float32)
        codes, scale, zp = oracle.quantize_row(x)
        mn, mx = min(x.min(), 0.0), max(x.max(), 0.0)
        assert codes[np.argmin(x)] == -128 or x.min() > 0
        # the max lands on 127 or one below it (both roundings are half-even)
        assert codes[np.argmax(x)] in (126, 127) or x.max() < 0
        # 0 maps to the zero point, and dequantises to exactly 0
        c0, s0, z0 = oracle.quantize_row(np.concatenate([x, [0.0]]).astype(np.float32))
        assert c0[-1] == z0
        # round trip: |deq(q(x)) - x| <= scale/2 plus fp32 rounding of the ops
        deq = oracle.dequantize(codes, scale, zp)
        bound = 0.5 * scale * (1 + 1e-6) + np.abs(x) * 2.0 ** -22
        assert (np.abs(deq - x) <= bound).all()
        # monotone
        order = np.argsort(x, kind="stable")
        assert (np.diff(codes[order].astype(int)) >= 0).all()


def test_planted_rounding_mistake_is_caught():
    # round-half-away-from-zero instead of half-to-even disagrees on the hand row
    x = np.array([-1.0, 0.0, 2.5, 3.5, -0.5, 254.0, 0.5, 1.5], np.float32)
    codes, scale, zp = oracle.quantize_row(x)
    away = (np.sign(x) * np.floor(np.abs(x) + 0.5)).astype(int) + zp
    assert not np.array_equal(codes.astype(int), away)


# ---- FP8 E4M3 (page 2 "ybb.press" §5.2: FP8 KV cache, per-head scales) -------

def test_e4m3_decode_table_matches_torch_float8():
    """All 256 codes decoded from the format definition equal torch's
    float8_e4m3fn values (NaN where torch has NaN)."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert ((dec == ref) | (np.isnan(dec) & np.isnan(ref))).all()
    assert np.nanmax(dec) == 448.0 and np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert dec[0x01] == 2.0 ** -9 and dec[0x08] == 2.0 ** -6    # smallest subnormal / normal


def test_e4m3_encode_matches_torch_below_overflow():
    """Round to nearest, ties to even, against torch's cast, on random values,
    exact ties between neighbours, and the subnormal range."""
    import torch
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.normal(size=20000) * 40, rng.normal(size=5000) * 0.01,
                        rng.uniform(-460, 460, size=5000)]).astype(np.float32)
    vals = np.unique(np.abs(oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))))
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)   # exact ties (representable)
    x = np.concatenate([x, mids, -mids, vals.astype(np.float32)])
    x = x[np.abs(x) < 464]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_e4m3_encode_saturates_and_round_trips():
    """Magnitudes past the largest finite value saturate to +-448 (the
    satfinite convention; a plain cast would give NaN from 464 up), NaN stays
    NaN, and every finite code round-trips."""
    big = np.array([448, 463.99, 464, 1e9, np.inf, -464, -np.inf], np.float32)
    assert oracle.e4m3_encode(big).tolist() == [0x7E] * 5 + [0xFE] * 2
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(finite).astype(np.float32)),
                          finite)


def test_planted_e4m3_bias_mistake_is_caught():
    """A decoder with exponent bias 8 instead of 7 disagrees with torch: the
    table pin above would fail."""
    import torch
    codes = np.arange(0x08, 0x78, dtype=np.uint8)
    wrong = oracle.e4m3_decode(codes) / 2.0                    # bias off by one
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert not np.array_equal(wrong, ref)
