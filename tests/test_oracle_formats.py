"""Pins of the oracle's number formats (BF16, FP32, E4M3, MXFP8) against things other
than itself: torch's and numpy's own conversions, the OCP format points in
tests/golden, and closed-form properties of the MX block rule."""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def test_bf16_rounding_matches_torch_on_ties_and_near_ties():
    # Every BF16 upper half with the low 16 bits at 0, just below/at/above the tie.
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    bits = (hi[:, None] | lows[None, :]).ravel()
    f = _bits_to_f32(bits)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = O.round_bf16(f.astype(np.float64))
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(got[fin], ref[fin])
    # torch overflows to inf exactly where the oracle does
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_rounding_random_f32():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    f = _bits_to_f32(bits)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = O.round_bf16(f.astype(np.float64))
    ok = np.isfinite(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_f32_rounding_matches_numpy():
    rng = np.random.default_rng(2)
    d = rng.standard_normal(1 << 18) * np.exp2(rng.integers(-140, 120, size=1 << 18))
    # exact ties halfway between float32 neighbours
    f = rng.standard_normal(4096).astype(np.float32)
    nxt = np.nextafter(f, np.float32(np.inf))
    ties = (f.astype(np.float64) + nxt.astype(np.float64)) / 2
    d = np.concatenate([d, ties])
    np.testing.assert_array_equal(O.round_f32(d), d.astype(np.float32).astype(np.float64))


def _torch_e4m3_table() -> np.ndarray:
    """Value of each E4M3 code per torch's own float8_e4m3fn decoder."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def test_e4m3_decode_matches_torch_all_codes():
    ref = _torch_e4m3_table()
    got = O.e4m3_decode(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    # sign of zero
    assert math.copysign(1.0, got[0x80]) == -1.0


def test_e4m3_golden_points():
    path = os.path.join(GOLDEN, "e4m3_points.txt")
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code_s, val_s = line.split()
        code, val = int(code_s, 16), float(val_s)
        got = O.lib().orc_e4m3_decode(code)
        if math.isnan(val):
            assert math.isnan(got)
            continue
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (code, got, val)
        assert O.lib().orc_e4m3_encode(val) == code


def test_e4m3_encode_exhaustive_bf16_matches_torch():
    # All 65536 BF16 bit patterns whose value lies within the E4M3 finite range.
    bits = (np.arange(1 << 16, dtype=np.uint32) << 16)
    f = _bits_to_f32(bits)
    f = f[np.isfinite(f) & (np.abs(f) <= 448.0)]
    ref = torch.from_numpy(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(f.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_midpoints_and_neighbours():
    # Midpoints between consecutive finite E4M3 values (from torch's table) and the
    # float32 neighbours on each side: ties go to the even code, the rest to nearest.
    tab = _torch_e4m3_table()[:127]            # codes 0..126, ascending magnitudes
    mids = (tab[:-1] + tab[1:]) / 2
    f32mid = mids.astype(np.float32)
    assert np.array_equal(f32mid.astype(np.float64), mids)   # midpoints exact in f32
    below = np.nextafter(f32mid, np.float32(0))
    above = np.nextafter(f32mid, np.float32(np.inf))
    for arr in (f32mid, below, above, -f32mid, -below, -above):
        ref = torch.from_numpy(arr).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = O.e4m3_encode(arr.astype(np.float64))
        np.testing.assert_array_equal(got, ref)
    # explicit ties: midpoint between codes c and c+1 goes to the even one
    got = O.e4m3_encode(mids)
    lo = np.arange(126)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    np.testing.assert_array_equal(got, expect)


def test_e4m3_saturates():
    for v, c in [(448.0, 0x7E), (449.0, 0x7E), (464.0, 0x7E), (500.0, 0x7E), (1e30, 0x7E),
                 (-470.0, 0xFE), (-1e30, 0xFE)]:
        assert O.lib().orc_e4m3_encode(v) == c, v
    # below half the smallest subnormal rounds to a signed zero
    assert O.lib().orc_e4m3_encode(2.0 ** -11) == 0x00
    assert O.lib().orc_e4m3_encode(-(2.0 ** -11)) == 0x80
    assert O.lib().orc_e4m3_encode(2.0 ** -10) == 0x00          # tie -> even (0)
    assert O.lib().orc_e4m3_encode(3 * 2.0 ** -10) == 0x02      # tie 1.5 -> 2


# ----------------------------------------------------------------------- MXFP8 blocks
def test_mxfp8_scale_for_power_of_two_amax():
    # amax = 2^m exactly -> s = m - 8 -> UE8M0 code m - 8 + 127 (clamped)
    for m in range(-140, 128):
        blk = np.zeros((1, 32))
        blk[0, 5] = 2.0 ** m
        blk[0, 9] = -(2.0 ** (m - 1))
        codes, scales = O.quantize_mxfp8(blk)
        s = min(max(m - 8, -127), 127)
        assert scales[0, 0] == s + 127, m
        if -127 <= m - 8:
            assert codes[0, 5] == 0x78        # 256 = 1.0 * 2^8
            assert codes[0, 9] == 0xF0        # -128


def test_mxfp8_round_trip_of_representable_blocks():
    rng = np.random.default_rng(3)
    for s in (-20, -3, 0, 5, 40):
        codes = rng.integers(0, 127, size=(8, 32)).astype(np.uint8)
        codes[:, 0] = rng.integers(0x78, 0x7F, size=8)      # amax exponent 8 -> scale s
        signs = rng.integers(0, 2, size=(8, 32)).astype(np.uint8) << 7
        codes = codes | signs
        vals = O.e4m3_decode(codes) * 2.0 ** s
        c2, s2 = O.quantize_mxfp8(vals)
        assert np.all(s2 == s + 127)
        # +0 and -0 may both appear; compare values and the non-zero codes
        np.testing.assert_array_equal(O.dequantize_mxfp8(c2, s2), vals)
        nz = (codes & 0x7F) != 0
        np.testing.assert_array_equal(c2[nz], codes[nz])


def test_mxfp8_saturation_and_zero_block():
    blk = np.zeros((2, 32))
    blk[0, 0] = 500.0          # floor(log2 500) = 8 -> s = 0 -> 500 saturates to 448
    blk[0, 1] = 3.0
    codes, scales = O.quantize_mxfp8(blk)
    assert scales[0, 0] == 127 and codes[0, 0] == 0x7E
    assert O.e4m3_decode(codes[0, 1]) == 3.0
    assert scales[1, 0] == 0 and np.all(codes[1] == 0)


def test_mxfp8_error_bound_random():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-30, 30, size=(64, 1)))
    codes, scales = O.quantize_mxfp8(v)
    d = O.dequantize_mxfp8(codes, scales)
    X = np.repeat(np.exp2(scales.astype(np.float64) - 127), 32, axis=1)
    r = np.abs(v) / X
    assert np.all(r < 512)
    sat = r > 464
    # saturated elements land on +-448 X; the rest are within half an E4M3 ulp
    np.testing.assert_array_equal(np.abs(d[sat]), 448 * X[sat])
    ns = ~sat
    bound = np.maximum(np.abs(v[ns]) * 2.0 ** -4, X[ns] * 2.0 ** -10)
    assert np.all(np.abs(d[ns] - v[ns]) <= bound)
    # the block's largest magnitude maps to exponent 8 of E4M3 (codes 0x78..0x7E)
    amax_code = (codes.reshape(64, -1, 32) & 0x7F).max(axis=2)
    assert np.all((amax_code >= 0x78) & (amax_code <= 0x7E))


def test_mxfp8_rows_are_independent():
    rng = np.random.default_rng(5)
    v = rng.standard_normal((16, 128))
    c_all, s_all = O.quantize_mxfp8(v)
    for r in (0, 7, 15):
        c_r, s_r = O.quantize_mxfp8(v[r:r + 1])
        np.testing.assert_array_equal(c_all[r], c_r[0])
        np.testing.assert_array_equal(s_all[r], s_r[0])
