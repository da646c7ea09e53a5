"""Pins for the oracle's NVFP4 format layer (E2M1 elements, an E4M3 scale per 16
elements along K, one FP32 scale per tensor).

"Смесь котят: как Cursor создал открытое ядро, ускоряющее обучение ИИ до 2.4 раз"
names NVFP4, beside MXFP8, as a format of the team's earlier training kernels
without defining it; the element type is the OCP MX specification's FP4 E2M1 and the two-level
scaling is NVIDIA's published NVFP4 recipe (tensor scale amax / (6 * 448)).
"""
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_points.txt")
MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _golden():
    pts = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            c, v = line.split()
            pts.append((int(c, 16), float(v)))
    return pts


def test_e2m1_decode_matches_format_table():
    pts = _golden()
    assert len(pts) == 16
    got = O.e2m1_decode(np.array([c for c, _ in pts], dtype=np.uint8))
    for (c, v), g in zip(pts, got):
        assert g == v and np.signbit(g) == np.signbit(v), hex(c)


def test_e2m1_encode_roundtrips_every_code():
    vals = O.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert np.array_equal(O.e2m1_encode(vals), np.arange(16, dtype=np.uint8))


def _nearest_even_brute(v):
    """Brute force over the eight magnitudes: nearest, ties to the code whose
    mantissa bit is 0, magnitudes past 6 saturate."""
    a = min(abs(v), 6.0)
    d = np.abs(MAGS - a)
    best = np.flatnonzero(d == d.min())
    code = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return code | (8 if np.signbit(v) else 0)


def test_e2m1_encode_is_round_to_nearest_even_with_saturation():
    rng = np.random.default_rng(3)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    vals = np.concatenate([ties, -ties, rng.uniform(-8, 8, 400), [6.0, 6.5, 7.0, 1e30, -1e30, 0.0, -0.0,
                                                                   1e-30, -1e-30, 0.2500001, 0.2499999]])
    got = O.e2m1_encode(vals)
    want = np.array([_nearest_even_brute(v) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, want)


def _exact_blocks(rng, rows, K, jmax):
    """Blocks of 16 that are E2M1 values times 2^j, each holding a +-6 so that its
    block amax is 6*2^j; the tensor amax is 6*2^jmax."""
    codes = rng.integers(0, 16, size=(rows, K)).astype(np.uint8)
    nb = K // 16
    j = rng.integers(jmax - 12, jmax + 1, size=(rows, nb))
    j[0, 0] = jmax
    for r in range(rows):
        for b in range(nb):
            p = rng.integers(0, 16)
            codes[r, b * 16 + p] = 0x7 | (codes[r, b * 16 + p] & 8)
    x = O.e2m1_decode(codes) * np.repeat(np.ldexp(1.0, j), 16, axis=1)
    return x, codes, j


@pytest.mark.parametrize("jmax", [0, 5, -7])
def test_nvfp4_reproduces_exactly_representable_blocks(jmax):
    rng = np.random.default_rng(11 + jmax)
    rows, K = 6, 96
    x, codes, j = _exact_blocks(rng, rows, K, jmax)
    q, s, st = O.quantize_nvfp4(x)
    # tensor scale: amax / (6 * 448), one FP32 rounding
    assert st == float(np.float32(6.0 * 2.0 ** jmax / 2688.0))
    # element codes: the constructed codes, two per byte, lower element in the low nibble
    assert np.array_equal(q & 15, codes[:, 0::2])
    assert np.array_equal(q >> 4, codes[:, 1::2])
    # block scales: E4M3 codes of 448 * 2^(j - jmax)
    e4 = {c: O.lib().orc_e4m3_decode(c) for c in range(256)}
    for r in range(rows):
        for b in range(K // 16):
            assert e4[int(s[r, b])] == 448.0 * 2.0 ** (j[r, b] - jmax)
    back = O.dequantize_nvfp4(q, s, st)
    np.testing.assert_allclose(back, x, rtol=2 ** -22, atol=0)


def test_nvfp4_zero_blocks_and_zero_tensor():
    x = np.zeros((2, 32))
    q, s, st = O.quantize_nvfp4(x)
    assert st == 1.0 and not q.any() and not s.any()
    x[1, 20] = -3.0
    q, s, st = O.quantize_nvfp4(x)
    assert not q[0].any() and not s[0].any()           # all-zero row: zero codes and scales
    assert not s[1, 0] and not q[1, :8].any()          # all-zero block beside a nonzero one
    assert O.dequantize_nvfp4(q, s, st)[1, 20] == pytest.approx(-3.0, rel=2 ** -20)


@pytest.mark.parametrize("seed", [0, 1])
def test_nvfp4_error_bound_and_scale_range(seed):
    """Where a block's scale is a normal E4M3 number, each element's error is at
    most one scale unit d (half the widest E2M1 step) and d * 6 is the block amax
    within E4M3's rounding; the largest block scale sits at E4M3's top (448).
    Blocks far below the tensor amax fall to subnormal or zero scales."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((8, 256)) * np.exp(rng.uniform(-6, 6, size=(8, 1)))).astype(np.float32)
    x[7] *= np.float32(1e-7)                        # a row whose block scales underflow
    x = x.astype(np.float64)
    q, s, st = O.quantize_nvfp4(x)
    back = O.dequantize_nvfp4(q, s, st)
    dec = np.vectorize(O.lib().orc_e4m3_decode)(s)
    assert dec.max() == 448.0
    normal = np.repeat(dec >= 2.0 ** -6, 16, axis=1)
    d = np.repeat(dec * st, 16, axis=1)
    assert normal.sum() > x.size // 4
    assert np.all((np.abs(back - x) <= d * (1 + 2 ** -20))[normal])
    amax_b = np.abs(x).reshape(8, 16, 16).max(axis=2)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = amax_b / (6.0 * dec * st)
    assert np.all(np.abs(ratio[dec >= 2.0 ** -6] - 1) <= 2 ** -4 + 1e-6)
    tiny = amax_b / 6.0 / st < 2.0 ** -10          # below half the smallest subnormal
    assert tiny[7].all()
    assert np.all(s[tiny] == 0) and np.all(back.reshape(8, 16, 16)[tiny] == 0)
