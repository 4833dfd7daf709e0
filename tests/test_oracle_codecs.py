"""Pins for the oracle's number formats (CPU only).

The oracle's E4M3 / E2M1 / bf16 codecs are checked against routines that do
not share its code: torch's float8_e4m3fn and bfloat16 conversions, the OCP
MX value table for E2M1, and brute-force nearest-value searches.
"""
import numpy as np
import pytest
import torch

from tests import refs


def _midpoints_and_neighbours(values: np.ndarray) -> np.ndarray:
    v = np.unique(values[np.isfinite(values)].astype(np.float64))
    mids = ((v[:-1] + v[1:]) / 2).astype(np.float32)
    out = [v.astype(np.float32), mids,
           np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf))]
    x = np.concatenate(out)
    return np.concatenate([x, -x])


def _random_log_uniform(n, lo_exp, hi_exp, seed):
    rng = np.random.default_rng(seed)
    mag = np.exp2(rng.uniform(lo_exp, hi_exp, n)).astype(np.float32)
    sign = np.where(rng.random(n) < 0.5, -1, 1).astype(np.float32)
    return mag * sign


# ---- E4M3 -----------------------------------------------------------------
def test_e4m3_decode_all_codes_match_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = refs.e4m3_decode(codes)
    got = np.array([orc.e4m3_value(c) for c in codes])
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.all(np.isnan(got[nan]))
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decode_landmarks(orc):
    # largest finite, smallest normal, smallest subnormal, one, negative zero
    assert orc.e4m3_value(0x7E) == 448.0
    assert orc.e4m3_value(0x08) == 2.0 ** -6
    assert orc.e4m3_value(0x01) == 2.0 ** -9
    assert orc.e4m3_value(0x38) == 1.0
    assert orc.e4m3_value(0xFE) == -448.0
    v = orc.e4m3_value(0x80)
    assert v == 0.0 and np.signbit(v)


def test_e4m3_encode_matches_torch_in_range(orc):
    grid = refs.e4m3_decode(np.arange(256, dtype=np.uint8))
    x = np.concatenate([
        _midpoints_and_neighbours(grid),
        _random_log_uniform(200_000, -14, np.log2(464.0), 1),
        np.array([0.0, -0.0, 2.0 ** -10, -(2.0 ** -10), 2.0 ** -11, 1e-30, 464.0, -464.0],
                 np.float32),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 464.0]
    got = orc.e4m3_codes(x)
    ref = refs.e4m3_encode_torch(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def test_e4m3_encode_matches_bruteforce(orc):
    grid = refs.e4m3_decode(np.arange(256, dtype=np.uint8))
    x = np.concatenate([
        _midpoints_and_neighbours(grid),
        _random_log_uniform(50_000, -14, 12, 2),
        np.array([np.inf, -np.inf, 1e38, -1e38, 480.0, 500.0], np.float32),
    ]).astype(np.float32)
    got = orc.e4m3_codes(x)
    ref = np.concatenate([refs.brute_e4m3(c) for c in np.array_split(x, 16)])
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def test_e4m3_encode_saturation_and_nan(orc):
    for v in [448.0, 463.99, 464.0, 465.0, 1e4, 3.0e38, np.inf]:
        assert orc.e4m3_code(v) == 0x7E
        assert orc.e4m3_code(-v) == 0xFE
    assert orc.e4m3_code(np.nan) == 0x7F
    assert orc.e4m3_code(-np.float32(np.nan)) == 0xFF
    assert orc.e4m3_code(-0.0) == 0x80
    assert orc.e4m3_code(-1e-30) == 0x80


# ---- E2M1 -----------------------------------------------------------------
def test_e2m1_decode_matches_ocp_table(orc):
    for c in range(16):
        mag = refs.E2M1_TABLE[c & 7]
        want = -mag if c & 8 else mag
        got = orc.e2m1_value(c)
        assert got == want
        assert np.signbit(got) == bool(c & 8)


def test_e2m1_encode_matches_bruteforce(orc):
    x = np.concatenate([
        _midpoints_and_neighbours(refs.E2M1_TABLE),
        _random_log_uniform(100_000, -6, 4, 3),
        np.array([0.0, -0.0, 6.0, 6.5, 7.0, 100.0, np.inf, -np.inf, 1e-40], np.float32),
    ]).astype(np.float32)
    got = orc.e2m1_codes(x)
    ref = np.concatenate([refs.brute_e2m1(c) for c in np.array_split(x, 8)])
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def test_e2m1_ties_go_to_even(orc):
    # value -> code at each midpoint of the grid
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for v, c in ties.items():
        assert orc.e2m1_code(v) == c, v
        assert orc.e2m1_code(-v) == c | 8, v
    assert orc.e2m1_code(np.nan) == 7


# ---- bf16 -----------------------------------------------------------------
def test_bf16_round_matches_torch(orc):
    rng = np.random.default_rng(4)
    bits = rng.integers(0, 2 ** 32, 20_000, dtype=np.uint64).astype(np.uint32)
    # force ties: low half exactly 0x8000
    ties = (bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    x = np.concatenate([bits, ties]).view(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_round(v) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_value_is_top_half(orc):
    for b in [0x0000, 0x3F80, 0xBF80, 0x7F7F, 0x0001, 0x8000]:
        want = refs.bf16_to_f64(np.array([b], np.uint16))[0]
        assert orc.bf16_value(b) == want


# ---- quantised round trips --------------------------------------------------
@pytest.mark.parametrize("scale", [1.0, 0.25, 4.0, 2.0 ** -7])
def test_fp8_round_trip_is_identity_on_codes(orc, scale):
    """q(deq(c)) == c for every finite code when the scale is a power of two."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = refs.e4m3_decode(codes) * scale
    back = orc.e4m3_codes((vals / scale).astype(np.float32))
    assert np.array_equal(back, codes)


def test_fp8_quantise_error_within_half_spacing(orc):
    x = _random_log_uniform(50_000, -8, 8.7, 5)
    codes = orc.e4m3_codes(x)
    deq = refs.e4m3_decode(codes)
    grid = np.sort(np.unique(np.abs(refs.e4m3_decode(np.arange(127, dtype=np.uint8)))))
    a = np.abs(x.astype(np.float64))
    i = np.clip(np.searchsorted(grid, a), 1, len(grid) - 1)
    spacing = grid[i] - grid[i - 1]
    assert np.all(np.abs(a - np.abs(deq)) <= spacing / 2 + 0.0)
    assert np.all(np.signbit(deq) == np.signbit(x))


def test_fp8_scale_is_absmax_over_448(orc):
    bits = np.array([0x3F80, 0xC2C8, 0x4000, 0x7FC0], np.uint16)  # 1, -100, 2, NaN
    amax = orc.absmax_bf16(bits)
    assert amax == 100.0
    assert orc.fp8_scale(amax) == np.float32(100.0) / np.float32(448.0)
    assert orc.fp8_scale(0.0) == 1.0
