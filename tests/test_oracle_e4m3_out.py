"""Pins for the oracle's decode with E4M3 output codes (CPU only).

Reading (the pages name an "E4M3 output variant" without defining it):
code = E4M3(o / out_scale), o the fp32 attention output before any bf16
rounding, IEEE fp32 division, the cache encoder's rounding (nearest, ties to
even, saturating). Pinned by cases whose o is known exactly: a length-1
sequence (o = v0) against a brute-force nearest-grid search, constant V
against hand-derived codes, and, for random cases, against the brute-force
encoding of oracle_decode's own fp32 output (which catches a bf16 rounding
slipped in before the encode)."""
import numpy as np
import pytest

from paged_kv_split_gb300 import inputs
from tests import refs
from tests.test_oracle_decode import build_cache


def _codes(orc, case, kc, vc, out_scale, kv_dtype=0, ks=1.0, vs=1.0):
    return orc.decode_e4m3_out(case.q, kc, vc, case.block_tables, case.seq_lens,
                               case.num_kv_heads, case.block_size, case.num_blocks, case.scale,
                               out_scale, case.sliding_window, kv_dtype, ks, vs)


@pytest.mark.parametrize("out_scale", [1.0, 0.0078125, 0.013, 3.0, 1e-3, 2.0 ** -12])
@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
def test_length_one_is_the_encoded_value(orc, kv_dtype, out_scale):
    case = inputs.make_case("e4o_l1", [1, 1, 1], 8, 4, 128, 16, seed=31)
    kc, vc, ks, vs = build_cache(orc, case, kv_dtype)
    codes = _codes(orc, case, kc, vc, out_scale, kv_dtype, ks, vs)
    vp = refs.dequant_pages(vc, kv_dtype, case.num_blocks, 16, 4, 128, vs)
    for b in range(case.num_seqs):
        v0 = vp[case.block_tables[b, 0], 0].astype(np.float32)     # [Hkv, D], exact
        # o = (0 + e_0 v_0) / e_0: the accumulation starts at +0, so a stored -0
        # (an NVFP4 code 0x8) comes out as +0, as IEEE addition gives
        o = np.float32(0.0) + np.repeat(v0, 2, axis=0)
        want = refs.brute_e4m3(o / np.float32(out_scale))
        assert np.array_equal(codes[b].ravel(), want)


@pytest.mark.parametrize("c,out_scale,code", [
    (1.5, 0.25, 0x4C),          # 6.0 = 1.5 * 2^2: exponent field 9, mantissa 4
    (-1.5, 0.25, 0xCC),         # the sign bit
    (1.5, 1.0 / 512, 0x7E),     # 768 saturates to 448
    (1.5, 1024.0, 0x01),        # 0.75 of the subnormal quantum 2^-9 rounds up to 1
    (0.0, 3.0, 0x00),
    (0.7109375, 0.7109375 / 8, 0x50),  # 8.0 = 2^3: field 10, mantissa 0
])
def test_constant_values_encode_as_derived_by_hand(orc, c, out_scale, code):
    case = inputs.make_case("e4o_cv", [45, 3], 8, 2, 64, 16, seed=32)
    case.value[:] = inputs.to_bf16_bits(np.array([c], np.float32))[0]
    kc, vc, _, _ = build_cache(orc, case, 0)
    codes = _codes(orc, case, kc, vc, np.float32(out_scale))
    assert np.all(codes == code)


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
def test_codes_encode_the_fp32_output(orc, kv_dtype):
    case = inputs.make_case("e4o_rnd", [17, 300, 64], 16, 4, 128, 16, seed=33,
                            sliding_window=0)
    kc, vc, ks, vs = build_cache(orc, case, kv_dtype)
    _, out_f32 = orc.decode(case.q, kc, vc, case.block_tables, case.seq_lens, case.num_kv_heads,
                            case.block_size, case.num_blocks, case.scale, 0, kv_dtype, ks, vs)
    for out_scale in (1.0 / 448, 0.002, 0.031):
        codes = _codes(orc, case, kc, vc, out_scale, kv_dtype, ks, vs)
        want = refs.brute_e4m3(out_f32.ravel() / np.float32(out_scale))
        assert np.array_equal(codes.ravel(), want)


@pytest.mark.parametrize("bad", [0.0, -1.0, float("inf"), float("nan")])
def test_bad_output_scale_is_refused(orc, bad):
    case = inputs.make_case("e4o_bad", [5], 4, 2, 64, 16, seed=34)
    kc, vc, _, _ = build_cache(orc, case, 0)
    with pytest.raises(ValueError):
        _codes(orc, case, kc, vc, bad)
