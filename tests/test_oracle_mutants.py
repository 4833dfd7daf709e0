"""The pins have teeth: plant plausible mistakes in a copy of the oracle.

Each mutant is the oracle source with one edit (a dropped term, a wrong
index, a wrong rounding rule...), compiled on the CPU into a temporary
library. The test passes only if at least one of the named pins fails on it.
The real oracle is never modified.
"""
import os

import pytest

import oracle
from tests import test_oracle_cache as TC
from tests import test_oracle_codecs as TX
from tests import test_oracle_decode as TD


def _sdpa_all(orc):
    for kv in (0, 1, 2):
        for i in range(len(TD.SMALL_CASES)):
            TD.test_oracle_matches_sdpa_f64(orc, kv, i)


def _e4m3_out_all(orc):
    from tests import test_oracle_e4m3_out as TE
    for kv in (0, 1, 2):
        for sc in (0.0078125, 0.013, 3.0):
            TE.test_length_one_is_the_encoded_value(orc, kv, sc)
        TE.test_codes_encode_the_fp32_output(orc, kv)


def _prefill_all(orc):
    from tests import test_oracle_prefill as TP
    for idx in range(len(TP.PREFILL_CASES)):
        for causal in (True, False):
            TP.test_prefill_matches_f64(orc, idx, 0, causal)


MUTANTS = [
    ("gqa kv head index", "const int32_t g = h / group;", "const int32_t g = h % num_kv_heads;",
     [_sdpa_all]),
    ("window start off by one", "len > sliding_window) ? len - sliding_window : 0",
     "len > sliding_window) ? len - sliding_window + 1 : 0", [_sdpa_all]),
    ("score scale dropped", "s[j - lo] = scale * dot;", "s[j - lo] = dot;", [_sdpa_all]),
    ("softmax max not subtracted", "s[j] = std::exp(s[j] - m);", "s[j] = std::exp(s[j]);",
     [lambda o: [TD.test_large_scores_stay_finite(o, k) for k in (0, 1, 2)]]),
    ("row offset within page", "read_row(k_cache, kv_dtype, page, j % block_size, g,",
     "read_row(k_cache, kv_dtype, page, (j + 1) % block_size, g,", [_sdpa_all]),
    ("v dequantised with k_scale", "v_scale, vrow.data()", "k_scale, vrow.data()", [_sdpa_all]),
    ("nvfp4 read layout token-major",
     "const uint8_t* data = base + (static_cast<int64_t>(head) * bs + off) * (d / 2);",
     "const uint8_t* data = base + (static_cast<int64_t>(off) * hkv + head) * (d / 2);",
     [_sdpa_all]),
    ("round half away from zero", "return (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;",
     "return fl + 1.0;", [TX.test_e4m3_encode_matches_torch_in_range]),
    ("e4m3 subnormal quantum", "round_half_even(a * 512.0)", "round_half_even(a * 256.0)",
     [TX.test_e4m3_encode_matches_torch_in_range]),
    ("e4m3 exponent bias", "mag = std::ldexp(1.0f + static_cast<float>(man) / 8.0f, ex - 7);",
     "mag = std::ldexp(1.0f + static_cast<float>(man) / 8.0f, ex - 8);",
     [TX.test_e4m3_decode_all_codes_match_torch]),
    ("e2m1 mantissa step", "double n = round_half_even(std::ldexp(a, 1 - e));",
     "double n = round_half_even(std::ldexp(a, 2 - e));", [TX.test_e2m1_encode_matches_bruteforce]),
    ("bf16 ties away", "(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)",
     [TX.test_bf16_round_matches_torch]),
    ("nvfp4 nibble order", "static_cast<uint8_t>(lo | (hi << 4))",
     "static_cast<uint8_t>(hi | (lo << 4))", [TC.test_nvfp4_cache_matches_definition]),
    ("nvfp4 scale divisor", "e4m3_code(amax / 6.0f)", "e4m3_code(amax / 4.0f)",
     [TC.test_nvfp4_cache_matches_definition]),
    ("fp8 calibration divisor", "amax / 448.0f : 1.0f", "amax / 240.0f : 1.0f",
     [TX.test_fp8_scale_is_absmax_over_448]),
    ("prefill causal bound excludes the query's own key", "const int32_t hi = pos + 1;",
     "const int32_t hi = pos;", [_prefill_all]),
    ("prefill first query position", "causal ? len - q_len + i : len - 1;",
     "causal ? len - q_len + i - 1 : len - 1;", [_prefill_all]),
    ("prefill window measured from the last key", "hi > sliding_window) ? hi - sliding_window",
     "len > sliding_window) ? len - sliding_window", [_prefill_all]),
    ("prefill q row offset", "const int64_t qrow = static_cast<int64_t>(cu_q[b]) + i;",
     "const int64_t qrow = static_cast<int64_t>(cu_q[b]) + i / 2;", [_prefill_all]),
    ("fp8 quantise multiplies", "return std::isnan(x) ? x : x / s;",
     "return std::isnan(x) ? x : x * s;", [TC.test_fp8_cache_matches_torch_e4m3]),
    ("e4m3 output scale multiplies", "out_codes[i] = e4m3_code(quotient(o[i], out_scale));",
     "out_codes[i] = e4m3_code(o[i] * out_scale);", [_e4m3_out_all]),
    ("e4m3 output encodes the bf16-rounded value",
     "out_codes[i] = e4m3_code(quotient(o[i], out_scale));",
     "out_codes[i] = e4m3_code(quotient(bf16_value(out_bf16[i]), out_scale));",
     [_e4m3_out_all]),
]


@pytest.mark.parametrize("name,old,new,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new, checks):
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
    mutated = tmp_path / "mutant.cpp"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutated), str(tmp_path / "libmutant.so"))
    mutant = oracle.Oracle(lib)
    caught = False
    for check in checks:
        try:
            check(mutant)
        except (AssertionError, ValueError):
            caught = True
            break
    assert caught, f"no pin caught the mutant: {name}"
    os.remove(lib)
