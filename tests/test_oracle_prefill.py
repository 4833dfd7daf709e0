"""Pins for the oracle's paged prefill (CPU only).

oracle_prefill is pinned to a float64 numpy reference that builds the whole
masked score tensor per sequence (different code, precision and order), to
the decode oracle it must reduce to (one query row is a decode over the keys
that row sees, bit for bit), and to closed forms.
"""
import numpy as np
import pytest

from paged_kv_split_gb300 import inputs
from tests import refs
from tests.test_oracle_decode import build_cache

PREFILL_CASES = [
    # (seq_lens, q_lens, Hq, Hkv, D, bs, window)
    ([17, 40], [17, 9], 4, 2, 64, 16, 0),
    ([70, 33, 5], [16, 33, 1], 8, 2, 64, 16, 0),
    ([64, 31], [40, 3], 16, 2, 128, 32, 0),
    ([69, 50], [23, 50], 4, 1, 64, 16, 20),
    ([48], [48], 8, 8, 64, 16, 16),
    ([90, 37], [30, 37], 4, 2, 256, 32, 0),
]


def case_of(idx, seed_base=300):
    lens, qls, hq, hkv, d, bs, w = PREFILL_CASES[idx]
    return inputs.make_prefill_case("pf", lens, qls, hq, hkv, d, bs, seed=seed_base + idx,
                                    sliding_window=w, extra_blocks=2)


def run_prefill(orc, case, kc, vc, kv_dtype, ks, vs, causal=True, window=None):
    w = case.sliding_window if window is None else window
    return orc.prefill(case.q, case.extra["cu_q"], kc, vc, case.block_tables, case.seq_lens,
                       case.num_kv_heads, case.block_size, case.num_blocks, case.scale,
                       causal, w, kv_dtype, ks, vs)


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("idx", range(len(PREFILL_CASES)))
def test_prefill_matches_f64(orc, idx, kv_dtype, causal):
    case = case_of(idx)
    kc, vc, ks, vs = build_cache(orc, case, kv_dtype)
    out, out_f32 = run_prefill(orc, case, kc, vc, kv_dtype, ks, vs, causal)
    kp = refs.dequant_pages(kc, kv_dtype, case.num_blocks, case.block_size, case.num_kv_heads,
                            case.head_dim, ks)
    vp = refs.dequant_pages(vc, kv_dtype, case.num_blocks, case.block_size, case.num_kv_heads,
                            case.head_dim, vs)
    ref = refs.prefill_f64(case.q, case.extra["cu_q"], kp, vp, case.block_tables,
                           case.seq_lens, case.scale, causal, case.sliding_window)
    np.testing.assert_allclose(out_f32, ref, rtol=1e-5, atol=2e-6)
    assert np.array_equal(out, inputs.to_bf16_bits(out_f32))


def _decode_rows(orc, case, kc, vc, kv_dtype, ks, vs, causal):
    """Each query row as its own decode: q = that row, length = its position + 1."""
    cu = case.extra["cu_q"]
    rows = []
    for b in range(case.num_seqs):
        L = int(case.seq_lens[b])
        ql = int(cu[b + 1] - cu[b])
        for i in range(ql):
            p = (L - ql + i) if causal else L - 1
            o, _ = orc.decode(case.q[cu[b] + i][None], kc, vc, case.block_tables[b:b + 1],
                              np.array([p + 1], np.int32), case.num_kv_heads, case.block_size,
                              case.num_blocks, case.scale, case.sliding_window, kv_dtype, ks, vs)
            rows.append(o[0])
    return np.stack(rows)


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
@pytest.mark.parametrize("kv_dtype", [0, 2])
@pytest.mark.parametrize("idx", [0, 3])
def test_rows_equal_decode_bit_for_bit(orc, idx, kv_dtype, causal):
    case = case_of(idx)
    kc, vc, ks, vs = build_cache(orc, case, kv_dtype)
    out, _ = run_prefill(orc, case, kc, vc, kv_dtype, ks, vs, causal)
    assert np.array_equal(out, _decode_rows(orc, case, kc, vc, kv_dtype, ks, vs, causal))


def test_one_query_per_sequence_is_decode(orc):
    case = inputs.make_prefill_case("pf1", [37, 64, 5], [1, 1, 1], 8, 2, 64, 16, seed=41)
    kc, vc, _, _ = build_cache(orc, case, 0)
    out, _ = run_prefill(orc, case, kc, vc, 0, 1.0, 1.0)
    dec, _ = orc.decode(case.q, kc, vc, case.block_tables, case.seq_lens, case.num_kv_heads,
                        case.block_size, case.num_blocks, case.scale)
    assert np.array_equal(out, dec)


def test_first_token_of_a_fresh_prompt_is_its_value(orc):
    """L == q_len, causal: query 0 sees key 0 alone, so its output is bf16(v_0)."""
    case = inputs.make_prefill_case("fresh", [21, 40], [21, 40], 4, 2, 64, 16, seed=42)
    kc, vc, _, _ = build_cache(orc, case, 0)
    out, _ = run_prefill(orc, case, kc, vc, 0, 1.0, 1.0)
    cu = case.extra["cu_q"]
    g = case.num_q_heads // case.num_kv_heads
    for b in range(2):
        v0 = case.value[int(np.sum(case.seq_lens[:b]))]  # token 0 of sequence b, write order
        for h in range(case.num_q_heads):
            assert np.array_equal(out[cu[b], h], v0[h // g])


def test_constant_values_give_the_constant(orc):
    case = inputs.make_prefill_case("const", [50, 19], [30, 19], 8, 2, 64, 16, seed=43,
                                    sliding_window=12)
    c = inputs.to_bf16_bits(np.float32(0.3125))
    case.value[:] = c
    kc, vc, _, _ = build_cache(orc, case, 0)
    for causal in (True, False):
        out, _ = run_prefill(orc, case, kc, vc, 0, 1.0, 1.0, causal)
        assert np.all(out == c)


def test_query_longer_than_sequence_is_refused(orc):
    case = inputs.make_prefill_case("bad", [10], [10], 4, 2, 64, 16, seed=44)
    kc, vc, _, _ = build_cache(orc, case, 0)
    lens = case.seq_lens.copy()
    lens[0] = 9
    with pytest.raises(ValueError):
        orc.prefill(case.q, case.extra["cu_q"], kc, vc, case.block_tables, lens,
                    case.num_kv_heads, case.block_size, case.num_blocks, case.scale)
