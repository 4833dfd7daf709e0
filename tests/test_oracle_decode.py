"""Pins for the oracle's decode attention (CPU only).

The oracle walks the block table token by token in fp32. It is pinned to
torch's scaled_dot_product_attention in float64 over the same keys gathered
contiguously by numpy (different code, different precision, different order),
and to closed forms and invariants that the definition implies.
"""
import math

import numpy as np
import pytest

from paged_kv_split_gb300 import inputs
from tests import refs


def build_cache(orc, case, kv_dtype):
    """Write the case's K/V through the oracle; returns caches and scales."""
    h, d, bs, nb = case.num_kv_heads, case.head_dim, case.block_size, case.num_blocks
    k_scale = v_scale = 1.0
    if kv_dtype == 1:
        k_scale = orc.fp8_scale(orc.absmax_bf16(case.key))
        v_scale = orc.fp8_scale(orc.absmax_bf16(case.value))
    n = orc.cache_bytes(kv_dtype, nb, bs, h, d)
    kc = np.zeros(n, np.uint8)
    vc = np.zeros(n, np.uint8)
    orc.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping, h, d, bs, nb, kv_dtype,
                          k_scale, v_scale)
    return kc, vc, k_scale, v_scale


def run_oracle(orc, case, kc, vc, kv_dtype, k_scale, v_scale, window=None):
    w = case.sliding_window if window is None else window
    return orc.decode(case.q, kc, vc, case.block_tables, case.seq_lens, case.num_kv_heads,
                      case.block_size, case.num_blocks, case.scale, w, kv_dtype, k_scale,
                      v_scale)


def run_sdpa(case, kc, vc, kv_dtype, k_scale, v_scale, window=None):
    w = case.sliding_window if window is None else window
    kp = refs.dequant_pages(kc, kv_dtype, case.num_blocks, case.block_size, case.num_kv_heads,
                            case.head_dim, k_scale)
    vp = refs.dequant_pages(vc, kv_dtype, case.num_blocks, case.block_size, case.num_kv_heads,
                            case.head_dim, v_scale)
    return refs.sdpa_f64(case.q, kp, vp, case.block_tables, case.seq_lens, case.scale, w)


SMALL_CASES = [
    # (seq_lens, Hq, Hkv, D, bs, window)
    ([17, 40], 4, 2, 64, 16, 0),
    ([1, 70, 33], 8, 2, 64, 16, 0),
    ([70, 5], 8, 8, 128, 16, 0),
    ([64, 31], 16, 2, 128, 32, 0),
    ([69, 50, 12], 4, 1, 64, 16, 20),
    ([48], 16, 1, 64, 16, 16),
]


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("idx", range(len(SMALL_CASES)))
def test_oracle_matches_sdpa_f64(orc, kv_dtype, idx):
    lens, hq, hkv, d, bs, w = SMALL_CASES[idx]
    case = inputs.make_case("s", lens, hq, hkv, d, bs, seed=100 + idx, sliding_window=w,
                            extra_blocks=3)
    kc, vc, ks, vs = build_cache(orc, case, kv_dtype)
    out, out_f32 = run_oracle(orc, case, kc, vc, kv_dtype, ks, vs)
    ref = run_sdpa(case, kc, vc, kv_dtype, ks, vs)
    np.testing.assert_allclose(out_f32, ref, rtol=1e-5, atol=2e-6)
    # the bf16 output is the round-to-nearest-even of the fp32 value
    assert np.array_equal(out, inputs.to_bf16_bits(out_f32))


def test_paged_layout_is_invisible(orc):
    """Permuting the page pool and remapping block_tables gives identical output."""
    case = inputs.make_case("p", [37, 64, 5], 8, 2, 64, 16, seed=7, extra_blocks=4)
    kc, vc, _, _ = build_cache(orc, case, 0)
    out1, _ = run_oracle(orc, case, kc, vc, 0, 1.0, 1.0)
    perm = inputs.permutation(99, case.num_blocks)
    pb = orc.page_bytes(0, case.block_size, case.num_kv_heads, case.head_dim)
    kp = kc.reshape(case.num_blocks, pb)
    vp = vc.reshape(case.num_blocks, pb)
    # page i moves to slot perm[i]
    kc2 = np.empty_like(kp)
    vc2 = np.empty_like(vp)
    kc2[perm] = kp
    vc2[perm] = vp
    bt2 = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1)
    case.block_tables = bt2.astype(np.int32)
    out2, _ = run_oracle(orc, case, kc2.ravel(), vc2.ravel(), 0, 1.0, 1.0)
    assert np.array_equal(out1, out2)


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
def test_length_one_returns_v0(orc, kv_dtype):
    case = inputs.make_case("l1", [1, 1], 8, 4, 128, 16, seed=8)
    kc, vc, ks, vs = build_cache(orc, case, kv_dtype)
    out, out_f32 = run_oracle(orc, case, kc, vc, kv_dtype, ks, vs)
    vp = refs.dequant_pages(vc, kv_dtype, case.num_blocks, 16, 4, 128, vs)
    for b in range(2):
        v0 = vp[case.block_tables[b, 0], 0]               # [Hkv, D]
        want = np.repeat(v0, 2, axis=0)                    # G = 2
        assert np.array_equal(out_f32[b], want.astype(np.float32))


def test_constant_v_returns_constant(orc):
    case = inputs.make_case("cv", [45, 3], 8, 2, 64, 16, seed=9)
    c_bits = inputs.to_bf16_bits(np.array([0.7109375], np.float32))[0]  # exact in bf16
    case.value[:] = c_bits
    kc, vc, _, _ = build_cache(orc, case, 0)
    out, out_f32 = run_oracle(orc, case, kc, vc, 0, 1.0, 1.0)
    np.testing.assert_allclose(out_f32, 0.7109375, rtol=2e-6)
    assert np.all(out == c_bits)


def test_zero_query_gives_mean_of_values(orc):
    case = inputs.make_case("q0", [29, 64], 4, 2, 64, 16, seed=10)
    case.q[:] = 0
    kc, vc, _, _ = build_cache(orc, case, 0)
    _, out_f32 = run_oracle(orc, case, kc, vc, 0, 1.0, 1.0)
    vp = refs.dequant_pages(vc, 0, case.num_blocks, 16, 2, 64)
    for b in range(2):
        V = refs.gather_sequence(vp, case.block_tables[b], int(case.seq_lens[b]))
        mean = V.mean(axis=0)                              # [Hkv, D]
        np.testing.assert_allclose(out_f32[b], np.repeat(mean, 2, axis=0), rtol=1e-5, atol=1e-6)


def test_two_tokens_sigmoid_weight(orc):
    case = inputs.make_case("two", [2], 2, 1, 64, 16, seed=11)
    kc, vc, _, _ = build_cache(orc, case, 0)
    _, out_f32 = run_oracle(orc, case, kc, vc, 0, 1.0, 1.0)
    q = refs.bf16_to_f64(case.q)[0]                        # [2, D]
    K = refs.bf16_to_f64(case.key)[:, 0]                   # [2, D]
    V = refs.bf16_to_f64(case.value)[:, 0]
    for h in range(2):
        s0, s1 = case.scale * (q[h] @ K[0]), case.scale * (q[h] @ K[1])
        w0 = 1.0 / (1.0 + math.exp(-(s0 - s1)))
        want = w0 * V[0] + (1.0 - w0) * V[1]
        np.testing.assert_allclose(out_f32[0, h], want, rtol=1e-5, atol=1e-6)


def test_window_at_least_length_is_no_window(orc):
    case = inputs.make_case("w", [40, 17], 4, 2, 64, 16, seed=12)
    kc, vc, _, _ = build_cache(orc, case, 0)
    full, _ = run_oracle(orc, case, kc, vc, 0, 1.0, 1.0, window=0)
    for w in (40, 41, 1000):
        got, _ = run_oracle(orc, case, kc, vc, 0, 1.0, 1.0, window=w)
        assert np.array_equal(full, got)


def test_window_equals_attention_over_last_w_tokens(orc):
    """A window of W over L is full attention over the last W tokens as their own sequence."""
    L, W, bs = 53, 20, 16
    case = inputs.make_case("w", [L], 4, 2, 64, bs, seed=13)
    kc, vc, _, _ = build_cache(orc, case, 0)
    win, _ = run_oracle(orc, case, kc, vc, 0, 1.0, 1.0, window=W)
    sub = inputs.make_case("w2", [W], 4, 2, 64, bs, seed=13)
    sub.q = case.q
    sub.key = case.key[L - W:]
    sub.value = case.value[L - W:]
    kc2, vc2, _, _ = build_cache(orc, sub, 0)
    ref, _ = run_oracle(orc, sub, kc2, vc2, 0, 1.0, 1.0, window=0)
    assert np.array_equal(win, ref)


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
def test_large_scores_stay_finite(orc, kv_dtype):
    case = inputs.make_case("big", [70, 33], 8, 2, 64, 16, seed=14)
    q = refs.bf16_to_f64(case.q) * 100.0
    case.q = inputs.to_bf16_bits(q.astype(np.float32))
    kc, vc, ks, vs = build_cache(orc, case, kv_dtype)
    out, out_f32 = run_oracle(orc, case, kc, vc, kv_dtype, ks, vs)
    assert np.all(np.isfinite(out_f32))
    ref = run_sdpa(case, kc, vc, kv_dtype, ks, vs)
    np.testing.assert_allclose(out_f32, ref, rtol=1e-4, atol=1e-4)


def test_fp8_scales_are_separate_for_k_and_v(orc):
    """k_scale multiplies scores, v_scale multiplies outputs (closed form with L = 1)."""
    case = inputs.make_case("sc", [1], 2, 1, 64, 16, seed=15)
    kc, vc, ks, vs = build_cache(orc, case, 1)
    _, out_a = run_oracle(orc, case, kc, vc, 1, ks, vs)
    _, out_b = run_oracle(orc, case, kc, vc, 1, ks, 2.0 * vs)
    np.testing.assert_array_equal(out_b, 2.0 * out_a)
