"""Pins for the oracle's cache write (CPU only).

Placement is checked by reading the pages back through numpy reshapes of the
documented layout; values through torch's own conversions (bf16 copy, E4M3)
and a brute-force E2M1 search.
"""
import numpy as np
import pytest

from paged_kv_split_gb300 import inputs
from tests import refs

SENTINEL = 0xA5


def _fresh_caches(orc, kv_dtype, nb, bs, h, d):
    n = orc.cache_bytes(kv_dtype, nb, bs, h, d)
    return np.full(n, SENTINEL, np.uint8), np.full(n, SENTINEL, np.uint8)


def test_page_bytes(orc):
    assert orc.page_bytes(0, 16, 8, 128) == 16 * 8 * 128 * 2
    assert orc.page_bytes(1, 16, 8, 128) == 16 * 8 * 128
    # NVFP4: 8 KiB data + 1 KiB scales, already a multiple of 128
    assert orc.page_bytes(2, 16, 8, 128) == 8192 + 1024
    # 16*1*16/2 = 128 data + 16 scale bytes -> padded to 256
    assert orc.page_bytes(2, 16, 1, 16) == 256


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
def test_slot_placement_and_untouched_slots(orc, kv_dtype):
    nb, bs, h, d = 6, 16, 2, 64
    T = 20
    key = inputs.normal_bf16(11, (T, h, d))
    value = inputs.normal_bf16(12, (T, h, d))
    # scattered slots, two padding tokens (-1) that must be skipped
    slots = inputs.permutation(13, nb * bs)[:T].astype(np.int32)
    slots[[3, 17]] = -1
    kc, vc = _fresh_caches(orc, kv_dtype, nb, bs, h, d)
    orc.reshape_and_cache(key, value, kc, vc, slots, h, d, bs, nb, kv_dtype, 0.5, 0.25)
    pb = orc.page_bytes(kv_dtype, bs, h, d)
    written = set()
    for t in range(T):
        if slots[t] < 0:
            continue
        written.add(int(slots[t]))
    # every byte that belongs to an unwritten slot keeps the sentinel
    for which, cache in ((0, kc), (1, vc)):
        pages = cache.reshape(nb, pb)
        for s in range(nb * bs):
            page, row = divmod(s, bs)
            if kv_dtype == 2:
                data_bytes, _ = refs.nvfp4_geometry(bs, h, d)
                rows = [pages[page, (hh * bs + row) * (d // 2):(hh * bs + row + 1) * (d // 2)]
                        for hh in range(h)]
                rows += [pages[page, data_bytes + (hh * bs + row) * (d // 16):
                               data_bytes + (hh * bs + row + 1) * (d // 16)] for hh in range(h)]
                chunk = np.concatenate(rows)
            else:
                esz = 2 if kv_dtype == 0 else 1
                chunk = pages[page, row * h * d * esz:(row + 1) * h * d * esz]
            if s in written:
                assert not np.all(chunk == SENTINEL)
            else:
                assert np.all(chunk == SENTINEL), (which, s)


def test_bf16_cache_is_a_copy(orc):
    nb, bs, h, d = 5, 16, 2, 64
    c = inputs.make_case("t", [33, 30], 4, h, d, bs, seed=20)
    kc, vc = _fresh_caches(orc, 0, c.num_blocks, bs, h, d)
    orc.reshape_and_cache(c.key, c.value, kc, vc, c.slot_mapping, h, d, bs, c.num_blocks, 0)
    kp = kc.view(np.uint16).reshape(c.num_blocks, bs, h, d)
    vp = vc.view(np.uint16).reshape(c.num_blocks, bs, h, d)
    s = c.slot_mapping.astype(np.int64)
    assert np.array_equal(kp[s // bs, s % bs], c.key)
    assert np.array_equal(vp[s // bs, s % bs], c.value)


def test_fp8_cache_matches_torch_e4m3(orc):
    bs, h, d = 16, 2, 128
    c = inputs.make_case("t", [40, 25], 4, h, d, bs, seed=21)
    k_scale = orc.fp8_scale(orc.absmax_bf16(c.key))
    v_scale = orc.fp8_scale(orc.absmax_bf16(c.value))
    kc, vc = _fresh_caches(orc, 1, c.num_blocks, bs, h, d)
    orc.reshape_and_cache(c.key, c.value, kc, vc, c.slot_mapping, h, d, bs, c.num_blocks, 1,
                          k_scale, v_scale)
    s = c.slot_mapping.astype(np.int64)
    for cache, x, sc in ((kc, c.key, k_scale), (vc, c.value, v_scale)):
        pages = cache.reshape(c.num_blocks, bs, h, d)
        xf = refs.bf16_to_f64(x).astype(np.float32) / np.float32(sc)   # IEEE fp32 division
        assert np.max(np.abs(xf)) <= 448.0 * (1 + 2 ** -20)
        assert np.array_equal(pages[s // bs, s % bs], refs.e4m3_encode_torch(xf))


def test_nvfp4_cache_matches_definition(orc):
    bs, h, d = 16, 2, 64
    c = inputs.make_case("t", [40, 25], 4, h, d, bs, seed=22)
    # add structure: an all-zero group, a tiny-amax group, a group of ties
    key = c.key.copy()
    key[0, 0, :16] = 0
    key[1, 0, :16] = inputs.to_bf16_bits(np.full(16, 1e-4, np.float32))
    key[2, 1, 16:32] = inputs.to_bf16_bits(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 2,
                                                    np.float32))
    kc, vc = _fresh_caches(orc, 2, c.num_blocks, bs, h, d)
    orc.reshape_and_cache(key, c.value, kc, vc, c.slot_mapping, h, d, bs, c.num_blocks, 2)
    data_bytes, stride = refs.nvfp4_geometry(bs, h, d)
    s = c.slot_mapping.astype(np.int64)
    for cache, x in ((kc, key), (vc, c.value)):
        pages = cache.reshape(c.num_blocks, stride)
        packed = pages[:, :data_bytes].reshape(c.num_blocks, h, bs, d // 2)
        scales = pages[:, data_bytes:data_bytes + bs * h * d // 16].reshape(c.num_blocks, h, bs,
                                                                            d // 16)
        got_packed = packed[s // bs, :, s % bs]          # [T, h, d/2]
        got_scales = scales[s // bs, :, s % bs]          # [T, h, d/16]
        xf = refs.bf16_to_f64(x).astype(np.float32).reshape(len(s), h, d // 16, 16)
        amax = np.max(np.abs(xf), axis=-1)
        want_scales = refs.e4m3_encode_torch(amax / np.float32(6.0))
        assert np.array_equal(got_scales, want_scales)
        sdec = refs.e4m3_decode(want_scales).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            y = xf / sdec[..., None]
        codes = refs.brute_e2m1(y.ravel()).reshape(y.shape)
        codes = np.where(sdec[..., None] == 0, 0, codes).astype(np.uint8).reshape(len(s), h, d)
        want_packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
        assert np.array_equal(got_packed, want_packed)
    # the zero group and the tiny group both store scale 0 and +0 codes
    t0 = s[0]
    assert np.all(kc.reshape(c.num_blocks, stride)[t0 // bs, data_bytes + (0 * bs + t0 % bs) * 4] == 0)


def test_nvfp4_round_trip_error_bound(orc):
    """|x - deq| <= half the E2M1 spacing at x/scale, times scale, unless saturated."""
    bs, h, d = 16, 1, 128
    T = 64
    key = inputs.normal_bf16(30, (T, h, d))
    slots = np.arange(T, dtype=np.int32)
    nb = T // bs
    kc = np.zeros(orc.cache_bytes(2, nb, bs, h, d), np.uint8)
    vc = kc.copy()
    orc.reshape_and_cache(key, key, kc, vc, slots, h, d, bs, nb, 2)
    deq = refs.dequant_pages(kc, 2, nb, bs, h, d).reshape(T, h, d)
    x = refs.bf16_to_f64(key)
    data_bytes, stride = refs.nvfp4_geometry(bs, h, d)
    sc = refs.e4m3_decode(kc.reshape(nb, stride)[:, data_bytes:data_bytes + bs * h * d // 16]
                          ).reshape(T, h, d // 16)
    s = np.repeat(sc, 16, axis=-1)
    y = np.abs(x) / s
    grid = refs.E2M1_TABLE
    i = np.clip(np.searchsorted(grid, y), 1, len(grid) - 1)
    half = (grid[i] - grid[i - 1]) / 2
    sat = y >= 6.0
    err = np.abs(x - deq)
    assert np.all(err[~sat] <= half[~sat] * s[~sat] * (1 + 1e-6))
    assert np.all(np.abs(deq[sat]) == 6.0 * s[sat])
