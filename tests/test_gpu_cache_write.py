"""GPU cache write / quantise vs the oracle: bit-exact bytes, slot placement
and untouched slots (sentinel-filled pools), exhaustive over bf16 inputs."""
import numpy as np
import pytest
import torch

from paged_kv_split_gb300 import inputs
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

SHAPES = [(2, 64, 16), (8, 128, 16), (8, 128, 32), (4, 256, 16), (2, 512, 16), (1, 64, 32)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_split_gb300 import binding
    binding.pd_device_status(reset=True)
    yield
    assert binding.pd_device_status(reset=True) == 0


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("hkv,d,bs", SHAPES)
def test_cache_bytes_match_oracle(orc, kv_dtype, hkv, d, bs):
    case = inputs.make_case("cw", [37, 5, 64, 1], 2 * hkv, hkv, d, bs, seed=40 + d + bs,
                            extra_blocks=3)
    ks, vs = U.fp8_scales(orc, case) if kv_dtype == 1 else (1.0, 1.0)
    kc, vc = U.gpu_write_cache(case, kv_dtype, ks, vs)
    okc, ovc = U.oracle_write_cache(orc, case, kv_dtype, ks, vs)
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(vc.cpu().numpy(), ovc)


def _all_bf16_case(hkv=1, d=128, bs=16, shuffle_seed=None):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    if shuffle_seed is not None:
        pats = pats[inputs.permutation(shuffle_seed, 65536)]
    T = 65536 // (hkv * d)
    key = pats.reshape(T, hkv, d)
    value = pats[::-1].copy().reshape(T, hkv, d)
    nb = T // bs
    case = inputs.make_case("all", [T], hkv, hkv, d, bs, seed=1)
    case.key, case.value = key, value
    case.slot_mapping = np.arange(T, dtype=np.int32)
    case.num_blocks = nb
    return case


@pytest.mark.parametrize("scale", [1.0, 2.0 ** -7, 1.7, 3.14159 / 448, 1e-3, 1e6, 2.0 ** -20])
def test_fp8_exhaustive_over_bf16(orc, scale):
    case = _all_bf16_case()
    kc, vc = U.gpu_write_cache(case, 1, scale, 1.0 / scale)
    okc, ovc = U.oracle_write_cache(orc, case, 1, scale, 1.0 / scale)
    k = kc.cpu().numpy()
    bad = np.nonzero(k != okc)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:5]}: {k[bad[:5]]} vs {okc[bad[:5]]}"
    assert np.array_equal(vc.cpu().numpy(), ovc)


@pytest.mark.parametrize("shuffle_seed", [None, 7, 8])
def test_nvfp4_exhaustive_over_bf16(orc, shuffle_seed):
    case = _all_bf16_case(hkv=2, d=64, shuffle_seed=shuffle_seed)
    kc, vc = U.gpu_write_cache(case, 2)
    okc, ovc = U.oracle_write_cache(orc, case, 2)
    k = kc.cpu().numpy()
    bad = np.nonzero(k != okc)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:5]}: {k[bad[:5]]} vs {okc[bad[:5]]}"
    assert np.array_equal(vc.cpu().numpy(), ovc)


@pytest.mark.parametrize("n", [1, 7, 8, 1000, 1_000_003, 8 * 2048 * 640 + 5])
def test_absmax_matches_oracle(orc, n):
    x = inputs.normal_bf16(60 + n % 97, (n,), std=3.0)
    if n > 10:
        x[n // 2] = 0x7FC0        # NaN: skipped
        x[n // 3] = inputs.to_bf16_bits(np.array([-97.5], np.float32))[0]
    from paged_kv_split_gb300 import binding
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    binding.pd_absmax_bf16(U.bf16_dev(x), out)
    assert out.item() == orc.absmax_bf16(x)


def test_fp8_calibrate_matches_oracle(orc):
    from paged_kv_split_gb300 import binding
    case = inputs.make_case("cal", [100, 60], 8, 4, 128, 16, seed=61)
    ks, vs = binding.fp8_calibrate(U.bf16_dev(case.key), U.bf16_dev(case.value))
    assert (ks, vs) == U.fp8_scales(orc, case)


def test_fp8_scales_from_absmax_match_oracle(orc):
    """The device scale kernel against oracle_fp8_scale, bit for bit, on
    special values (0, NaN, denormals, the largest finite) and random ones."""
    from paged_kv_split_gb300 import binding
    special = np.array([0.0, -0.0, np.nan, 1e-45, 1.17e-38, 448.0, 1.0, 3.4e38, np.inf, -2.0],
                       np.float32)
    rnd = (inputs.normal_bf16(63, (5000,), std=40.0).astype(np.uint32) << 16).view(np.float32)
    bits = inputs.uniform_int(64, 5000, 0, 0x7F7FFFFF).astype(np.uint32).view(np.float32)
    amax = np.concatenate([special, np.abs(rnd), bits]).astype(np.float32)
    a = torch.from_numpy(amax).cuda()
    out = torch.empty_like(a)
    binding.pd_fp8_scales_from_absmax(a, out)
    got = out.cpu().numpy()
    want = np.array([orc.fp8_scale(float(x)) for x in amax], np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_slots_out_of_pool_are_skipped_and_flagged(orc):
    from paged_kv_split_gb300 import binding
    case = inputs.make_case("bad", [20], 4, 2, 64, 16, seed=62, extra_blocks=1)
    case.slot_mapping = case.slot_mapping.copy()
    case.slot_mapping[3] = case.num_blocks * 16 + 5     # beyond the pool
    case.slot_mapping[4] = -1                           # padding
    binding.pd_device_status(reset=True)
    kc, vc = U.gpu_write_cache(case, 0)
    flags = binding.pd_device_status(reset=True)
    assert flags & 4
    ok = case.slot_mapping.copy()
    ok[3] = -1
    case.slot_mapping = ok
    okc, ovc = U.oracle_write_cache(orc, case, 0)
    assert np.array_equal(kc.cpu().numpy(), okc)
