"""GPU decode (split-KV partials + combine) vs the oracle, through the C ABI.

Tolerance |gpu - oracle| <= 1e-2 + 1e-2 |oracle| elementwise on the bf16
outputs. Quantised caches: the GPU-written cache bytes are first checked
bit-exact against the oracle's, then the oracle decodes those same bytes.
"""
import zlib

import numpy as np
import pytest
import torch

from paged_kv_split_gb300 import inputs
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_split_gb300 import binding
    binding.pd_device_status(reset=True)
    yield


def _scales(orc, case, kv_dtype):
    return U.fp8_scales(orc, case) if kv_dtype == 1 else (1.0, 1.0)


def run_parity(orc, case, kv_dtype, splits, check_cache=True):
    """Write the cache on the GPU, check its bytes, then decode with every S in
    `splits` and compare each against one oracle decode of the same bytes."""
    ks, vs = _scales(orc, case, kv_dtype)
    kc, vc = U.gpu_write_cache(case, kv_dtype, ks, vs)
    kh, vh = kc.cpu().numpy(), vc.cpu().numpy()
    if check_cache:
        okc, ovc = U.oracle_write_cache(orc, case, kv_dtype, ks, vs)
        assert np.array_equal(kh, okc) and np.array_equal(vh, ovc), "cache bytes differ"
    ref, _ = U.oracle_decode(orc, case, kh, vh, kv_dtype, ks, vs)
    outs = {}
    for S in splits:
        got = U.gpu_decode(case, kc, vc, kv_dtype, S, ks, vs)
        U.assert_close(got, ref, what=f"{case.name} dtype={kv_dtype} S={S}")
        outs[S] = got
    return outs, ref


def test_tiny_config(orc):
    """2 seqs {17, 40}, GQA 2, D=64, bs=16, a permuted 16-page pool, S in {1, 2}."""
    case = inputs.tiny()
    outs, _ = run_parity(orc, case, 0, [1, 2])
    from paged_kv_split_gb300 import binding
    assert binding.pd_device_status() == 0


SMALL = [
    # (name, seq_lens, Hq, Hkv, D, bs, window)
    ("g1_d64", [1, 15, 16, 17, 100], 4, 4, 64, 16, 0),
    ("g2_d128_bs32", [31, 32, 33, 200], 8, 4, 128, 32, 0),
    ("g4_d128", [333, 1, 64, 129], 16, 4, 128, 16, 0),
    ("g8_d128", [257, 90], 32, 4, 128, 16, 0),
    ("g16_d64", [70, 300], 16, 1, 64, 16, 0),
    ("g8_d256_win", [300, 45], 16, 2, 256, 16, 100),
    ("g8_d512", [130, 19], 16, 2, 512, 16, 0),
    ("g2_d256_win_bs32", [500, 33, 1], 8, 4, 256, 32, 64),
    ("g16_d512_win", [97], 16, 1, 512, 32, 50),
]


@pytest.mark.parametrize("kv_dtype", [0, 1, 2], ids=["bf16", "fp8", "nvfp4"])
@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_small_parity(orc, kv_dtype, spec):
    name, lens, hq, hkv, d, bs, w = spec
    case = inputs.make_case(name, lens, hq, hkv, d, bs, seed=zlib.crc32(name.encode()) % 1000, sliding_window=w,
                            extra_blocks=2)
    run_parity(orc, case, kv_dtype, [1, 3, 0])


def test_two_step_partial_then_combine(orc):
    """pd_decode_partial + pd_decode_combine (two calls) agree with the oracle
    like pd_decode (the same two kernels in one call, the combine launched as
    a programmatic dependent of the partial kernel)."""
    from paged_kv_split_gb300 import binding
    case = inputs.make_case("twostep", [700, 33, 1290, 0], 32, 8, 128, 16, seed=21)
    case.block_tables[case.block_tables < 0] = 0
    kc, vc = U.gpu_write_cache(case, 0)
    ref, _ = U.oracle_decode(orc, case, kc.cpu().numpy(), vc.cpu().numpy(), 0)
    q = U.bf16_dev(case.q)
    bt, lens = U.to_dev(case.block_tables), U.to_dev(case.seq_lens)
    for S in (1, 4, 9):
        ws = torch.empty(binding.pd_decode_workspace_bytes(4, 32, 128, S), dtype=torch.uint8,
                         device="cuda")
        out = torch.empty_like(q)
        binding.pd_decode_partial(q, kc, vc, bt, lens, ws, num_kv_heads=8, block_size=16,
                                  num_blocks=case.num_blocks, scale=case.scale, num_splits=S)
        binding.pd_decode_combine(ws, lens, out, block_size=16,
                                  max_blocks_per_seq=case.max_blocks_per_seq, num_splits=S)
        torch.cuda.synchronize()
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        U.assert_close(got, ref, what=f"two-step S={S}")
        fused = U.gpu_decode(case, kc, vc, 0, S)
        U.assert_close(fused, ref, what=f"fused S={S}")


def test_many_sequences(orc):
    """Over a thousand short sequences, some empty."""
    lens = inputs.uniform_int(77, 1100, 1, 60)
    lens[::97] = 0
    case = inputs.make_case("many", lens, 4, 2, 64, 16, seed=12, extra_blocks=1)
    case.block_tables[case.block_tables < 0] = 0
    for kv_dtype in (0, 2):
        run_parity(orc, case, kv_dtype, [1, 3])


def test_split_independence(orc):
    case = inputs.make_case("splits", [2000, 777, 64], 32, 8, 128, 16, seed=5)
    outs, _ = run_parity(orc, case, 0, [1, 2, 4, 16, 64])
    base = U.bf16_bits_to_f32(outs[1]).astype(np.float64)
    # The split count changes only rounding (summation order, the bf16 rounding
    # of the softmax weights relative to each split's running max), whose size
    # follows the scale of the whole output row, not of each element.
    rms = np.sqrt(np.mean(base ** 2, axis=-1, keepdims=True))
    for S, o in outs.items():
        d = np.abs(U.bf16_bits_to_f32(o) - base)
        bound = 2.0 ** -7 * (2 * np.abs(base) + rms)
        assert np.all(d <= bound), f"S={S}: max change {d.max():.3g} beyond rounding"


def test_page_permutation_is_bit_identical(orc):
    case = inputs.make_case("perm", [300, 77], 16, 4, 128, 16, seed=6, extra_blocks=5)
    kc, vc = U.gpu_write_cache(case, 0)
    a = U.gpu_decode(case, kc, vc, 0, 4)
    perm = inputs.permutation(77, case.num_blocks)
    pb = kc.numel() // case.num_blocks
    kp, vp = kc.view(case.num_blocks, pb), vc.view(case.num_blocks, pb)
    idx = torch.from_numpy(perm).cuda()
    kc2, vc2 = torch.empty_like(kp), torch.empty_like(vp)
    kc2[idx] = kp
    vc2[idx] = vp
    bt2 = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1)
    b = U.gpu_decode(case, kc2.view(-1), vc2.view(-1), 0, 4, block_tables=bt2.astype(np.int32))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("S", [1, 2])
def test_length_one_returns_v0_exactly(orc, S):
    case = inputs.make_case("l1", [1, 1, 1], 16, 4, 128, 16, seed=7)
    kc, vc = U.gpu_write_cache(case, 0)
    out = U.gpu_decode(case, kc, vc, 0, S)
    v0 = case.value.reshape(3, 4, 128)
    assert np.array_equal(out, np.repeat(v0, 4, axis=1))


def test_constant_v_returns_constant(orc):
    case = inputs.make_case("cv", [500, 3], 8, 2, 64, 16, seed=8)
    c_bits = inputs.to_bf16_bits(np.array([-1.3125], np.float32))[0]
    case.value[:] = c_bits
    kc, vc = U.gpu_write_cache(case, 0)
    for S in (1, 4):
        out = U.gpu_decode(case, kc, vc, 0, S)
        assert np.all(np.abs(U.bf16_bits_to_f32(out) + 1.3125) <= 1.3125 * 2.0 ** -8)


def test_large_scores_stay_finite(orc):
    case = inputs.make_case("big", [600, 40], 16, 4, 128, 16, seed=9, q_std=100.0)
    for kv_dtype in (0, 1, 2):
        run_parity(orc, case, kv_dtype, [1, 8])


def test_zero_length_and_empty_batch(orc):
    case = inputs.make_case("z", [0, 40, 0], 8, 2, 64, 16, seed=10, extra_blocks=1)
    case.block_tables[case.block_tables < 0] = 0
    kc, vc = U.gpu_write_cache(case, 0)
    out = U.gpu_decode(case, kc, vc, 0, 2)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    kh, vh = kc.cpu().numpy(), vc.cpu().numpy()
    ref, _ = U.oracle_decode(orc, case, kh, vh, 0)
    U.assert_close(out, ref, what="zero-length rows")
    # an empty batch is a no-op
    from paged_kv_split_gb300 import binding
    q = torch.empty(0, 8, 64, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(0, 1, dtype=torch.int32, device="cuda")
    lens = torch.zeros(0, dtype=torch.int32, device="cuda")
    binding.pd_decode(q, kc, vc, bt, lens, torch.empty_like(q), num_kv_heads=2, block_size=16,
                      num_blocks=case.num_blocks, scale=0.125, num_splits=1)


def test_bad_block_table_entry_is_flagged_not_faulted(orc):
    from paged_kv_split_gb300 import binding
    case = inputs.make_case("badpage", [50, 20], 8, 2, 64, 16, seed=11)
    kc, vc = U.gpu_write_cache(case, 0)
    bt = case.block_tables.copy()
    bt[0, 1] = case.num_blocks + 3          # out of the pool
    bt[1, 0] = -7
    binding.pd_device_status(reset=True)
    out = U.gpu_decode(case, kc, vc, 0, 2, block_tables=bt)
    flags = binding.pd_device_status(reset=True)
    assert flags & 1
    assert np.all(np.isfinite(U.bf16_bits_to_f32(out)))


# ---- the full-size workloads (all outputs compared) -------------------------
def test_llama8b_batch32(orc):
    run_parity(orc, inputs.llama8b(), 0, [0], check_cache=False)


@pytest.mark.parametrize("num_seqs", [1, 4])
@pytest.mark.parametrize("seq_len", [1024, 8192, 32768])
def test_long_context(orc, num_seqs, seq_len):
    run_parity(orc, inputs.long_context(num_seqs, seq_len), 0, [1, 4, 16, 64, 0],
               check_cache=False)


def test_wide_head_d512(orc):
    run_parity(orc, inputs.wide_head(), 0, [0], check_cache=False)


def test_sliding_window_d256(orc):
    run_parity(orc, inputs.sliding(), 0, [0], check_cache=False)


@pytest.mark.parametrize("kv_dtype", [1, 2], ids=["fp8", "nvfp4"])
def test_quantised_batch64(orc, kv_dtype):
    run_parity(orc, inputs.quantised(kv_dtype), kv_dtype, [0], check_cache=True)


@pytest.mark.parametrize("d,splits", [(64, (130, 400)), (128, (100, 257)), (256, (70, 150))])
def test_many_splits_per_row(orc, d, splits):
    """Split counts far above a combine CTA's first round of loads (its lane
    groups x 8 rows): the combine takes the rest in further rounds, the
    lane-group count capped by its 256 threads."""
    case = inputs.make_case(f"many_splits_d{d}", [16000, 2100], 8, 2, d, 16, seed=31 + d)
    kc, vc = U.gpu_write_cache(case, 0)
    ref, _ = U.oracle_decode(orc, case, kc.cpu().numpy(), vc.cpu().numpy(), 0)
    for S in splits:
        got = U.gpu_decode(case, kc, vc, 0, S)
        U.assert_close(got, ref, what=f"D={d} S={S}")
