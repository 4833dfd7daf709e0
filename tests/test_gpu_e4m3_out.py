"""pd_decode_e4m3_out (E4M3 output codes) against the oracle, through the C ABI.

The codes are E4M3(o / out_scale) of the fp32 attention output o. The GPU's o
differs from the oracle's within the decode tolerance (1e-2 + 1e-2 |o|), so a
code may differ where o / out_scale sits near a rounding boundary: each GPU
code must decode to a value between the codes of (o - tol) / out_scale and
(o + tol) / out_scale (E4M3 rounding is monotone, so every o within the
tolerance band encodes into that range), and nearly all codes equal the
oracle's exactly."""
import zlib

import numpy as np
import pytest
import torch

from paged_kv_split_gb300 import inputs
from tests import gpu_util as U
from tests import refs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def gpu_e4m3(case, kc, vc, kv_dtype, S, out_scale, ks=1.0, vs=1.0):
    from paged_kv_split_gb300 import binding as B
    q = U.bf16_dev(case.q)
    out = torch.full(case.q.shape, 0xA5, dtype=torch.uint8, device="cuda")
    B.pd_decode_e4m3_out(q, kc, vc, U.to_dev(case.block_tables), U.to_dev(case.seq_lens), out,
                         out_scale=out_scale, num_kv_heads=case.num_kv_heads,
                         block_size=case.block_size, num_blocks=case.num_blocks,
                         scale=case.scale, num_splits=S, sliding_window=case.sliding_window,
                         kv_dtype=kv_dtype, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def check_codes(orc, got, o_ref, out_scale, what):
    o = o_ref.astype(np.float64).ravel()
    tol = U.ATOL + U.RTOL * np.abs(o)
    lo = np.nextafter(((o - tol) / out_scale).astype(np.float32), np.float32(-np.inf))
    hi = np.nextafter(((o + tol) / out_scale).astype(np.float32), np.float32(np.inf))
    v_lo = refs.e4m3_decode(orc.e4m3_codes(lo))
    v_hi = refs.e4m3_decode(orc.e4m3_codes(hi))
    v = refs.e4m3_decode(got.ravel())
    ok = (v >= v_lo) & (v <= v_hi)
    assert ok.all(), (f"{what}: {int((~ok).sum())} codes outside the tolerance band; first "
                      f"at {int(np.argmin(ok))}: gpu {v[~ok][0]} band [{v_lo[~ok][0]}, "
                      f"{v_hi[~ok][0]}]")


CASES = [
    ("e4_g4_d128", [333, 1, 64, 1290], 16, 4, 128, 16, 0),
    ("e4_g8_d128_bs32", [700, 33, 0], 32, 4, 128, 32, 0),
    ("e4_g2_d256_win", [500, 33], 8, 4, 256, 16, 100),
    ("e4_g8_d512", [130, 19], 16, 2, 512, 16, 0),
    ("e4_g16_d64", [70, 300], 16, 1, 64, 16, 0),
]


@pytest.mark.parametrize("kv_dtype", [0, 1, 2], ids=["bf16", "fp8", "nvfp4"])
@pytest.mark.parametrize("spec", CASES, ids=[c[0] for c in CASES])
def test_e4m3_output_matches_oracle(orc, kv_dtype, spec):
    name, lens, hq, hkv, d, bs, w = spec
    case = inputs.make_case(name, lens, hq, hkv, d, bs, seed=zlib.crc32(name.encode()) % 1000,
                            sliding_window=w, extra_blocks=2)
    ks, vs = U.fp8_scales(orc, case) if kv_dtype == 1 else (1.0, 1.0)
    kc, vc = U.gpu_write_cache(case, kv_dtype, ks, vs)
    kh, vh = kc.cpu().numpy(), vc.cpu().numpy()
    _, o_ref = U.oracle_decode(orc, case, kh, vh, kv_dtype, ks, vs)
    for out_scale in (1.0 / 448, 0.004, 0.05):
        want = orc.decode_e4m3_out(case.q, kh, vh, case.block_tables, case.seq_lens,
                                   case.num_kv_heads, case.block_size, case.num_blocks,
                                   case.scale, out_scale, case.sliding_window, kv_dtype, ks, vs)
        for S in (1, 3, 0):
            got = gpu_e4m3(case, kc, vc, kv_dtype, S, out_scale, ks, vs)
            check_codes(orc, got, o_ref, out_scale, f"{name} dtype={kv_dtype} S={S} "
                                                    f"out_scale={out_scale}")
            assert np.mean(got == want) > 0.9, f"{name}: too few codes equal the oracle's"


def test_e4m3_output_agrees_with_bf16_output(orc):
    """The same step through pd_decode (bf16) and pd_decode_e4m3_out: the codes
    are the encodings of values within bf16 rounding of the bf16 outputs."""
    case = inputs.make_case("e4_vs_bf16", [2000, 777, 64], 32, 8, 128, 16, seed=88)
    kc, vc = U.gpu_write_cache(case, 0)
    bf = U.bf16_bits_to_f32(U.gpu_decode(case, kc, vc, 0, 4)).astype(np.float64)
    s = 0.003
    got = gpu_e4m3(case, kc, vc, 0, 4, s)
    check_codes(orc, got, bf, s, "e4m3 vs bf16 output")


def test_bad_output_scale_is_refused():
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_case("e4_bad", [20], 4, 2, 64, 16, seed=89)
    kc, vc = U.gpu_write_cache(case, 0)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(B.PdError):
            gpu_e4m3(case, kc, vc, 0, 1, bad)
