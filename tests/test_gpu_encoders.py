"""The cache write's device encoders against the oracle's, over every fp32
input.

The FP8 and NVFP4 cache writes quantise fp32 quotients x / scale, which reach
values that no bf16 input and scale produce (mantissas just off a rounding
midpoint, subnormal quotients, NaN payloads). pd_test_encode runs the very
device functions the cache write uses (E4M3 for FP8 codes and NVFP4 scales,
E2M1 for NVFP4 values) on fp32 bit patterns generated from the index, and
this test compares all 2^32 patterns, for both formats, with
oracle_e4m3_code_array / oracle_e2m1_code_array, byte for byte."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("fmt", [0, 1], ids=["e4m3", "e2m1"])
def test_device_encoder_matches_oracle_on_every_fp32(orc, fmt):
    from paged_kv_split_gb300 import binding as B
    codes_d = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    host = torch.empty(CHUNK, dtype=torch.uint8).pin_memory()
    fn = orc.lib.oracle_e4m3_code_array if fmt == 0 else orc.lib.oracle_e2m1_code_array
    pool = ThreadPoolExecutor(16)
    sub = CHUNK // 16
    mismatches = 0
    first_bad = None
    # buffers reused for every chunk (no per-chunk allocation)
    base = np.arange(CHUNK, dtype=np.uint32)
    bits = np.empty(CHUNK, np.uint32)
    want = np.empty(CHUNK, np.uint8)
    x = bits.view(np.float32)

    def oracle_part(k):
        fn(x[k * sub:].ctypes.data, sub, want[k * sub:].ctypes.data)

    for first in range(0, 1 << 32, CHUNK):
        B.pd_test_encode(fmt, first, codes_d)
        host.copy_(codes_d, non_blocking=True)
        np.add(base, np.uint32(first), out=bits)  # wraps modulo 2^32 like the device
        list(pool.map(oracle_part, range(16)))
        torch.cuda.synchronize()
        got = host.numpy()
        if np.array_equal(got, want):
            continue
        bad = np.nonzero(got != want)[0]
        if bad.size:
            mismatches += int(bad.size)
            if first_bad is None:
                i = int(bad[0])
                first_bad = (hex(first + i), int(got[i]), int(want[i]))
    pool.shutdown()
    assert mismatches == 0, (f"{mismatches} fp32 patterns encode differently; first "
                             f"(bits, device, oracle) = {first_bad}")
