"""The CUDA-core partial kernel stays an independent cross-check of the
tensor-core one: pd_decode_crosscheck (scores by warp reductions, P V in
plain fp32 loops, every partial through the workspace and the combine) runs
the tiny case and the small parity grid against the oracle, all three cache
forms."""
import functools
import zlib

import pytest
import torch

from paged_kv_split_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _crosscheck_decode(monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_split_gb300 import binding as B
    monkeypatch.setattr(B, "pd_decode", functools.partial(B.pd_decode, crosscheck=True))


def test_crosscheck_tiny_config(orc):
    from tests.test_gpu_decode import run_parity
    run_parity(orc, inputs.tiny(), 0, [1, 2])


@pytest.mark.parametrize("kv_dtype", [0, 1, 2], ids=["bf16", "fp8", "nvfp4"])
def test_crosscheck_small_parity(orc, kv_dtype):
    from tests.test_gpu_decode import SMALL, run_parity
    for name, lens, hq, hkv, d, bs, w in SMALL:
        case = inputs.make_case(name, lens, hq, hkv, d, bs, seed=zlib.crc32(name.encode()) % 1000,
                                sliding_window=w, extra_blocks=2)
        run_parity(orc, case, kv_dtype, [1, 3, 0])
