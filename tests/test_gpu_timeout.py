"""The decode kernels' bounded waits, made to run out on purpose.

pd_test_set_consumer_wait_ns(0) turns every consumer-side wait for a stage of
keys into a single non-blocking probe, so a consumer warp gives up on the
first stage whose copies have not landed yet (certain in an HBM-bound kernel
over long sequences). The call must still end (no hang, no CUDA error),
report PD_DEV_TIMEOUT, and leave the device usable: the next ordinary calls
on the same stream match the oracle. Nothing here faults the GPU or leaves a
wait without a limit: the producer drains every copy it issued before its
CTA ends."""
import numpy as np
import pytest
import torch

from paged_kv_split_gb300 import inputs
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

PD_DEV_TIMEOUT = 8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_split_gb300 import binding
    binding.pd_device_status(reset=True)
    yield
    binding.pd_test_set_consumer_wait_ns(0xFFFFFFFF)


CASES = [
    # (name, lens, Hq, Hkv, D, bs, kv_dtype): head_dim 128 (warps split the keys)
    # and 256 (warps split head_dim and meet at a named barrier every tile)
    ("to_d128_bf16", [6000, 3000, 4500, 2500], 32, 8, 128, 16, 0),
    ("to_d128_nvfp4", [6000, 3000, 4500, 2500], 32, 8, 128, 16, 2),
    ("to_d256_fp8", [5000, 2600], 8, 4, 256, 16, 1),
]


def _balanced(case, kc, vc, kv_dtype, ks, vs):
    from paged_kv_split_gb300 import binding as B
    plan = B.pd_balanced_plan(case.seq_lens, num_q_heads=case.num_q_heads,
                              num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
                              block_size=case.block_size,
                              max_blocks_per_seq=case.max_blocks_per_seq,
                              sliding_window=case.sliding_window, kv_dtype=kv_dtype,
                              num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    q = U.bf16_dev(case.q)
    out = torch.empty_like(q)
    B.pd_decode_balanced(q, kc, vc, U.to_dev(case.block_tables), plan.to("cuda"), plan, out,
                         num_kv_heads=case.num_kv_heads, block_size=case.block_size,
                         num_blocks=case.num_blocks, scale=case.scale,
                         sliding_window=case.sliding_window, kv_dtype=kv_dtype, k_scale=ks,
                         v_scale=vs)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("spec", CASES, ids=[c[0] for c in CASES])
def test_consumer_waits_run_out_and_the_device_recovers(orc, spec):
    from paged_kv_split_gb300 import binding as B
    name, lens, hq, hkv, d, bs, kv_dtype = spec
    case = inputs.make_case(name, lens, hq, hkv, d, bs, seed=80 + d)
    ks, vs = U.fp8_scales(orc, case) if kv_dtype == 1 else (1.0, 1.0)
    kc, vc = U.gpu_write_cache(case, kv_dtype, ks, vs)
    ref, _ = U.oracle_decode(orc, case, kc.cpu().numpy(), vc.cpu().numpy(), kv_dtype, ks, vs)
    B.pd_device_status(reset=True)
    prev = B.pd_test_set_consumer_wait_ns(0)
    try:
        # split schedule (S=4: several tiles per CTA), then the balanced one
        U.gpu_decode(case, kc, vc, kv_dtype, 4, ks, vs)
        assert B.pd_device_status(reset=True) & PD_DEV_TIMEOUT, "split kernel: no timeout seen"
        _balanced(case, kc, vc, kv_dtype, ks, vs)
        assert B.pd_device_status(reset=True) & PD_DEV_TIMEOUT, "balanced kernel: no timeout seen"
    finally:
        B.pd_test_set_consumer_wait_ns(0xFFFFFFFF)
    assert prev == 2_000_000_000
    # the same stream, ordinary limits: correct again, and no flag raised
    got = U.gpu_decode(case, kc, vc, kv_dtype, 4, ks, vs)
    U.assert_close(got, ref, what=f"{name}: split after the timeout")
    got_b = _balanced(case, kc, vc, kv_dtype, ks, vs)
    U.assert_close(got_b, ref, what=f"{name}: balanced after the timeout")
    assert B.pd_device_status(reset=True) == 0
