"""Strided rows (a fused QKV buffer: each token's row holds q, then k, then v;
an output buffer with padded rows): pd_decode_strided /
pd_decode_balanced_strided must give exactly what pd_decode /
pd_decode_balanced give on packed q and out, and leave the padding alone."""
import numpy as np
import pytest
import torch

from paged_kv_split_gb300 import inputs
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv_dtype", [0, 1, 2], ids=["bf16", "fp8", "nvfp4"])
def test_fused_qkv_rows_match_packed_q(orc, kv_dtype):
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_case("strided", [300, 17, 1000, 64], 16, 4, 128, 16, seed=31)
    ks, vs = U.fp8_scales(orc, case) if kv_dtype == 1 else (1.0, 1.0)
    kc, vc = U.gpu_write_cache(case, kv_dtype, ks, vs)
    Bn, Hq, D, Hkv = case.num_seqs, case.num_q_heads, case.head_dim, case.num_kv_heads
    q = U.bf16_dev(case.q)
    row = (Hq + 2 * Hkv) * D
    fused = U.bf16_dev(inputs.normal_bf16(32, (Bn, row)))
    fused.view(Bn, Hq + 2 * Hkv, D)[:, :Hq] = q
    bt, lens = U.to_dev(case.block_tables), U.to_dev(case.seq_lens)
    kw = dict(num_kv_heads=Hkv, block_size=case.block_size, num_blocks=case.num_blocks,
              scale=case.scale, kv_dtype=kv_dtype, k_scale=ks, v_scale=vs)
    pad = 8 * D  # output rows padded by 8 heads
    sentinel = -12345

    def strided_out():
        o = torch.full((Bn, Hq * D + pad), 0, dtype=torch.int16, device="cuda")
        o[:, Hq * D:] = sentinel
        return o.view(torch.bfloat16)

    def check(packed, rows, what):
        r = rows.view(torch.int16)
        assert torch.equal(packed.view(torch.int16).view(Bn, Hq * D), r[:, :Hq * D]), what
        assert bool((r[:, Hq * D:] == sentinel).all()), what + ": padding written"

    for S in (1, 3):
        a, b = torch.empty_like(q), strided_out()
        B.pd_decode(q, kc, vc, bt, lens, a, num_splits=S, **kw)
        B.pd_decode_strided(fused, kc, vc, bt, lens, b, num_q_heads=Hq, head_dim=D,
                            num_splits=S, **kw)
        torch.cuda.synchronize()
        check(a, b, f"split S={S}")
    plan = B.pd_balanced_plan(case.seq_lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                              block_size=case.block_size,
                              max_blocks_per_seq=case.max_blocks_per_seq, kv_dtype=kv_dtype,
                              num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    pdev = plan.to("cuda")
    a, b = torch.empty_like(q), strided_out()
    B.pd_decode_balanced(q, kc, vc, bt, pdev, plan, a, **kw)
    B.pd_decode_balanced_strided(fused, kc, vc, bt, pdev, plan, b, num_q_heads=Hq, head_dim=D,
                                 **kw)
    torch.cuda.synchronize()
    check(a, b, "balanced")


def test_bad_strides_are_refused():
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_case("badstride", [40], 8, 2, 64, 16, seed=33)
    kc, vc = U.gpu_write_cache(case, 0)
    bt, lens = U.to_dev(case.block_tables), U.to_dev(case.seq_lens)
    out = torch.empty(1, 8 * 64, dtype=torch.bfloat16, device="cuda")
    kw = dict(num_q_heads=8, head_dim=64, num_kv_heads=2, block_size=16,
              num_blocks=case.num_blocks, scale=0.125, num_splits=1)
    short = torch.zeros(1, 8 * 64 - 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        B.pd_decode_strided(short, kc, vc, bt, lens, out, **kw)
    odd = torch.zeros(1, 8 * 64 + 4, dtype=torch.bfloat16, device="cuda")  # rows not 16-B aligned
    with pytest.raises(B.PdError):
        B.pd_decode_strided(odd, kc, vc, bt, lens, out, **kw)
