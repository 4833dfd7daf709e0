"""Balanced decode (pd_balanced_plan on the host + pd_decode_balanced) against
the oracle, through the C ABI: same tolerance and the same cases as the
split-KV path, plus plans whose shares cut heads in several places, empty
sequences and a malformed plan entry."""
import zlib

import numpy as np
import pytest
import torch

from paged_kv_split_gb300 import inputs
from tests import gpu_util as U
from tests.test_gpu_decode import SMALL

pytestmark = pytest.mark.gpu


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def gpu_decode_balanced(case, kc, vc, kv_dtype, ks=1.0, vs=1.0, num_sms=None, plan_edit=None):
    from paged_kv_split_gb300 import binding as B
    plan = B.pd_balanced_plan(case.seq_lens, num_q_heads=case.num_q_heads,
                              num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
                              block_size=case.block_size,
                              max_blocks_per_seq=case.max_blocks_per_seq,
                              sliding_window=case.sliding_window, kv_dtype=kv_dtype,
                              num_sms=num_sms or _sms())
    if plan_edit is not None:
        plan_edit(plan)
    q = U.bf16_dev(case.q)
    out = torch.full_like(q, float("nan"))
    B.pd_decode_balanced(q, kc, vc, U.to_dev(case.block_tables), plan.to("cuda"), plan, out,
                         num_kv_heads=case.num_kv_heads, block_size=case.block_size,
                         num_blocks=case.num_blocks, scale=case.scale,
                         sliding_window=case.sliding_window, kv_dtype=kv_dtype, k_scale=ks,
                         v_scale=vs)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16), plan


def run_balanced(orc, case, kv_dtype, num_sms_list=(None,)):
    ks, vs = U.fp8_scales(orc, case) if kv_dtype == 1 else (1.0, 1.0)
    kc, vc = U.gpu_write_cache(case, kv_dtype, ks, vs)
    ref, _ = U.oracle_decode(orc, case, kc.cpu().numpy(), vc.cpu().numpy(), kv_dtype, ks, vs)
    for n in num_sms_list:
        got, plan = gpu_decode_balanced(case, kc, vc, kv_dtype, ks, vs, num_sms=n)
        U.assert_close(got, ref, what=f"balanced {case.name} dtype={kv_dtype} sms={n} "
                                      f"ctas={plan.num_ctas} pieces={plan.num_pieces}")
    return ref


@pytest.mark.parametrize("kv_dtype", [0, 1, 2], ids=["bf16", "fp8", "nvfp4"])
@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_small_parity(orc, kv_dtype, spec):
    name, lens, hq, hkv, d, bs, w = spec
    case = inputs.make_case(name, lens, hq, hkv, d, bs, seed=zlib.crc32(name.encode()) % 1000,
                            sliding_window=w, extra_blocks=2)
    # few SMs: shares of many pages, several heads per CTA; many SMs: heads
    # cut into many pieces
    run_balanced(orc, case, kv_dtype, num_sms_list=(1, 3, None))


def test_many_sequences_and_empty_ones(orc):
    from paged_kv_split_gb300 import binding as B
    lens = inputs.uniform_int(78, 1100, 1, 60)
    lens[::97] = 0
    case = inputs.make_case("many_bal", lens, 4, 2, 64, 16, seed=13, extra_blocks=1)
    case.block_tables[case.block_tables < 0] = 0
    B.pd_device_status(reset=True)
    for kv_dtype in (0, 2):
        run_balanced(orc, case, kv_dtype)
    assert B.pd_device_status(reset=True) == 0


def test_all_sequences_empty():
    case = inputs.make_case("empty_bal", [0, 0], 8, 2, 64, 16, seed=14, extra_blocks=2)
    case.block_tables[:] = 0
    kc, vc = U.gpu_write_cache(case, 0)
    got, plan = gpu_decode_balanced(case, kc, vc, 0)
    assert plan.num_ctas == 0 and np.all(got == 0)


def test_malformed_plan_entry_is_flagged_not_faulted(orc):
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_case("badplan", [300, 70], 8, 2, 64, 16, seed=15)
    kc, vc = U.gpu_write_cache(case, 0)

    def corrupt(plan):
        w = plan.words
        poff = (8 + plan.num_ctas + 1 + 3) // 4 * 4
        w[poff + 0] = 10 ** 6  # first piece: a head that does not exist

    B.pd_device_status(reset=True)
    got, _ = gpu_decode_balanced(case, kc, vc, 0, plan_edit=corrupt)
    assert B.pd_device_status(reset=True) & 16  # PD_DEV_BAD_PLAN


def test_matches_split_path(orc):
    case = inputs.make_case("vs_split", [2000, 777, 64, 1500], 32, 8, 128, 16, seed=16)
    kc, vc = U.gpu_write_cache(case, 0)
    a, _ = gpu_decode_balanced(case, kc, vc, 0)
    b = U.gpu_decode(case, kc, vc, 0, 4)
    base = U.bf16_bits_to_f32(b).astype(np.float64)
    rms = np.sqrt(np.mean(base ** 2, axis=-1, keepdims=True))
    d = np.abs(U.bf16_bits_to_f32(a) - base)
    assert np.all(d <= 2.0 ** -7 * (2 * np.abs(base) + rms))


# ---- the full-size workloads (all outputs compared) -------------------------
def test_llama8b_batch32(orc):
    run_balanced(orc, inputs.llama8b(), 0)


@pytest.mark.parametrize("num_seqs,seq_len", [(1, 32768), (4, 8192), (4, 32768)])
def test_long_context(orc, num_seqs, seq_len):
    run_balanced(orc, inputs.long_context(num_seqs, seq_len), 0)


def test_wide_head_d512(orc):
    run_balanced(orc, inputs.wide_head(), 0)


def test_sliding_window_d256(orc):
    run_balanced(orc, inputs.sliding(), 0)


@pytest.mark.parametrize("kv_dtype", [1, 2], ids=["fp8", "nvfp4"])
def test_quantised_batch64(orc, kv_dtype):
    run_balanced(orc, inputs.quantised(kv_dtype), kv_dtype)


def test_partial_then_combine_equals_one_call(orc):
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_case("halves", [900, 40, 0, 2100], 16, 4, 128, 16, seed=17,
                            extra_blocks=1)
    case.block_tables[case.block_tables < 0] = 0
    kc, vc = U.gpu_write_cache(case, 0)
    fused, plan = gpu_decode_balanced(case, kc, vc, 0)
    q = U.bf16_dev(case.q)
    out = torch.full_like(q, float("nan"))
    kw = dict(num_kv_heads=case.num_kv_heads, block_size=case.block_size,
              num_blocks=case.num_blocks, scale=case.scale)
    pdev, bt = plan.to("cuda"), U.to_dev(case.block_tables)
    ws = torch.empty(max(plan.workspace_bytes, 16), dtype=torch.uint8, device="cuda")
    B.pd_decode_balanced_partial(q, kc, vc, bt, pdev, plan, out, workspace=ws, **kw)
    B.pd_decode_balanced_combine(q, kc, vc, bt, pdev, plan, out, workspace=ws, **kw)
    torch.cuda.synchronize()
    halves = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(fused, halves)


# ---- workspace contents, skewed plans, graph replays -------------------------
def _balanced_call(case, kc, vc, plan, pdev, q, out, ws, kv_dtype=0, fn=None):
    from paged_kv_split_gb300 import binding as B
    (fn or B.pd_decode_balanced)(q, kc, vc, U.to_dev(case.block_tables), pdev, plan, out,
                                 num_kv_heads=case.num_kv_heads, block_size=case.block_size,
                                 num_blocks=case.num_blocks, scale=case.scale,
                                 sliding_window=case.sliding_window, kv_dtype=kv_dtype,
                                 workspace=ws)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_workspace_contents_do_not_matter(orc):
    """Whatever the workspace held before the call (zeros, all-ones, random
    bytes, the previous call's partials for another q) the output has the
    same bits, equal to the oracle's."""
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_case("ws_any", [1500, 40, 0, 2600, 333, 17], 32, 8, 128, 16, seed=21,
                            extra_blocks=1)
    case.block_tables[case.block_tables < 0] = 0
    kc, vc = U.gpu_write_cache(case, 0)
    ref, _ = U.oracle_decode(orc, case, kc.cpu().numpy(), vc.cpu().numpy(), 0)
    plan = B.pd_balanced_plan(case.seq_lens, num_q_heads=case.num_q_heads,
                              num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
                              block_size=case.block_size,
                              max_blocks_per_seq=case.max_blocks_per_seq, num_sms=_sms())
    assert plan.num_pieces > case.num_seqs * case.num_kv_heads  # some ranges have pieces to merge
    pdev = plan.to("cuda")
    q = U.bf16_dev(case.q)
    nbytes = max(plan.workspace_bytes, 16)
    fills = [torch.zeros(nbytes, dtype=torch.uint8, device="cuda"),
             torch.full((nbytes,), 255, dtype=torch.uint8, device="cuda"),
             torch.from_numpy(inputs.uniform_int(22, nbytes, 0, 255).astype(np.uint8)).cuda()]
    outs = []
    for ws in fills:
        out = torch.full_like(q, float("nan"))
        _balanced_call(case, kc, vc, plan, pdev, q, out, ws)
        torch.cuda.synchronize()
        outs.append(_bits(out))
    U.assert_close(outs[0], ref, what="balanced, zeroed workspace")
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    # leftovers of a call with another q, then this q again on the same bytes
    ws = fills[2]
    q2 = U.bf16_dev(inputs.make_case("ws_any2", list(case.seq_lens), 32, 8, 128, 16,
                                     seed=23).q)
    out2 = torch.full_like(q, float("nan"))
    _balanced_call(case, kc, vc, plan, pdev, q2, out2, ws)
    out = torch.full_like(q, float("nan"))
    _balanced_call(case, kc, vc, plan, pdev, q, out, ws)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), outs[0])
    assert not np.array_equal(_bits(out2), outs[0])


def test_long_range_among_short_ones(orc):
    """One long sequence among short ones: few pieces per range on average,
    so the combine's CTAs are sized for a few partials, but the long
    sequence's ranges have dozens (several rounds of loads per thread). Equal
    to the oracle, and bit-equal to the two halves called one by one."""
    from paged_kv_split_gb300 import binding as B
    lens = [30000] + [int(x) for x in inputs.uniform_int(24, 63, 1, 200)]
    case = inputs.make_case("long_among_short", lens, 32, 8, 128, 16, seed=25)
    kc, vc = U.gpu_write_cache(case, 0)
    ref, _ = U.oracle_decode(orc, case, kc.cpu().numpy(), vc.cpu().numpy(), 0)
    got, plan = gpu_decode_balanced(case, kc, vc, 0)
    segs = case.num_seqs * case.num_kv_heads
    assert plan.num_pieces <= 8 * segs and plan.num_pieces - segs > 20
    U.assert_close(got, ref, what="long range among short ones")
    q = U.bf16_dev(case.q)
    out = torch.full_like(q, float("nan"))
    pdev = plan.to("cuda")
    ws = torch.empty(max(plan.workspace_bytes, 16), dtype=torch.uint8, device="cuda")
    _balanced_call(case, kc, vc, plan, pdev, q, out, ws, fn=B.pd_decode_balanced_partial)
    _balanced_call(case, kc, vc, plan, pdev, q, out, ws, fn=B.pd_decode_balanced_combine)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), got)


@pytest.mark.parametrize("kv_dtype", [0, 1, 2], ids=["bf16", "fp8", "nvfp4"])
def test_graph_replays_follow_q(orc, kv_dtype):
    """pd_decode_balanced captured in a CUDA graph: q changes between replays
    (copied into the captured buffer); each replay equals an eager call on
    that q."""
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_case("graph_bal", [700, 1900, 64, 1200], 16, 4, 128, 16, seed=26)
    ks, vs = U.fp8_scales(orc, case) if kv_dtype == 1 else (1.0, 1.0)
    kc, vc = U.gpu_write_cache(case, kv_dtype, ks, vs)
    plan = B.pd_balanced_plan(case.seq_lens, num_q_heads=case.num_q_heads,
                              num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
                              block_size=case.block_size,
                              max_blocks_per_seq=case.max_blocks_per_seq, kv_dtype=kv_dtype,
                              num_sms=_sms())
    pdev = plan.to("cuda")
    bt = U.to_dev(case.block_tables)
    kw = dict(num_kv_heads=case.num_kv_heads, block_size=case.block_size,
              num_blocks=case.num_blocks, scale=case.scale, kv_dtype=kv_dtype, k_scale=ks,
              v_scale=vs)
    qs = [U.bf16_dev(inputs.make_case("graph_bal_q", list(case.seq_lens), 16, 4, 128, 16,
                                      seed=27 + i).q) for i in range(3)]
    q = qs[0].clone()
    out = torch.empty_like(q)
    ws = torch.empty(max(plan.workspace_bytes, 16), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        B.pd_decode_balanced(q, kc, vc, bt, pdev, plan, out, workspace=ws, stream=s, **kw)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.pd_decode_balanced(q, kc, vc, bt, pdev, plan, out, workspace=ws, stream=s, **kw)
    for qi in qs + qs[::-1]:
        q.copy_(qi)
        g.replay()
        torch.cuda.synchronize()
        got = _bits(out)
        eager = torch.full_like(q, float("nan"))
        B.pd_decode_balanced(qi, kc, vc, bt, pdev, plan, eager, **kw)
        torch.cuda.synchronize()
        assert np.array_equal(got, _bits(eager))
