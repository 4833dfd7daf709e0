"""A decode step as serving runs it - write one new token per sequence into the
paged cache, then decode - captured once in a CUDA graph and replayed: each
replay must match the same calls made eagerly bit for bit (output and cache
bytes), and the final step must match the oracle run over the same writes."""
import numpy as np
import pytest
import torch

from paged_kv_split_gb300 import inputs
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _step_inputs(st, device="cuda"):
    return (U.bf16_dev(st.q, device), U.bf16_dev(st.key, device), U.bf16_dev(st.value, device),
            U.to_dev(st.slot_mapping, device=device), U.to_dev(st.seq_lens, device=device))


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
def test_graph_replay_of_write_then_decode(orc, kv_dtype):
    from paged_kv_split_gb300 import binding as B
    steps, S = 4, 3
    final = inputs.uniform_int(911 + kv_dtype, 6, 70, 900)
    case = inputs.make_case(f"graph_{kv_dtype}", final, 32, 8, 128, 16, seed=40 + kv_dtype)
    plan = inputs.decode_steps(case, steps, seed=50 + kv_dtype)
    ks, vs = U.fp8_scales(orc, case) if kv_dtype == 1 else (1.0, 1.0)

    kc_e, vc_e = U.gpu_write_cache(case, kv_dtype, ks, vs)   # eager copy
    kc_g, vc_g = kc_e.clone(), vc_e.clone()                   # graph copy
    bt = U.to_dev(case.block_tables)
    common = dict(num_kv_heads=case.num_kv_heads, block_size=case.block_size,
                  num_blocks=case.num_blocks, scale=case.scale, num_splits=S, kv_dtype=kv_dtype,
                  k_scale=ks, v_scale=vs)
    wbytes = B.pd_decode_workspace_bytes(case.num_seqs, case.num_q_heads, case.head_dim, S)
    ws_e = torch.empty(wbytes, dtype=torch.uint8, device="cuda")
    ws_g = torch.empty(wbytes, dtype=torch.uint8, device="cuda")

    def step_calls(kc, vc, q, key, value, slots, lens, out, ws):
        B.pd_reshape_and_cache(key, value, kc, vc, slots, num_blocks=case.num_blocks,
                               block_size=case.block_size, kv_dtype=kv_dtype, k_scale=ks,
                               v_scale=vs)
        B.pd_decode(q, kc, vc, bt, lens, out, workspace=ws, **common)

    # static buffers the graph reads and writes
    q_s, key_s, val_s, slot_s, lens_s = _step_inputs(plan[0])
    out_s = torch.empty_like(q_s)
    # first calls outside capture (per-device set-up), on throwaway caches
    step_calls(kc_e.clone(), vc_e.clone(), q_s, key_s, val_s, slot_s, lens_s, out_s, ws_g)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step_calls(kc_g, vc_g, q_s, key_s, val_s, slot_s, lens_s, out_s, ws_g)
    torch.cuda.synchronize()

    out_e = torch.empty_like(q_s)
    for i, st in enumerate(plan):
        q, key, value, slots, lens = _step_inputs(st)
        for dst, src in ((q_s, q), (key_s, key), (val_s, value), (slot_s, slots), (lens_s, lens)):
            dst.copy_(src)
        g.replay()
        step_calls(kc_e, vc_e, q, key, value, slots, lens, out_e, ws_e)
        torch.cuda.synchronize()
        assert torch.equal(out_s.view(torch.int16), out_e.view(torch.int16)), f"step {i}: out"
        assert torch.equal(kc_g, kc_e) and torch.equal(vc_g, vc_e), f"step {i}: cache bytes"

    # the oracle over the same writes: full fill, then each step's token
    kc_h, vc_h = U.oracle_write_cache(orc, case, kv_dtype, ks, vs)
    for st in plan:
        orc.reshape_and_cache(st.key, st.value, kc_h, vc_h, st.slot_mapping, case.num_kv_heads,
                              case.head_dim, case.block_size, case.num_blocks, kv_dtype, ks, vs)
    assert np.array_equal(kc_h, kc_g.cpu().numpy()) and np.array_equal(vc_h, vc_g.cpu().numpy())
    last = plan[-1]
    ref, _ = orc.decode(last.q, kc_h, vc_h, case.block_tables, last.seq_lens, case.num_kv_heads,
                        case.block_size, case.num_blocks, case.scale, 0, kv_dtype, ks, vs)
    got = out_s.view(torch.int16).cpu().numpy().view(np.uint16)
    U.assert_close(got, ref, what=f"graph replay vs oracle (kv_dtype {kv_dtype})")
