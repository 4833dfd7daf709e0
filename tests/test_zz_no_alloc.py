"""pd_decode_static_ws: the decode entry point that allocates nothing.

It serves callers that are only given their inputs and outputs and cannot
call cudaMalloc (an operator hosted inside another runtime that owns all
device memory, or code with a fixed memory budget). Its split workspace is
a fixed array inside libpd.so. This file runs last so that a failure here
never hides the other tests; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_split_gb300 import inputs
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

_P, _i32, _i64, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float


def _static_ws_fn():
    from paged_kv_split_gb300 import binding
    f = binding.lib().pd_decode_static_ws
    f.argtypes = [_P, _P, _P, _P, _P, _P, _i32, _i32, _i32, _i32, _i32, _i32, _i64, _f32, _i32,
                  _i32, _i32, _f32, _f32, _P]
    f.restype = ctypes.c_int
    return f


def _call_static(f, case, kc, vc, S, kv_dtype=0, k_scale=1.0, v_scale=1.0, free_mem=None):
    """One pd_decode_static_ws call through the C ABI. Its inputs and output
    are allocated (by torch) first; when `free_mem` is a list, the device's
    free memory just before and just after the call itself is appended."""
    q = U.bf16_dev(case.q)
    bt = U.to_dev(case.block_tables)
    lens = U.to_dev(case.seq_lens)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    if free_mem is not None:
        free_mem.append(torch.cuda.mem_get_info()[0])
    rc = f(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), lens.data_ptr(),
           out.data_ptr(), case.num_seqs, case.num_q_heads, case.num_kv_heads, case.head_dim,
           case.block_size, case.max_blocks_per_seq, case.num_blocks, case.scale, S,
           case.sliding_window, kv_dtype, k_scale, v_scale, stream)
    torch.cuda.synchronize()
    if free_mem is not None:
        free_mem.append(torch.cuda.mem_get_info()[0])
    return rc, out.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_static_workspace_matches_pd_decode_twice_in_a_row(orc):
    """Same kernels, same split count, same inputs: the output equals
    pd_decode's bit for bit, for every cache form, on two calls in a row that
    follow a larger call (so the shared array holds another call's partials),
    and the device's free memory does not move across the calls."""
    f = _static_ws_fn()
    big = inputs.make_case("nalloc_big_first", [3000, 2500, 4000, 1000], 32, 8, 128, 16,
                           seed=500)
    kb, vb = U.gpu_write_cache(big, 0)
    rc, _ = _call_static(f, big, kb, vb, 16)
    assert rc == 0
    cases = [
        (inputs.make_case("nalloc_a", [700, 33, 1290], 32, 8, 128, 16, seed=501), 0, 5),
        (inputs.make_case("nalloc_b", [64, 2000], 16, 2, 256, 16, seed=502, sliding_window=900),
         0, 0),
        (inputs.make_case("nalloc_fp8", [900, 17, 1500], 32, 8, 128, 16, seed=504), 1, 3),
        (inputs.make_case("nalloc_nvfp4", [1200, 5, 611], 64, 8, 128, 16, seed=505), 2, 0),
    ]
    for case, kv_dtype, S in cases:
        ks, vs = U.fp8_scales(orc, case) if kv_dtype == 1 else (1.0, 1.0)
        kc, vc = U.gpu_write_cache(case, kv_dtype, ks, vs)
        want = U.gpu_decode(case, kc, vc, kv_dtype, S, ks, vs)
        for _ in range(2):
            free = []
            rc, got = _call_static(f, case, kc, vc, S, kv_dtype, ks, vs, free_mem=free)
            assert rc == 0, f"pd_decode_static_ws returned {rc}"
            assert free[0] == free[1], f"device free memory moved by {free[0] - free[1]} bytes"
            assert np.array_equal(got, want), f"static workspace differs from pd_decode ({case.name})"


def test_static_workspace_refuses_oversize_requests():
    from paged_kv_split_gb300 import binding
    f = _static_ws_fn()
    case = inputs.make_case("nalloc_big", [40] * 8, 64, 8, 512, 16, seed=503)
    need = binding.pd_decode_workspace_bytes(case.num_seqs, 64, 512, 1024)
    assert need > (8 << 20)
    kc, vc = U.gpu_write_cache(case, 0)
    rc, _ = _call_static(f, case, kc, vc, 1024)
    assert rc == 3  # PD_ERR_WORKSPACE_TOO_SMALL, before anything is launched
