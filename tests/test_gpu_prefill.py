"""Paged prefill (pd_prefill) against the oracle, through the C ABI.

Small cases compare every output element with oracle_prefill on the same
cache bytes; the chunked-prefill workload at full size compares sampled
query rows, each computed by the oracle as its own decode over the keys the
row sees (the oracle pins make that bit-identical to oracle_prefill).
Edge cases: empty sequences, a fresh prompt (q_len == L), one query per
sequence, group sizes that do not divide the CTA's rows, more work items
than the tcgen05 kernel ranks, a q_len above max_q_len, pages outside the
pool, strided rows and graph replay. Every test
runs on both kernels (tcgen05 through pd_prefill, mma.sync through
pd_prefill_crosscheck)."""
import functools
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from paged_kv_split_gb300 import inputs
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["tcgen05", "mma_sync"], autouse=True)
def prefill_kernel(request, monkeypatch):
    """Every test runs on both prefill kernels: pd_prefill (tcgen05) and
    pd_prefill_crosscheck (mma.sync), chosen through the binding's
    `crosscheck` argument."""
    if request.param == "mma_sync":
        from paged_kv_split_gb300 import binding as B
        monkeypatch.setattr(B, "pd_prefill", functools.partial(B.pd_prefill, crosscheck=True))
        monkeypatch.setattr(B, "pd_prefill_strided",
                            functools.partial(B.pd_prefill_strided, crosscheck=True))
    return request.param

CASES = [
    # (name, seq_lens, q_lens, Hq, Hkv, D, bs, window)
    ("two_seq_d64", [17, 40], [17, 9], 4, 2, 64, 16, 0),
    ("three_seq", [70, 33, 5], [16, 33, 1], 8, 2, 64, 16, 0),
    ("d128_bs32", [64, 31], [40, 3], 16, 2, 128, 32, 0),
    ("window", [69, 50], [23, 50], 4, 1, 64, 16, 20),
    ("g1_long_chunk", [300, 129], [150, 129], 8, 8, 128, 16, 0),
    ("g3", [200, 77], [90, 40], 12, 4, 128, 16, 0),
    ("g16", [150, 60], [33, 60], 16, 1, 64, 32, 0),
    ("g8_window_ragged", [500, 211, 64], [130, 211, 1], 32, 4, 128, 16, 100),
    ("empty_and_zero_q", [0, 90, 40], [0, 0, 40], 8, 2, 64, 16, 0),
    # two query tiles per CTA: tiles whose windows barely overlap, a partial
    # second tile, head_dim 64 with 32-row pages
    ("pair_window_g1", [600, 260], [300, 260], 4, 4, 128, 16, 32),
    ("pair_g4_bs32", [900, 140], [200, 140], 16, 4, 64, 32, 64),
    ("d256", [300, 77], [130, 77], 8, 2, 256, 16, 0),
    ("d256_g8_window_bs32", [400, 129], [200, 64], 16, 2, 256, 32, 100),
]


def _case(spec, seed_base=500):
    name, lens, qls, hq, hkv, d, bs, w = spec
    return inputs.make_prefill_case(name, lens, qls, hq, hkv, d, bs,
                                    seed=seed_base + zlib.crc32(name.encode()) % 1000,
                                    sliding_window=w, extra_blocks=2)


def gpu_prefill(case, kc, vc, causal=True, max_q_len=None, block_tables=None, kv_dtype=0,
                k_scale=1.0, v_scale=1.0):
    from paged_kv_split_gb300 import binding as B
    cu = case.extra["cu_q"]
    q = U.bf16_dev(case.q)
    out = torch.full_like(q, float("nan"))
    mq = int(case.extra["q_lens"].max()) if max_q_len is None else max_q_len
    bt = case.block_tables if block_tables is None else block_tables
    B.pd_prefill(q, U.to_dev(cu), kc, vc, U.to_dev(bt), U.to_dev(case.seq_lens), out,
                 max_q_len=mq, num_kv_heads=case.num_kv_heads, block_size=case.block_size,
                 num_blocks=case.num_blocks, scale=case.scale, causal=causal,
                 sliding_window=case.sliding_window, kv_dtype=kv_dtype, k_scale=k_scale,
                 v_scale=v_scale)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_prefill(orc, case, kc_host, vc_host, causal=True, threads=16, kv_dtype=0,
                   k_scale=1.0, v_scale=1.0):
    """oracle_prefill, one call per sequence on a thread pool (the ctypes call
    releases the GIL; each call is the plain single-threaded oracle)."""
    cu = case.extra["cu_q"]

    def run(b):
        r0, r1 = int(cu[b]), int(cu[b + 1])
        sub_cu = np.array([0, r1 - r0], np.int32)
        return orc.prefill(case.q[r0:r1], sub_cu, kc_host, vc_host, case.block_tables[b:b + 1],
                           case.seq_lens[b:b + 1], case.num_kv_heads, case.block_size,
                           case.num_blocks, case.scale, causal, case.sliding_window, kv_dtype,
                           k_scale, v_scale)[0]

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(run, range(case.num_seqs)))
    return np.concatenate(parts) if parts else np.zeros(case.q.shape, np.uint16)


@pytest.mark.parametrize("kv_dtype", [0, 1, 2], ids=["bf16", "fp8", "nvfp4"])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
@pytest.mark.parametrize("spec", CASES, ids=[c[0] for c in CASES])
def test_small_parity(orc, spec, causal, kv_dtype):
    """Every element against oracle_prefill, the quantised caches read from the
    same GPU-written bytes (checked bit-exact against the oracle's first)."""
    case = _case(spec)
    ks, vs = U.fp8_scales(orc, case) if kv_dtype == 1 else (1.0, 1.0)
    kc, vc = U.gpu_write_cache(case, kv_dtype, ks, vs)
    kh, vh = kc.cpu().numpy(), vc.cpu().numpy()
    if kv_dtype:
        okc, ovc = U.oracle_write_cache(orc, case, kv_dtype, ks, vs)
        assert np.array_equal(kh, okc) and np.array_equal(vh, ovc), "cache bytes differ"
    got = gpu_prefill(case, kc, vc, causal, kv_dtype=kv_dtype, k_scale=ks, v_scale=vs)
    ref = oracle_prefill(orc, case, kh, vh, causal, kv_dtype=kv_dtype, k_scale=ks, v_scale=vs)
    U.assert_close(got, ref, what=f"prefill {case.name} causal={causal} dtype={kv_dtype}")


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_more_items_than_ranked(orc, causal):
    """More (sequence, pair of query tiles) items than the tcgen05 kernel ranks
    by cost (256): 40 sequences, two of them with 500-row chunks, so every
    sequence has 8 pair slots (320 items) and the CTAs take them in grid
    order instead; most slots have no rows. Every element against the
    oracle."""
    lens = [520, 517] + [30 + 7 * i for i in range(38)]
    qls = [500, 497] + [1 + i % 5 for i in range(38)]
    case = inputs.make_prefill_case("many_items", lens, qls, 8, 2, 64, 16, seed=811,
                                    extra_blocks=2)
    kc, vc = U.gpu_write_cache(case, 0, 1.0, 1.0)
    got = gpu_prefill(case, kc, vc, causal)
    ref = oracle_prefill(orc, case, kc.cpu().numpy(), vc.cpu().numpy(), causal)
    U.assert_close(got, ref, what=f"prefill many items causal={causal}")


def test_fresh_prompt_first_row_is_its_value(orc):
    """L == q_len: query 0 sees key 0 alone; bf16 V passes through exactly."""
    case = inputs.make_prefill_case("fresh", [130, 64], [130, 64], 8, 2, 128, 16, seed=61)
    kc, vc = U.gpu_write_cache(case, 0)
    got = gpu_prefill(case, kc, vc)
    cu = case.extra["cu_q"]
    g = case.num_q_heads // case.num_kv_heads
    for b in range(case.num_seqs):
        v0 = case.value[int(np.sum(case.seq_lens[:b]))]
        for h in range(case.num_q_heads):
            assert np.array_equal(got[cu[b], h], v0[h // g])


def test_one_query_per_sequence_matches_decode(orc):
    case = inputs.make_prefill_case("as_decode", [700, 45, 1, 300], [1, 1, 1, 1], 32, 8, 128, 16,
                                    seed=62)
    kc, vc = U.gpu_write_cache(case, 0)
    got = gpu_prefill(case, kc, vc)
    ref, _ = U.oracle_decode(orc, case, kc.cpu().numpy(), vc.cpu().numpy(), 0)
    U.assert_close(got, ref, what="prefill q_len=1")
    dec = U.gpu_decode(case, kc, vc, 0, 0)
    U.assert_close(got, dec, what="prefill q_len=1 vs pd_decode")


def test_q_len_above_max_q_len_is_flagged():
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_prefill_case("over", [100, 100], [80, 20], 8, 2, 64, 16, seed=63)
    kc, vc = U.gpu_write_cache(case, 0)
    B.pd_device_status(reset=True)
    gpu_prefill(case, kc, vc, max_q_len=40)
    assert B.pd_device_status(reset=True) & 2  # PD_DEV_BAD_SEQ_LEN


def test_page_outside_the_pool_is_flagged_not_faulted(orc):
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_prefill_case("badpage", [200, 90], [60, 90], 8, 2, 128, 16, seed=64)
    kc, vc = U.gpu_write_cache(case, 0)
    bt = case.block_tables.copy()
    bt[0, 2] = case.num_blocks + 5  # keys 32..47 of sequence 0 are gone
    B.pd_device_status(reset=True)
    got = gpu_prefill(case, kc, vc, block_tables=bt)
    assert B.pd_device_status(reset=True) & 1  # PD_DEV_BAD_PAGE
    assert np.all(np.isfinite(U.bf16_bits_to_f32(got)))
    # sequence 1 does not touch the bad page: still exact to the oracle
    ref = oracle_prefill(orc, case, kc.cpu().numpy(), vc.cpu().numpy())
    cu = case.extra["cu_q"]
    U.assert_close(got[cu[1]:cu[2]], ref[cu[1]:cu[2]], what="prefill bad page, other sequence")


def test_strided_rows_are_bit_identical():
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_prefill_case("strided", [300, 77], [120, 77], 32, 8, 128, 16, seed=65)
    kc, vc = U.gpu_write_cache(case, 0)
    packed = gpu_prefill(case, kc, vc)
    T, hq, d = case.q.shape
    row = hq * d + 2 * 8 * d  # a fused QKV row: q heads, then k and v heads
    q_rows = torch.zeros(T, row, dtype=torch.bfloat16, device="cuda")
    q_rows[:, :hq * d] = U.bf16_dev(case.q).view(T, hq * d)
    out_rows = torch.full((T, hq * d + 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.pd_prefill_strided(q_rows, U.to_dev(case.extra["cu_q"]), kc, vc,
                         U.to_dev(case.block_tables), U.to_dev(case.seq_lens), out_rows,
                         num_q_heads=hq, head_dim=d, max_q_len=120,
                         num_kv_heads=case.num_kv_heads, block_size=case.block_size,
                         num_blocks=case.num_blocks, scale=case.scale)
    torch.cuda.synchronize()
    got = out_rows[:, :hq * d].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got.reshape(T, hq, d), packed)
    assert torch.isnan(out_rows[:, hq * d:].float()).all()  # padding untouched


def test_graph_replay_is_bit_exact():
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_prefill_case("graph", [400, 150], [128, 150], 32, 8, 128, 16, seed=66)
    kc, vc = U.gpu_write_cache(case, 0)
    eager = gpu_prefill(case, kc, vc)
    q = U.bf16_dev(case.q)
    cu, bt, lens = (U.to_dev(case.extra["cu_q"]), U.to_dev(case.block_tables),
                    U.to_dev(case.seq_lens))
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            B.pd_prefill(q, cu, kc, vc, bt, lens, out, max_q_len=150,
                         num_kv_heads=case.num_kv_heads, block_size=case.block_size,
                         num_blocks=case.num_blocks, scale=case.scale)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), eager)


def test_unsupported_forms_are_refused():
    from paged_kv_split_gb300 import binding as B
    case = inputs.make_prefill_case("unsup", [40], [8], 8, 2, 512, 16, seed=67)
    kc, vc = U.gpu_write_cache(case, 0)
    q = U.bf16_dev(case.q)
    out = torch.empty_like(q)
    for kw in ({"kv_dtype": 0}, {"kv_dtype": 2}):  # head_dim 512 is not built for prefill
        with pytest.raises(B.PdError):
            B.pd_prefill(q, U.to_dev(case.extra["cu_q"]), kc, vc, U.to_dev(case.block_tables),
                         U.to_dev(case.seq_lens), out, max_q_len=8,
                         num_kv_heads=case.num_kv_heads, block_size=case.block_size,
                         num_blocks=case.num_blocks, scale=case.scale, **kw)


# ---- the chunked-prefill workload at full size, every row ------------------
_FULL_REF = {}


def _oracle_prefill_row_blocks(orc, case, kh, vh, parts=4, threads=16):
    """Causal oracle_prefill over every query row, each sequence cut into
    `parts` blocks of rows so that all host cores work. Rows [i0, i1) of a
    sequence with L keys and q_len queries are presented as their own
    sequence of i1 - i0 queries over its first L - q_len + i1 keys: query j
    then sits at position L - q_len + i0 + j and sees exactly the keys that
    row i0 + j sees in the whole sequence."""
    cu = case.extra["cu_q"]
    tasks = []
    for b in range(case.num_seqs):
        ql, L = int(cu[b + 1] - cu[b]), int(case.seq_lens[b])
        edges = np.linspace(0, ql, parts + 1).astype(int)
        tasks += [(b, int(i0), int(i1), L, ql) for i0, i1 in zip(edges[:-1], edges[1:]) if i1 > i0]

    def run(t):
        b, i0, i1, L, ql = t
        r0 = int(cu[b])
        return orc.prefill(case.q[r0 + i0:r0 + i1], np.array([0, i1 - i0], np.int32), kh, vh,
                           case.block_tables[b:b + 1], np.array([L - ql + i1], np.int32),
                           case.num_kv_heads, case.block_size, case.num_blocks, case.scale,
                           True, case.sliding_window)[0]

    with ThreadPoolExecutor(threads) as ex:
        parts_out = list(ex.map(run, tasks))
    return np.concatenate(parts_out)


def test_chunked_prefill_workload_every_row(orc):
    """The bench's chunked-prefill workload (8 sequences, 512-token chunks after
    up to 3584 cached tokens, 32 q / 8 kv heads, D=128): every element of all
    4096 query rows against oracle_prefill, on both kernels (the oracle's
    result is computed once per process and reused)."""
    case = inputs.prefill_chunked()
    kc, vc = U.gpu_write_cache(case, 0)
    got = gpu_prefill(case, kc, vc)
    assert np.all(np.isfinite(U.bf16_bits_to_f32(got)))
    if case.name not in _FULL_REF:
        _FULL_REF[case.name] = _oracle_prefill_row_blocks(orc, case, kc.cpu().numpy(),
                                                          vc.cpu().numpy())
    ref = _FULL_REF[case.name]
    assert got.shape == ref.shape == (int(case.extra["cu_q"][-1]), case.num_q_heads,
                                      case.head_dim)
    U.assert_close(got, ref, what=f"prefill {case.name} (all {got.shape[0]} rows)")
