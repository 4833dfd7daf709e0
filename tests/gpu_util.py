"""Helpers for the GPU parity tests: run a case through libpd.so (C ABI, via
the binding) and through the oracle on the same inputs, and compare."""
from __future__ import annotations

import json
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

SENTINEL = 0xA5
ATOL = 1e-2
RTOL = 1e-2


def pd():
    from paged_kv_split_gb300 import binding
    return binding


def to_dev(a: np.ndarray, dtype=None, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


def bf16_dev(bits: np.ndarray, device="cuda"):
    return to_dev(bits.view(np.int16), device=device).view(torch.bfloat16)


def gpu_write_cache(case, kv_dtype, k_scale=1.0, v_scale=1.0, device="cuda"):
    """Sentinel-filled caches written by pd_reshape_and_cache; returns device tensors."""
    B = pd()
    kc = B.empty_cache(kv_dtype, case.num_blocks, case.block_size, case.num_kv_heads,
                       case.head_dim, device)
    vc = torch.empty_like(kc)
    kc.fill_(SENTINEL)
    vc.fill_(SENTINEL)
    key = bf16_dev(case.key, device)
    value = bf16_dev(case.value, device)
    slots = to_dev(case.slot_mapping, device=device)
    B.pd_reshape_and_cache(key, value, kc, vc, slots, num_blocks=case.num_blocks,
                           block_size=case.block_size, kv_dtype=kv_dtype, k_scale=k_scale,
                           v_scale=v_scale)
    return kc, vc


def oracle_write_cache(orc, case, kv_dtype, k_scale=1.0, v_scale=1.0):
    n = orc.cache_bytes(kv_dtype, case.num_blocks, case.block_size, case.num_kv_heads,
                        case.head_dim)
    kc = np.full(n, SENTINEL, np.uint8)
    vc = np.full(n, SENTINEL, np.uint8)
    orc.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping, case.num_kv_heads,
                          case.head_dim, case.block_size, case.num_blocks, kv_dtype, k_scale,
                          v_scale)
    return kc, vc


def gpu_decode(case, kc, vc, kv_dtype, num_splits, k_scale=1.0, v_scale=1.0, device="cuda",
               block_tables=None, window=None):
    B = pd()
    q = bf16_dev(case.q, device)
    bt = to_dev(case.block_tables if block_tables is None else block_tables, device=device)
    lens = to_dev(case.seq_lens, device=device)
    out = torch.empty_like(q)
    w = case.sliding_window if window is None else window
    B.pd_decode(q, kc, vc, bt, lens, out, num_kv_heads=case.num_kv_heads,
                block_size=case.block_size, num_blocks=case.num_blocks, scale=case.scale,
                num_splits=num_splits, sliding_window=w, kv_dtype=kv_dtype,
                k_scale=k_scale, v_scale=v_scale)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_decode(orc, case, kc_host, vc_host, kv_dtype, k_scale=1.0, v_scale=1.0,
                  block_tables=None, window=None, threads=16):
    """The oracle over all sequences, split by sequence across threads (the
    ctypes call releases the GIL; each call is the plain single-threaded oracle)."""
    bt = case.block_tables if block_tables is None else block_tables
    w = case.sliding_window if window is None else window
    Bn = case.num_seqs
    chunks = [c for c in np.array_split(np.arange(Bn), min(threads, max(Bn, 1))) if len(c)]

    def run(idx):
        lo, hi = int(idx[0]), int(idx[-1]) + 1
        return orc.decode(case.q[lo:hi], kc_host, vc_host, bt[lo:hi], case.seq_lens[lo:hi],
                          case.num_kv_heads, case.block_size, case.num_blocks, case.scale, w,
                          kv_dtype, k_scale, v_scale)

    with ThreadPoolExecutor(len(chunks)) as ex:
        parts = list(ex.map(run, chunks))
    out = np.concatenate([p[0] for p in parts]) if parts else np.zeros(case.q.shape, np.uint16)
    out_f32 = np.concatenate([p[1] for p in parts]) if parts else np.zeros(case.q.shape,
                                                                          np.float32)
    return out, out_f32


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def assert_close(gpu_bits, ref_bits, atol=ATOL, rtol=RTOL, what=""):
    """|gpu - oracle| <= atol + rtol * |oracle| elementwise, on bf16 outputs."""
    g = bf16_bits_to_f32(gpu_bits).astype(np.float64)
    r = bf16_bits_to_f32(ref_bits).astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - r)
    bound = atol + rtol * np.abs(r)
    bad = err > bound
    log = os.environ.get("PD_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": what, "n": int(err.size), "max_abs_err": float(err.max()),
                                "max_err_over_bound": float((err / bound).max()),
                                "max_abs_ref": float(np.abs(r).max())}) + "\n")
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at "
                             f"{tuple(i)}: gpu {g[tuple(i)]} oracle {r[tuple(i)]}; "
                             f"max err {err.max():.3g}")
    return float(err.max())


def fp8_scales(orc, case):
    return (orc.fp8_scale(orc.absmax_bf16(case.key)), orc.fp8_scale(orc.absmax_bf16(case.value)))
