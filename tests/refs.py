"""Independent references used to pin the oracle (and, through it, the kernels).

Nothing here calls the oracle. Each helper reaches its result by a different
route from the oracle's code: torch's own float8_e4m3fn and bfloat16
conversions, brute-force nearest-grid searches over the format's value table,
numpy reshapes of the page layout, and torch's scaled_dot_product_attention in
float64.
"""
from __future__ import annotations

import numpy as np
import torch

# OCP Microscaling spec, E2M1 element values for codes 0..7 (bit 3 is the sign).
E2M1_TABLE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 code bytes -> float64 through torch.float8_e4m3fn."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def e4m3_encode_torch(x: np.ndarray) -> np.ndarray:
    """float32 -> E4M3 bytes through torch (valid where |x| <= 464: torch gives NaN above)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.int64)
    mag = E2M1_TABLE[codes & 7]
    return np.where(codes & 8, -mag, mag)


def _brute_nearest(x: np.ndarray, mags: np.ndarray) -> np.ndarray:
    """Index of the nearest magnitude in an ascending table (ties -> even index),
    saturating at the end of the table; NaN -> last index."""
    a = np.abs(x.astype(np.float64))
    a = np.where(np.isnan(a), np.inf, a)
    d = np.abs(a[:, None] - mags[None, :])
    best = np.argmin(d, axis=1)
    dmin = d[np.arange(len(a)), best]
    # a tie means a second index with the same distance; keep the even one
    tie = np.zeros(len(a), bool)
    alt = best.copy()
    for k in (-1, 1):
        j = np.clip(best + k, 0, len(mags) - 1)
        is_tie = (j != best) & (d[np.arange(len(a)), j] == dmin)
        alt = np.where(is_tie & (j % 2 == 0), j, alt)
        tie |= is_tie
    idx = np.where(tie, alt, best)
    # at or beyond the largest magnitude: saturate (also avoids float64 absorption)
    idx = np.where(a >= mags[-1], len(mags) - 1, idx)
    return idx


def brute_e2m1(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32).ravel()
    idx = _brute_nearest(x, E2M1_TABLE)
    return (idx | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def brute_e4m3(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32).ravel()
    mags = e4m3_decode(np.arange(127, dtype=np.uint8))  # codes 0..126 = 0 .. 448
    idx = _brute_nearest(x, mags)
    code = idx | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F | np.where(np.signbit(x), 0x80, 0), code)
    return code.astype(np.uint8)


# ---- page layout, read back independently --------------------------------
def nvfp4_geometry(block_size, num_kv_heads, head_dim):
    data = block_size * num_kv_heads * head_dim // 2
    raw = data + block_size * num_kv_heads * head_dim // 16
    stride = (raw + 127) // 128 * 128
    return data, stride


def dequant_pages(cache: np.ndarray, kv_dtype: int, num_blocks, block_size, num_kv_heads,
                  head_dim, scale=1.0) -> np.ndarray:
    """Whole cache -> float64 [num_blocks, block_size, num_kv_heads, head_dim]."""
    nb, bs, h, d = num_blocks, block_size, num_kv_heads, head_dim
    if kv_dtype == 0:
        return bf16_to_f64(cache[:nb * bs * h * d * 2].view(np.uint16)).reshape(nb, bs, h, d)
    if kv_dtype == 1:
        return e4m3_decode(cache[:nb * bs * h * d]).reshape(nb, bs, h, d) * np.float64(scale)
    data_bytes, stride = nvfp4_geometry(bs, h, d)
    pages = cache[:nb * stride].reshape(nb, stride)
    packed = pages[:, :data_bytes].reshape(nb, h, bs, d // 2)
    codes = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(nb, h, bs, d)
    scales = pages[:, data_bytes:data_bytes + bs * h * d // 16].reshape(nb, h, bs, d // 16)
    vals = e2m1_decode(codes) * np.repeat(e4m3_decode(scales), 16, axis=-1)
    return vals.transpose(0, 2, 1, 3)


def gather_sequence(pages: np.ndarray, block_table_row: np.ndarray, seq_len: int) -> np.ndarray:
    """Contiguous [L, Hkv, D] of one sequence from dequantised pages."""
    bs = pages.shape[1]
    j = np.arange(seq_len)
    return pages[block_table_row[j // bs], j % bs]


def sdpa_f64(q_bits: np.ndarray, kpages: np.ndarray, vpages: np.ndarray, block_tables,
             seq_lens, scale: float, sliding_window: int = 0) -> np.ndarray:
    """Reference attention in float64 via torch.nn.functional.scaled_dot_product_attention."""
    B, Hq, D = q_bits.shape
    hkv = kpages.shape[2]
    q = bf16_to_f64(q_bits)
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(seq_lens[b])
        lo = max(0, L - sliding_window) if sliding_window > 0 else 0
        if L - lo <= 0:
            continue
        K = gather_sequence(kpages, block_tables[b], L)[lo:]
        V = gather_sequence(vpages, block_tables[b], L)[lo:]
        Kt = torch.from_numpy(np.ascontiguousarray(K.transpose(1, 0, 2)))  # [Hkv, n, D]
        Vt = torch.from_numpy(np.ascontiguousarray(V.transpose(1, 0, 2)))
        g = Hq // hkv
        Kt = Kt.repeat_interleave(g, dim=0)
        Vt = Vt.repeat_interleave(g, dim=0)
        qt = torch.from_numpy(q[b]).unsqueeze(1)                           # [Hq, 1, D]
        o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=float(scale))
        out[b] = o[:, 0, :].numpy()
    return out


def prefill_f64(q_bits: np.ndarray, cu_q, kpages: np.ndarray, vpages: np.ndarray, block_tables,
                seq_lens, scale: float, causal: bool = True,
                sliding_window: int = 0) -> np.ndarray:
    """Reference paged prefill in float64: per sequence, one [q_len, Hq, L]
    score tensor with the causal / window mask, a masked softmax and one
    contraction with V (numpy einsum; no loop over keys)."""
    T, Hq, D = q_bits.shape
    hkv = kpages.shape[2]
    g = Hq // hkv
    q = bf16_to_f64(q_bits)
    out = np.zeros((T, Hq, D))
    for b in range(len(seq_lens)):
        L = int(seq_lens[b])
        r0, r1 = int(cu_q[b]), int(cu_q[b + 1])
        ql = r1 - r0
        if ql == 0:
            continue
        K = np.repeat(gather_sequence(kpages, block_tables[b], L), g, axis=1)  # [L, Hq, D]
        V = np.repeat(gather_sequence(vpages, block_tables[b], L), g, axis=1)
        pos = (L - ql + np.arange(ql)) if causal else np.full(ql, L - 1)
        j = np.arange(L)
        keep = j[None, :] <= pos[:, None]
        if sliding_window > 0:
            keep &= (pos[:, None] - j[None, :]) < sliding_window
        s = np.einsum("qhd,lhd->qhl", q[r0:r1], K) * float(scale)
        s = np.where(keep[:, None, :], s, -np.inf)
        s = s - s.max(axis=-1, keepdims=True)
        e = np.exp(s)
        e = e / e.sum(axis=-1, keepdims=True)
        out[r0:r1] = np.einsum("qhl,lhd->qhd", e, V)
    return out
