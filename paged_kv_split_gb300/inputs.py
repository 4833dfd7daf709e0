"""Seeded synthetic inputs for paged decode attention.

This module holds no arithmetic of the method: it only draws random numbers
and lays out the bookkeeping arrays (sequence lengths, page pool permutation,
block tables, slot mapping) that both the CUDA path and the CPU oracle
consume. Everything is derived from a splitmix64 counter stream, so a case is
reproduced exactly from its seeds on any machine.

Seeds: q = base+1, k = base+2, v = base+3, page permutation = base+4,
sequence lengths = base+5.

Workload shapes follow the configurations named in the benchmark plan: a tiny
GQA-2 case, a Llama-3-8B-shaped batch, long-context batches, wide-head and
sliding-window cases, and a quantised-cache batch with lognormal lengths.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset..offset+n-1 of the splitmix64 stream started at `seed`."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform01(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Doubles in (0, 1] from the top 53 bits of the stream."""
    z = splitmix64(seed, n, offset)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def normal_f32(seed: int, n: int) -> np.ndarray:
    """n standard normals (Box-Muller over consecutive uniform pairs), float32."""
    out = np.empty(n, np.float32)
    chunk = 1 << 24
    for start in range(0, n, chunk):
        m = min(chunk, n - start)
        pairs = (m + 1) // 2
        u = uniform01(seed, 2 * pairs, offset=start)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * math.pi * u2
        z = np.empty(2 * pairs, np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        out[start:start + m] = z[:m]
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), via torch's conversion."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def normal_bf16(seed: int, shape, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    x = normal_f32(seed, n)
    if std != 1.0:
        x = x * np.float32(std)
    return to_bf16_bits(x).reshape(shape)


def uniform_int(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] (inclusive)."""
    z = splitmix64(seed, n)
    return (lo + (z % np.uint64(hi - lo + 1)).astype(np.int64)).astype(np.int64)


def permutation(seed: int, n: int) -> np.ndarray:
    """A seeded random permutation of range(n) (argsort of random keys)."""
    return np.argsort(splitmix64(seed, n), kind="stable").astype(np.int64)


def lognormal_lengths(seed: int, n: int, mu: float, sigma: float, lo: int, hi: int) -> np.ndarray:
    u = uniform01(seed, 2 * n)
    z = np.sqrt(-2.0 * np.log(u[0::2])) * np.cos(2.0 * math.pi * u[1::2])
    return np.clip(np.round(np.exp(mu + sigma * z)), lo, hi).astype(np.int64)


@dataclass
class Case:
    """One decode workload: shapes, bookkeeping and host inputs."""
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    seq_lens: np.ndarray             # int32 [B]
    block_tables: np.ndarray         # int32 [B, MBS], unused entries -1
    num_blocks: int
    slot_mapping: np.ndarray         # int32 [T]
    q: np.ndarray                    # uint16 bf16 bits [B, Hq, D]
    key: np.ndarray                  # uint16 bf16 bits [T, Hkv, D]
    value: np.ndarray                # uint16 bf16 bits [T, Hkv, D]
    sliding_window: int = 0
    num_splits: int = 0
    kv_dtype: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return float(np.float32(1.0) / np.sqrt(np.float32(self.head_dim)))

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])


def make_case(name, seq_lens, num_q_heads, num_kv_heads, head_dim, block_size, *, seed=0,
              sliding_window=0, extra_blocks=0, max_blocks_per_seq=None, fill="all",
              num_splits=0, kv_dtype=0, q_std=1.0, kv_std=1.0) -> Case:
    """Build a paged case.

    Each sequence b owns ceil(L_b / block_size) pages taken in order from a
    seeded random permutation of the pool (num_blocks = total pages +
    extra_blocks). fill="all" writes every token of every sequence;
    fill="window" writes only the tokens inside the sliding window.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    B = len(seq_lens)
    pages = (seq_lens + block_size - 1) // block_size
    total_pages = int(pages.sum())
    num_blocks = total_pages + extra_blocks
    mbs = int(max_blocks_per_seq or max(1, int(pages.max()) if B else 1))
    perm = permutation(seed + 4, num_blocks)
    bt = np.full((B, mbs), -1, np.int32)
    off = 0
    for b in range(B):
        p = int(pages[b])
        bt[b, :p] = perm[off:off + p]
        off += p
    # slot mapping: token j of sequence b -> page bt[b, j // bs], row j % bs
    slots = []
    for b in range(B):
        L = int(seq_lens[b])
        lo = 0
        if fill == "window" and sliding_window > 0:
            lo = max(0, L - sliding_window)
        j = np.arange(lo, L, dtype=np.int64)
        slots.append(bt[b, j // block_size].astype(np.int64) * block_size + j % block_size)
    slot_mapping = (np.concatenate(slots) if slots else np.zeros(0, np.int64)).astype(np.int32)
    T = slot_mapping.shape[0]
    q = normal_bf16(seed + 1, (B, num_q_heads, head_dim), q_std)
    key = normal_bf16(seed + 2, (T, num_kv_heads, head_dim), kv_std)
    value = normal_bf16(seed + 3, (T, num_kv_heads, head_dim), kv_std)
    return Case(name=name, num_seqs=B, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, block_size=block_size, seq_lens=seq_lens.astype(np.int32),
                block_tables=bt, num_blocks=num_blocks, slot_mapping=slot_mapping, q=q, key=key,
                value=value, sliding_window=sliding_window, num_splits=num_splits,
                kv_dtype=kv_dtype)


@dataclass
class DecodeStep:
    """The inputs of one decode step that appends a token to every sequence."""
    q: np.ndarray             # uint16 bf16 bits [B, Hq, D]
    key: np.ndarray           # uint16 bf16 bits [B, Hkv, D], the new token's K
    value: np.ndarray         # uint16 bf16 bits [B, Hkv, D], the new token's V
    slot_mapping: np.ndarray  # int32 [B], slot of the new token
    seq_lens: np.ndarray      # int32 [B], lengths including the new token


def decode_steps(case: Case, steps: int, seed: int = 0) -> list:
    """`steps` decode steps over `case`, whose lengths are the lengths after
    the last step: step i appends position L_b - steps + i of sequence b
    (its page is already in the block table) and attends over L_b - steps +
    i + 1 keys. Sequences shorter than `steps` are not allowed."""
    B = case.num_seqs
    L_final = case.seq_lens.astype(np.int64)
    if B and int(L_final.min()) < steps:
        raise ValueError("every sequence needs at least `steps` tokens")
    bs = case.block_size
    out = []
    for i in range(steps):
        pos = L_final - steps + i
        page = case.block_tables[np.arange(B), pos // bs].astype(np.int64)
        slots = (page * bs + pos % bs).astype(np.int32)
        out.append(DecodeStep(
            q=normal_bf16(seed + 100 + 3 * i, (B, case.num_q_heads, case.head_dim)),
            key=normal_bf16(seed + 101 + 3 * i, (B, case.num_kv_heads, case.head_dim)),
            value=normal_bf16(seed + 102 + 3 * i, (B, case.num_kv_heads, case.head_dim)),
            slot_mapping=slots, seq_lens=(pos + 1).astype(np.int32)))
    return out


# ---- the named workloads -------------------------------------------------
def tiny(num_splits: int = 1, seed: int = 0) -> Case:
    """2 seqs {17, 40}, 4 q / 2 kv heads, D=64, bs=16, a 16-page pool."""
    return make_case("tiny_bf16", [17, 40], 4, 2, 64, 16, seed=seed, extra_blocks=11,
                     num_splits=num_splits)


def llama8b(seed: int = 0, num_seqs: int = 32, lo: int = 1024, hi: int = 4096) -> Case:
    """Batch 32, 32 q / 8 kv heads, D=128, bs=16, L ~ U[1024, 4096]."""
    lens = uniform_int(seed + 5, num_seqs, lo, hi)
    return make_case(f"llama8b_b{num_seqs}", lens, 32, 8, 128, 16, seed=seed)


def long_context(num_seqs: int, seq_len: int, num_splits: int = 0, seed: int = 0) -> Case:
    """Batch 1 or 4 at 1K / 8K / 32K, 32 q / 8 kv heads, D=128, bs=32."""
    return make_case(f"long_b{num_seqs}_{seq_len}", [seq_len] * num_seqs, 32, 8, 128, 32,
                     seed=seed, num_splits=num_splits)


def wide_head(seed: int = 0, num_seqs: int = 8, seq_len: int = 8192) -> Case:
    """Batch 8, 16 q / 2 kv heads, D=512, L=8192, bs=16."""
    return make_case(f"wide_d512_b{num_seqs}_{seq_len}", [seq_len] * num_seqs, 16, 2, 512, 16,
                     seed=seed)


def sliding(seed: int = 0, num_seqs: int = 8, seq_len: int = 16384, window: int = 4096,
            fill: str = "window") -> Case:
    """Batch 8, 8 q / 4 kv heads, D=256, L=16384, sliding window 4096, bs=16."""
    return make_case(f"window_d256_b{num_seqs}_{seq_len}_w{window}", [seq_len] * num_seqs, 8, 4,
                     256, 16, seed=seed, sliding_window=window, fill=fill)


def quantised(kv_dtype: int, seed: int = 0, num_seqs: int = 64, lo: int = 512,
              hi: int = 16384) -> Case:
    """Batch 64, 64 q / 8 kv heads, D=128, bs=16, L lognormal(ln 2048, 1) in [512, 16384]."""
    lens = lognormal_lengths(seed + 5, num_seqs, math.log(2048.0), 1.0, lo, hi)
    tag = {1: "fp8", 2: "nvfp4"}[kv_dtype]
    return make_case(f"quant_{tag}_b{num_seqs}", lens, 64, 8, 128, 16, seed=seed,
                     kv_dtype=kv_dtype)


def make_prefill_case(name, seq_lens, q_lens, num_q_heads, num_kv_heads, head_dim, block_size,
                      *, seed=0, sliding_window=0, extra_blocks=0, q_std=1.0,
                      kv_std=1.0) -> Case:
    """A chunked-prefill workload over the same paged cache: every token of
    every sequence is in the cache (as in make_case), and sequence b has
    q_lens[b] query rows, its newest tokens. q becomes [sum(q_lens), Hq, D];
    extra["cu_q"] holds the row offsets [B+1] and extra["q_lens"] the lengths."""
    case = make_case(name, seq_lens, num_q_heads, num_kv_heads, head_dim, block_size, seed=seed,
                     sliding_window=sliding_window, extra_blocks=extra_blocks, q_std=q_std,
                     kv_std=kv_std)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    assert q_lens.shape == (case.num_seqs,) and np.all(q_lens <= case.seq_lens)
    cu_q = np.zeros(case.num_seqs + 1, np.int32)
    cu_q[1:] = np.cumsum(q_lens)
    case.q = normal_bf16(seed + 6, (int(cu_q[-1]), num_q_heads, head_dim), q_std)
    case.extra["cu_q"] = cu_q
    case.extra["q_lens"] = q_lens
    return case


def prefill_chunked(seed: int = 0, num_seqs: int = 8, chunk: int = 512,
                    max_context: int = 3584) -> Case:
    """Chunked prefill at Llama-3-8B shapes (32 q / 8 kv heads, D=128, bs=16):
    each of num_seqs sequences adds a chunk of `chunk` tokens after a context
    of U[0, max_context] tokens already in the cache."""
    ctx = uniform_int(seed + 5, num_seqs, 0, max_context)
    lens = ctx + chunk
    return make_prefill_case(f"prefill_b{num_seqs}_c{chunk}", lens, np.full(num_seqs, chunk),
                             32, 8, 128, 16, seed=seed)
