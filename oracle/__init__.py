"""ctypes binding for the plain CPU oracle in ``pd_oracle.cpp``.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of bench.py may import this
package. The product package ``paged_kv_split_gb300`` never imports it, and
the two share no code.

Arrays are numpy; bf16 tensors travel as ``uint16`` bit patterns and caches
as ``uint8`` byte arrays laid out exactly like the device caches.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pd_oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")
_lock = threading.Lock()

KV_BF16, KV_FP8_E4M3, KV_NVFP4 = 0, 1, 2

# fp32 arithmetic exactly as written: no contraction into FMA, no fast-math.
CXXFLAGS = ["-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def compile_source(src: str, out: str) -> str:
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["g++", *CXXFLAGS, "-o", tmp, src], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++ if it is missing or older than the source."""
    with _lock:
        stale = (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)
        if force or stale:
            compile_source(SRC, LIB)
    return LIB


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


class Oracle:
    """One loaded copy of the oracle library (the default one, or a test copy)."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f32, u8, u16 = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                  ctypes.c_uint8, ctypes.c_uint16)
        L.oracle_bf16_value.argtypes, L.oracle_bf16_value.restype = [u16], f32
        L.oracle_bf16_round.argtypes, L.oracle_bf16_round.restype = [f32], u16
        L.oracle_e4m3_value.argtypes, L.oracle_e4m3_value.restype = [u8], f32
        L.oracle_e4m3_code.argtypes, L.oracle_e4m3_code.restype = [f32], u8
        L.oracle_e2m1_value.argtypes, L.oracle_e2m1_value.restype = [u8], f32
        L.oracle_e2m1_code.argtypes, L.oracle_e2m1_code.restype = [f32], u8
        L.oracle_e4m3_code_array.argtypes, L.oracle_e4m3_code_array.restype = [P, i64, P], None
        L.oracle_e2m1_code_array.argtypes, L.oracle_e2m1_code_array.restype = [P, i64, P], None
        L.oracle_page_bytes.argtypes, L.oracle_page_bytes.restype = [i32, i32, i32, i32], i64
        L.oracle_absmax_bf16.argtypes, L.oracle_absmax_bf16.restype = [P, i64], f32
        L.oracle_fp8_scale.argtypes, L.oracle_fp8_scale.restype = [f32], f32
        L.oracle_reshape_and_cache.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64, i32, f32,
                                               f32]
        L.oracle_reshape_and_cache.restype = ctypes.c_int
        L.oracle_decode.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64,
                                    f32, i32, i32, f32, f32]
        L.oracle_decode.restype = ctypes.c_int
        L.oracle_decode_e4m3_out.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                             i64, f32, i32, i32, f32, f32, f32]
        L.oracle_decode_e4m3_out.restype = ctypes.c_int
        L.oracle_prefill.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64,
                                     f32, i32, i32, i32, f32, f32]
        L.oracle_prefill.restype = ctypes.c_int
        self.lib = L
        self.path = path

    # ---- codecs ---------------------------------------------------------
    def bf16_value(self, b: int) -> float:
        return self.lib.oracle_bf16_value(int(b))

    def bf16_round(self, x: float) -> int:
        return self.lib.oracle_bf16_round(float(x))

    def e4m3_value(self, c: int) -> float:
        return self.lib.oracle_e4m3_value(int(c))

    def e2m1_value(self, c: int) -> float:
        return self.lib.oracle_e2m1_value(int(c))

    def e4m3_code(self, x: float) -> int:
        return self.lib.oracle_e4m3_code(float(x))

    def e2m1_code(self, x: float) -> int:
        return self.lib.oracle_e2m1_code(float(x))

    def e4m3_codes(self, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, np.uint8)
        self.lib.oracle_e4m3_code_array(_ptr(x), x.size, _ptr(out))
        return out

    def e2m1_codes(self, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, np.uint8)
        self.lib.oracle_e2m1_code_array(_ptr(x), x.size, _ptr(out))
        return out

    # ---- cache ----------------------------------------------------------
    def page_bytes(self, kv_dtype: int, block_size: int, num_kv_heads: int,
                   head_dim: int) -> int:
        return int(self.lib.oracle_page_bytes(kv_dtype, block_size, num_kv_heads, head_dim))

    def cache_bytes(self, kv_dtype, num_blocks, block_size, num_kv_heads, head_dim) -> int:
        return num_blocks * self.page_bytes(kv_dtype, block_size, num_kv_heads, head_dim)

    def absmax_bf16(self, data: np.ndarray) -> float:
        data = np.ascontiguousarray(data, dtype=np.uint16)
        return float(self.lib.oracle_absmax_bf16(_ptr(data), data.size))

    def fp8_scale(self, amax: float) -> float:
        return float(self.lib.oracle_fp8_scale(float(amax)))

    def reshape_and_cache(self, key, value, k_cache, v_cache, slot_mapping, num_kv_heads,
                          head_dim, block_size, num_blocks, kv_dtype, k_scale=1.0, v_scale=1.0):
        """Write key/value (uint16 bf16 bits [T, Hkv, D]) into the uint8 caches in place."""
        key = np.ascontiguousarray(key, dtype=np.uint16)
        value = np.ascontiguousarray(value, dtype=np.uint16)
        slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int32)
        assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
        need = self.cache_bytes(kv_dtype, num_blocks, block_size, num_kv_heads, head_dim)
        assert k_cache.nbytes >= need and v_cache.nbytes >= need
        rc = self.lib.oracle_reshape_and_cache(
            _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
            slot_mapping.size, num_kv_heads, head_dim, block_size, num_blocks, kv_dtype,
            float(k_scale), float(v_scale))
        if rc != 0:
            raise ValueError("oracle_reshape_and_cache: invalid arguments")

    def decode(self, q, k_cache, v_cache, block_tables, seq_lens, num_kv_heads, block_size,
               num_blocks, scale, sliding_window=0, kv_dtype=KV_BF16, k_scale=1.0, v_scale=1.0):
        """Return (out bf16 bits uint16 [B, Hq, D], out before rounding float32 [B, Hq, D])."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, Hq, D = q.shape
        out = np.empty((B, Hq, D), np.uint16)
        out_f32 = np.empty((B, Hq, D), np.float32)
        rc = self.lib.oracle_decode(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(seq_lens),
            _ptr(out), _ptr(out_f32), B, Hq, num_kv_heads, D, block_size, block_tables.shape[1],
            num_blocks, float(scale), int(sliding_window), kv_dtype, float(k_scale),
            float(v_scale))
        if rc != 0:
            raise ValueError("oracle_decode: invalid arguments")
        return out, out_f32


    def decode_e4m3_out(self, q, k_cache, v_cache, block_tables, seq_lens, num_kv_heads,
                        block_size, num_blocks, scale, out_scale, sliding_window=0,
                        kv_dtype=KV_BF16, k_scale=1.0, v_scale=1.0):
        """Decode with E4M3 output: codes uint8 [B, Hq, D] = E4M3(o / out_scale)."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, Hq, D = q.shape
        codes = np.empty((B, Hq, D), np.uint8)
        rc = self.lib.oracle_decode_e4m3_out(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(seq_lens),
            _ptr(codes), B, Hq, num_kv_heads, D, block_size, block_tables.shape[1], num_blocks,
            float(scale), int(sliding_window), kv_dtype, float(k_scale), float(v_scale),
            float(out_scale))
        if rc != 0:
            raise ValueError("oracle_decode_e4m3_out: invalid arguments")
        return codes

    def prefill(self, q, cu_q, k_cache, v_cache, block_tables, seq_lens, num_kv_heads,
                block_size, num_blocks, scale, causal=True, sliding_window=0, kv_dtype=KV_BF16,
                k_scale=1.0, v_scale=1.0):
        """Paged prefill: q uint16 bf16 bits [total_q, Hq, D], cu_q int32 [B+1] query-row
        offsets. Returns (out bf16 bits [total_q, Hq, D], out before rounding float32)."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        cu_q = np.ascontiguousarray(cu_q, dtype=np.int32)
        block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        T, Hq, D = q.shape
        B = seq_lens.shape[0]
        assert cu_q.shape == (B + 1,) and cu_q[-1] == T
        out = np.empty((T, Hq, D), np.uint16)
        out_f32 = np.empty((T, Hq, D), np.float32)
        rc = self.lib.oracle_prefill(
            _ptr(q), _ptr(cu_q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
            _ptr(seq_lens), _ptr(out), _ptr(out_f32), B, Hq, num_kv_heads, D, block_size,
            block_tables.shape[1], num_blocks, float(scale), int(bool(causal)),
            int(sliding_window), kv_dtype, float(k_scale), float(v_scale))
        if rc != 0:
            raise ValueError("oracle_prefill: invalid arguments")
        return out, out_f32


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from pd_oracle.cpp (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default
