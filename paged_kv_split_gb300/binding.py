"""Python binding of libpd.so (include/pd.h): argument marshalling only.

Every function here takes torch tensors on a CUDA device, checks their
dtypes, shapes and devices, and passes raw pointers, sizes and torch's
current CUDA stream to the C entry point of the same name. All compute runs
in libpd.so's kernels; there is no fallback path. Importing this module
raises ImportError when libpd.so has not been built
(``python -m paged_kv_split_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB as _LIB_PATH

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is not built; run `python -m paged_kv_split_gb300.build` "
                      "(or __graft_entry__.build()) on a machine with nvcc")

_lib = ctypes.CDLL(_LIB_PATH)

PD_OK = 0
PD_KV_BF16, PD_KV_FP8_E4M3, PD_KV_NVFP4 = 0, 1, 2
KV_DTYPES = {"bf16": PD_KV_BF16, "fp8": PD_KV_FP8_E4M3, "nvfp4": PD_KV_NVFP4}

_P = ctypes.c_void_p
_i32, _i64, _f32, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

_lib.pd_status_string.argtypes, _lib.pd_status_string.restype = [ctypes.c_int], ctypes.c_char_p
_lib.pd_cache_bytes.argtypes, _lib.pd_cache_bytes.restype = [_i32, _i64, _i32, _i32, _i32], _sz
_lib.pd_page_bytes.argtypes, _lib.pd_page_bytes.restype = [_i32, _i32, _i32, _i32], _sz
_lib.pd_decode_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32]
_lib.pd_decode_workspace_bytes.restype = _sz
_lib.pd_choose_num_splits.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_int]
_lib.pd_choose_num_splits.restype = ctypes.c_int
_lib.pd_plan_num_splits.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32]
_lib.pd_plan_num_splits.restype = ctypes.c_int
_lib.pd_plan_num_splits_for_lengths.argtypes = [_P, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                                _i32, _i32]
_lib.pd_plan_num_splits_for_lengths.restype = ctypes.c_int
_lib.pd_reshape_and_cache.argtypes = [_P, _P, _P, _P, _P, _i32, _i32, _i32, _i32, _i64, _i32,
                                      _f32, _f32, _P]
_lib.pd_reshape_and_cache.restype = ctypes.c_int
_lib.pd_absmax_bf16.argtypes, _lib.pd_absmax_bf16.restype = [_P, _i64, _P, _P], ctypes.c_int
_lib.pd_fp8_scale.argtypes, _lib.pd_fp8_scale.restype = [_f32], _f32
_lib.pd_fp8_scales_from_absmax.argtypes = [_P, _P, _i32, _P]
_lib.pd_fp8_scales_from_absmax.restype = ctypes.c_int
_lib.pd_test_encode.argtypes, _lib.pd_test_encode.restype = [_i32, ctypes.c_uint32, _i64, _P,
                                                              _P], ctypes.c_int
_lib.pd_test_set_consumer_wait_ns.argtypes = [ctypes.c_uint32]
_lib.pd_test_set_consumer_wait_ns.restype = ctypes.c_uint32
_DECODE_ARGS = [_P, _P, _P, _P, _P, _P, _i32, _i32, _i32, _i32, _i32, _i32, _i64, _f32, _i32,
                _i32, _i32, _f32, _f32, _P, _sz, _P]
_lib.pd_decode.argtypes, _lib.pd_decode.restype = _DECODE_ARGS, ctypes.c_int
_lib.pd_decode_crosscheck.argtypes = _DECODE_ARGS
_lib.pd_decode_crosscheck.restype = ctypes.c_int
_lib.pd_decode_e4m3_out.argtypes = _DECODE_ARGS[:19] + [_f32] + _DECODE_ARGS[19:]
_lib.pd_decode_e4m3_out.restype = ctypes.c_int
_lib.pd_decode_strided.argtypes = [_P, _i64] + _DECODE_ARGS[1:6] + [_i64] + _DECODE_ARGS[6:]
_lib.pd_decode_strided.restype = ctypes.c_int
_lib.pd_decode_partial.argtypes = [_P, _P, _P, _P, _P, _i32, _i32, _i32, _i32, _i32, _i32, _i64,
                                   _f32, _i32, _i32, _i32, _f32, _f32, _P, _sz, _P]
_lib.pd_decode_partial.restype = ctypes.c_int
_lib.pd_decode_combine.argtypes = [_P, _sz, _P, _P, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _P]
_lib.pd_decode_combine.restype = ctypes.c_int
_lib.pd_device_status.argtypes, _lib.pd_device_status.restype = [_P, _i32], ctypes.c_int
_lib.pd_prefill.argtypes = [_P, _i64, _P, _P, _P, _P, _P, _P, _i64, _i32, _i32, _i32, _i32, _i32,
                            _i32, _i32, _i64, _f32, _i32, _i32, _i32, _f32, _f32, _P]
_lib.pd_prefill.restype = ctypes.c_int
_lib.pd_prefill_crosscheck.argtypes = _lib.pd_prefill.argtypes
_lib.pd_prefill_crosscheck.restype = ctypes.c_int
_lib.pd_prefer_balanced.argtypes = [_P, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32]
_lib.pd_prefer_balanced.restype = ctypes.c_int
_lib.pd_balanced_plan_bytes.argtypes = [_i32, _i32, _i32]
_lib.pd_balanced_plan_bytes.restype = _sz
_lib.pd_balanced_plan.argtypes = [_P, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _P,
                                  _sz, _P, _P, _P]
_lib.pd_balanced_plan.restype = ctypes.c_int
_lib.pd_decode_balanced.argtypes = [_P, _P, _P, _P, _P, _sz, _P, _i32, _i32, _i32, _i32, _i32,
                                    _i32, _i64, _f32, _i32, _i32, _f32, _f32, _i32, _i32, _P,
                                    _sz, _P]
_lib.pd_decode_balanced.restype = ctypes.c_int
_lib.pd_decode_balanced_strided.argtypes = ([_P, _i64] + _lib.pd_decode_balanced.argtypes[1:7] +
                                            [_i64] + _lib.pd_decode_balanced.argtypes[7:])
_lib.pd_decode_balanced_strided.restype = ctypes.c_int
for _fn in ("pd_decode_balanced_partial", "pd_decode_balanced_combine"):
    getattr(_lib, _fn).argtypes = _lib.pd_decode_balanced.argtypes
    getattr(_lib, _fn).restype = ctypes.c_int


class PdError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {pd_status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded libpd.so handle (for callers that want the raw C entry points)."""
    return _lib


def pd_status_string(status: int) -> str:
    return _lib.pd_status_string(int(status)).decode()


def _check(fn: str, rc: int) -> None:
    if rc != PD_OK:
        raise PdError(fn, rc)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(getattr(stream, "cuda_stream", stream) or 0)


def _dev(t: torch.Tensor, name: str, dtype=None, device=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t.data_ptr()


def _dtype_code(kv_dtype) -> int:
    return KV_DTYPES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)


# ---- sizes ----------------------------------------------------------------
def pd_cache_bytes(kv_dtype, num_blocks, block_size, num_kv_heads, head_dim) -> int:
    return int(_lib.pd_cache_bytes(_dtype_code(kv_dtype), num_blocks, block_size, num_kv_heads,
                                   head_dim))


def pd_page_bytes(kv_dtype, block_size, num_kv_heads, head_dim) -> int:
    return int(_lib.pd_page_bytes(_dtype_code(kv_dtype), block_size, num_kv_heads, head_dim))


def pd_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, num_splits) -> int:
    return int(_lib.pd_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, num_splits))


def pd_plan_num_splits(num_seqs, num_kv_heads, max_blocks_per_seq, block_size, sliding_window,
                       head_dim, kv_dtype, num_sms) -> int:
    s = _lib.pd_plan_num_splits(num_seqs, num_kv_heads, max_blocks_per_seq, block_size,
                                sliding_window, head_dim, _dtype_code(kv_dtype), num_sms)
    if s < 1:
        raise PdError("pd_plan_num_splits", -s)
    return s


def pd_plan_num_splits_for_lengths(seq_lens, num_q_heads, num_kv_heads, max_blocks_per_seq,
                                   block_size, sliding_window, head_dim, kv_dtype, num_sms) -> int:
    """Split count for host-known sequence lengths (an int sequence or array)."""
    import numpy as np
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    s = _lib.pd_plan_num_splits_for_lengths(lens.ctypes.data, lens.size, num_q_heads,
                                            num_kv_heads, max_blocks_per_seq, block_size,
                                            sliding_window, head_dim, _dtype_code(kv_dtype),
                                            num_sms)
    if s < 1:
        raise PdError("pd_plan_num_splits_for_lengths", -s)
    return s


def pd_choose_num_splits(num_seqs, num_kv_heads, max_blocks_per_seq, block_size, sliding_window,
                         head_dim, kv_dtype, device=None) -> int:
    dev = torch.cuda.current_device() if device is None else int(device)
    s = _lib.pd_choose_num_splits(num_seqs, num_kv_heads, max_blocks_per_seq, block_size,
                                  sliding_window, head_dim, _dtype_code(kv_dtype), dev)
    if s < 1:
        raise PdError("pd_choose_num_splits", -s)
    return s


def empty_cache(kv_dtype, num_blocks, block_size, num_kv_heads, head_dim, device="cuda"):
    """One K (or V) cache as a flat uint8 tensor of pd_cache_bytes bytes."""
    n = pd_cache_bytes(kv_dtype, num_blocks, block_size, num_kv_heads, head_dim)
    if n == 0:
        raise ValueError("unsupported cache shape")
    return torch.empty(n, dtype=torch.uint8, device=device)


# ---- operations -----------------------------------------------------------
def pd_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, *, num_blocks, block_size,
                         kv_dtype=PD_KV_BF16, k_scale=1.0, v_scale=1.0, stream=None) -> None:
    """Write key/value (bf16 [T, Hkv, D]) into the caches at slot_mapping (int32 [T])."""
    T, hkv, d = key.shape
    dev = key.device
    if value.shape != key.shape:
        raise ValueError("key and value shapes differ")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    rc = _lib.pd_reshape_and_cache(
        _dev(key, "key", torch.bfloat16, dev), _dev(value, "value", torch.bfloat16, dev),
        _dev(k_cache, "k_cache", None, dev), _dev(v_cache, "v_cache", None, dev),
        _dev(slot_mapping, "slot_mapping", torch.int32, dev), T, hkv, d, block_size, num_blocks,
        _dtype_code(kv_dtype), float(k_scale), float(v_scale), _stream(stream))
    _check("pd_reshape_and_cache", rc)


def pd_absmax_bf16(data, out_max, stream=None) -> None:
    """Fold max |data| into out_max (float32 [1], caller-zeroed)."""
    rc = _lib.pd_absmax_bf16(_dev(data, "data", torch.bfloat16), data.numel(),
                             _dev(out_max, "out_max", torch.float32), _stream(stream))
    _check("pd_absmax_bf16", rc)


def pd_fp8_scale(absmax: float) -> float:
    """FP8 scale of a tensor from its absmax (libpd.so's pd_fp8_scale)."""
    return float(_lib.pd_fp8_scale(float(absmax)))


def pd_fp8_scales_from_absmax(absmax, scales, stream=None) -> None:
    """scales[i] = pd_fp8_scale(absmax[i]) on the device (float32 tensors)."""
    if absmax.shape != scales.shape:
        raise ValueError("absmax and scales must have the same shape")
    rc = _lib.pd_fp8_scales_from_absmax(_dev(absmax, "absmax", torch.float32),
                                        _dev(scales, "scales", torch.float32, absmax.device),
                                        absmax.numel(), _stream(stream))
    _check("pd_fp8_scales_from_absmax", rc)


def fp8_calibrate(key, value, stream=None):
    """Per-tensor FP8 scales for key and value: pd_absmax_bf16 of each, then
    pd_fp8_scales_from_absmax, both on the device; the two scales are read
    back once (a synchronising copy: calibration is a one-off step, not part
    of decode)."""
    amax = torch.zeros(2, dtype=torch.float32, device=key.device)
    pd_absmax_bf16(key, amax[0:1], stream)
    pd_absmax_bf16(value, amax[1:2], stream)
    scales = torch.empty_like(amax)
    pd_fp8_scales_from_absmax(amax, scales, stream)
    ks, vs = scales.cpu().tolist()
    return ks, vs


def pd_test_encode(fmt: int, first_bits: int, codes, stream=None) -> None:
    """Test hook: codes[i] = the device encoder's code (0 = E4M3, 1 = E2M1) of
    the fp32 bit pattern first_bits + i (codes: CUDA uint8 tensor)."""
    rc = _lib.pd_test_encode(int(fmt), int(first_bits) & 0xFFFFFFFF, codes.numel(),
                             _dev(codes, "codes", torch.uint8), _stream(stream))
    _check("pd_test_encode", rc)


def pd_test_set_consumer_wait_ns(ns: int) -> int:
    """Test hook: the decode kernels' consumer wait limit (0xFFFFFFFF = default).
    Returns the previous limit."""
    return int(_lib.pd_test_set_consumer_wait_ns(int(ns) & 0xFFFFFFFF))


def _decode_shape(q, block_tables, seq_lens, out=None):
    B, hq, d = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
    if seq_lens.shape != (B,):
        raise ValueError("seq_lens must be [num_seqs]")
    if out is not None and out.shape != q.shape:
        raise ValueError("out must have q's shape")
    return B, hq, d, block_tables.shape[1]


def pd_decode(q, k_cache, v_cache, block_tables, seq_lens, out, *, num_kv_heads, block_size,
              num_blocks, scale, num_splits=0, sliding_window=0, kv_dtype=PD_KV_BF16,
              k_scale=1.0, v_scale=1.0, workspace=None, stream=None, crosscheck=False):
    """One decode step (split-KV partials + combine) into out (bf16 [B, Hq, D]).

    workspace: a CUDA uint8 tensor of at least pd_decode_workspace_bytes for
    the split count used; when None, one is allocated here with torch.
    crosscheck: call pd_decode_crosscheck (the CUDA-core partial kernel)."""
    B, hq, d, mbs = _decode_shape(q, block_tables, seq_lens, out)
    code = _dtype_code(kv_dtype)
    S = num_splits
    if workspace is None:
        if S == 0:
            S = pd_choose_num_splits(B, num_kv_heads, mbs, block_size, sliding_window, d, code,
                                     q.device.index)
        workspace = torch.empty(max(pd_decode_workspace_bytes(B, hq, d, S), 16), dtype=torch.uint8,
                                device=q.device)
    dev = q.device
    fn = "pd_decode_crosscheck" if crosscheck else "pd_decode"
    rc = getattr(_lib, fn)(
        _dev(q, "q", torch.bfloat16, dev), _dev(k_cache, "k_cache", None, dev),
        _dev(v_cache, "v_cache", None, dev), _dev(block_tables, "block_tables", torch.int32, dev),
        _dev(seq_lens, "seq_lens", torch.int32, dev), _dev(out, "out", torch.bfloat16, dev), B,
        hq, num_kv_heads, d, block_size, mbs, num_blocks, float(scale), S, sliding_window, code,
        float(k_scale), float(v_scale), _dev(workspace, "workspace", None, dev),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(fn, rc)
    return out


def pd_decode_e4m3_out(q, k_cache, v_cache, block_tables, seq_lens, out, *, out_scale,
                       num_kv_heads, block_size, num_blocks, scale, num_splits=0,
                       sliding_window=0, kv_dtype=PD_KV_BF16, k_scale=1.0, v_scale=1.0,
                       workspace=None, stream=None):
    """One decode step writing E4M3 codes E4M3(o / out_scale) into out
    (uint8 [B, Hq, D]); otherwise as pd_decode."""
    B, hq, d, mbs = _decode_shape(q, block_tables, seq_lens)
    if tuple(out.shape) != (B, hq, d):
        raise ValueError("out must be uint8 [num_seqs, num_q_heads, head_dim]")
    code = _dtype_code(kv_dtype)
    S = num_splits
    if workspace is None:
        if S == 0:
            S = pd_choose_num_splits(B, num_kv_heads, mbs, block_size, sliding_window, d, code,
                                     q.device.index)
        workspace = torch.empty(max(pd_decode_workspace_bytes(B, hq, d, S), 16), dtype=torch.uint8,
                                device=q.device)
    dev = q.device
    rc = _lib.pd_decode_e4m3_out(
        _dev(q, "q", torch.bfloat16, dev), _dev(k_cache, "k_cache", None, dev),
        _dev(v_cache, "v_cache", None, dev), _dev(block_tables, "block_tables", torch.int32, dev),
        _dev(seq_lens, "seq_lens", torch.int32, dev), _dev(out, "out", torch.uint8, dev), B,
        hq, num_kv_heads, d, block_size, mbs, num_blocks, float(scale), S, sliding_window, code,
        float(k_scale), float(v_scale), float(out_scale), _dev(workspace, "workspace", None, dev),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check("pd_decode_e4m3_out", rc)
    return out


def pd_decode_partial(q, k_cache, v_cache, block_tables, seq_lens, workspace, *, num_kv_heads,
                      block_size, num_blocks, scale, num_splits, sliding_window=0,
                      kv_dtype=PD_KV_BF16, k_scale=1.0, v_scale=1.0, stream=None):
    B, hq, d, mbs = _decode_shape(q, block_tables, seq_lens)
    dev = q.device
    rc = _lib.pd_decode_partial(
        _dev(q, "q", torch.bfloat16, dev), _dev(k_cache, "k_cache", None, dev),
        _dev(v_cache, "v_cache", None, dev), _dev(block_tables, "block_tables", torch.int32, dev),
        _dev(seq_lens, "seq_lens", torch.int32, dev), B, hq, num_kv_heads, d, block_size, mbs,
        num_blocks, float(scale), num_splits, sliding_window, _dtype_code(kv_dtype),
        float(k_scale), float(v_scale), _dev(workspace, "workspace", None, dev),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check("pd_decode_partial", rc)


def pd_decode_combine(workspace, seq_lens, out, *, block_size, max_blocks_per_seq, num_splits,
                      sliding_window=0, stream=None):
    B, hq, d = out.shape
    dev = out.device
    rc = _lib.pd_decode_combine(
        _dev(workspace, "workspace", None, dev), workspace.numel() * workspace.element_size(),
        _dev(seq_lens, "seq_lens", torch.int32, dev), _dev(out, "out", torch.bfloat16, dev), B, hq,
        d, block_size, max_blocks_per_seq, num_splits, sliding_window, _stream(stream))
    _check("pd_decode_combine", rc)


def pd_device_status(reset: bool = False) -> int:
    """pd_device_flag bits raised by kernels on the current device (synchronises)."""
    v = ctypes.c_int32(0)
    _check("pd_device_status", _lib.pd_device_status(ctypes.addressof(v), int(bool(reset))))
    return int(v.value)


# ---- balanced decode -------------------------------------------------------
class BalancedPlan:
    """A host plan from pd_balanced_plan: `host` (CPU int32 tensor whose bytes
    are the device plan), `num_ctas`, `num_pieces`, `workspace_bytes`."""

    def __init__(self, host, num_ctas, num_pieces, workspace_bytes):
        self.host = host
        self.num_ctas = num_ctas
        self.num_pieces = num_pieces
        self.workspace_bytes = workspace_bytes

    @property
    def words(self):
        """The plan as a numpy int32 array (a view of `host`)."""
        return self.host.numpy()

    def to(self, device):
        """The plan as a device int32 tensor (what pd_decode_balanced reads)."""
        return self.host.to(device)


def balanced_plan_buffer(num_seqs, num_kv_heads, num_sms, pin=False):
    """A host int32 buffer large enough for any plan of these shapes."""
    nbytes = int(_lib.pd_balanced_plan_bytes(num_seqs, num_kv_heads, num_sms))
    if nbytes == 0:
        raise ValueError("bad plan shape")
    buf = torch.zeros((nbytes + 15) // 16 * 4, dtype=torch.int32)
    return buf.pin_memory() if pin else buf


def pd_balanced_plan(seq_lens_host, *, num_q_heads, num_kv_heads, head_dim, block_size,
                     max_blocks_per_seq, sliding_window=0, kv_dtype=PD_KV_BF16, num_sms,
                     out=None):
    """Build a balanced plan on the host from host lengths (int32 [B], numpy or
    CPU tensor). `out`: a buffer from balanced_plan_buffer to plan into (it is
    reused, so a scheduler can plan every step without allocating)."""
    import numpy as np
    lens = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
    B = int(lens.shape[0])
    if out is None:
        out = balanced_plan_buffer(B, num_kv_heads, num_sms)
    nc, npc, wsb = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_size_t(0)
    rc = _lib.pd_balanced_plan(lens.ctypes.data if B else None, B, num_q_heads, num_kv_heads,
                               head_dim, block_size, max_blocks_per_seq, sliding_window,
                               _dtype_code(kv_dtype), num_sms, out.data_ptr(),
                               out.numel() * 4, ctypes.byref(nc), ctypes.byref(npc),
                               ctypes.byref(wsb))
    _check("pd_balanced_plan", rc)
    return BalancedPlan(out, nc.value, npc.value, wsb.value)


def pd_decode_balanced(q, k_cache, v_cache, block_tables, plan_dev, plan, out, *, num_kv_heads,
                       block_size, num_blocks, scale, sliding_window=0, kv_dtype=PD_KV_BF16,
                       k_scale=1.0, v_scale=1.0, workspace=None, stream=None, _fn="pd_decode_balanced"):
    """One balanced decode step into out; plan_dev is plan.to(device)."""
    B, hq, d = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    mbs = block_tables.shape[1]
    dev = q.device
    if workspace is None:
        workspace = torch.empty(max(plan.workspace_bytes, 16), dtype=torch.uint8, device=dev)
    rc = getattr(_lib, _fn)(
        _dev(q, "q", torch.bfloat16, dev), _dev(k_cache, "k_cache", None, dev),
        _dev(v_cache, "v_cache", None, dev), _dev(block_tables, "block_tables", torch.int32, dev),
        _dev(plan_dev, "plan", torch.int32, dev), plan_dev.numel() * 4,
        _dev(out, "out", torch.bfloat16, dev), B, hq, num_kv_heads, d, block_size, mbs,
        num_blocks, float(scale), sliding_window, _dtype_code(kv_dtype), float(k_scale),
        float(v_scale), plan.num_ctas, plan.num_pieces, _dev(workspace, "workspace", None, dev),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(_fn, rc)
    return out


def pd_decode_balanced_partial(*args, **kw):
    """The partial kernel of pd_decode_balanced alone (same arguments)."""
    return pd_decode_balanced(*args, _fn="pd_decode_balanced_partial", **kw)


def pd_decode_balanced_combine(*args, **kw):
    """The combine kernel of pd_decode_balanced alone (same arguments)."""
    return pd_decode_balanced(*args, _fn="pd_decode_balanced_combine", **kw)


def pd_prefer_balanced(seq_lens_host, *, num_q_heads, num_kv_heads, max_blocks_per_seq,
                       block_size, head_dim, sliding_window=0, kv_dtype=PD_KV_BF16, num_sms):
    """True if the balanced schedule is expected faster for these host lengths."""
    import numpy as np
    lens = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
    r = _lib.pd_prefer_balanced(lens.ctypes.data if lens.size else None, int(lens.shape[0]),
                                num_q_heads, num_kv_heads, max_blocks_per_seq, block_size,
                                sliding_window, head_dim, _dtype_code(kv_dtype), num_sms)
    if r < 0:
        raise PdError("pd_prefer_balanced", -r)
    return bool(r)


# ---- strided q (fused QKV buffers) -----------------------------------------
def _strided_rows(rows, num_q_heads, head_dim, name):
    """rows: bf16 [B, row] (contiguous), the heads in the first Hq * D of a row."""
    if rows.dim() != 2 or rows.dtype != torch.bfloat16 or not rows.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bf16 [num_seqs, row] tensor")
    if rows.shape[1] < num_q_heads * head_dim:
        raise ValueError(f"a {name} row is shorter than num_q_heads * head_dim")
    return int(rows.shape[0]), int(rows.shape[1])


def _strided_q(q_rows, num_q_heads, head_dim):
    return _strided_rows(q_rows, num_q_heads, head_dim, "q_rows")


def pd_decode_strided(q_rows, k_cache, v_cache, block_tables, seq_lens, out_rows, *,
                      num_q_heads, head_dim, num_kv_heads, block_size, num_blocks, scale,
                      num_splits=0, sliding_window=0, kv_dtype=PD_KV_BF16, k_scale=1.0,
                      v_scale=1.0, workspace=None, stream=None):
    """pd_decode with sequence b's q heads at q_rows[b, :Hq * D] and its output
    heads written to out_rows[b, :Hq * D] (both bf16 [B, row] tensors)."""
    B, stride = _strided_q(q_rows, num_q_heads, head_dim)
    Bo, ostride = _strided_rows(out_rows, num_q_heads, head_dim, "out_rows")
    if Bo != B:
        raise ValueError("q_rows and out_rows have different numbers of sequences")
    mbs = block_tables.shape[1]
    code = _dtype_code(kv_dtype)
    S = num_splits
    dev = q_rows.device
    if workspace is None:
        if S == 0:
            S = pd_choose_num_splits(B, num_kv_heads, mbs, block_size, sliding_window, head_dim,
                                     code, dev.index)
        workspace = torch.empty(max(pd_decode_workspace_bytes(B, num_q_heads, head_dim, S), 16),
                                dtype=torch.uint8, device=dev)
    rc = _lib.pd_decode_strided(
        _dev(q_rows, "q_rows", torch.bfloat16, dev), stride,
        _dev(k_cache, "k_cache", None, dev), _dev(v_cache, "v_cache", None, dev),
        _dev(block_tables, "block_tables", torch.int32, dev),
        _dev(seq_lens, "seq_lens", torch.int32, dev),
        _dev(out_rows, "out_rows", torch.bfloat16, dev), ostride, B,
        num_q_heads, num_kv_heads, head_dim, block_size, mbs, num_blocks, float(scale), S,
        sliding_window, code, float(k_scale), float(v_scale),
        _dev(workspace, "workspace", None, dev), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check("pd_decode_strided", rc)
    return out_rows


def pd_decode_balanced_strided(q_rows, k_cache, v_cache, block_tables, plan_dev, plan,
                               out_rows, *, num_q_heads, head_dim, num_kv_heads, block_size,
                               num_blocks, scale, sliding_window=0, kv_dtype=PD_KV_BF16,
                               k_scale=1.0, v_scale=1.0, workspace=None, stream=None):
    """pd_decode_balanced with strided q rows and output rows (as pd_decode_strided)."""
    B, stride = _strided_q(q_rows, num_q_heads, head_dim)
    Bo, ostride = _strided_rows(out_rows, num_q_heads, head_dim, "out_rows")
    if Bo != B:
        raise ValueError("q_rows and out_rows have different numbers of sequences")
    dev = q_rows.device
    if workspace is None:
        workspace = torch.empty(max(plan.workspace_bytes, 16), dtype=torch.uint8, device=dev)
    rc = _lib.pd_decode_balanced_strided(
        _dev(q_rows, "q_rows", torch.bfloat16, dev), stride,
        _dev(k_cache, "k_cache", None, dev), _dev(v_cache, "v_cache", None, dev),
        _dev(block_tables, "block_tables", torch.int32, dev),
        _dev(plan_dev, "plan", torch.int32, dev), plan_dev.numel() * 4,
        _dev(out_rows, "out_rows", torch.bfloat16, dev), ostride, B, num_q_heads, num_kv_heads,
        head_dim,
        block_size, block_tables.shape[1], num_blocks, float(scale), sliding_window,
        _dtype_code(kv_dtype), float(k_scale), float(v_scale), plan.num_ctas, plan.num_pieces,
        _dev(workspace, "workspace", None, dev), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check("pd_decode_balanced_strided", rc)
    return out_rows


# ---- paged prefill ---------------------------------------------------------
def pd_prefill(q, cu_q, k_cache, v_cache, block_tables, seq_lens, out, *, max_q_len,
               num_kv_heads, block_size, num_blocks, scale, causal=True, sliding_window=0,
               kv_dtype=PD_KV_BF16, k_scale=1.0, v_scale=1.0, stream=None, crosscheck=False):
    """Paged (chunked) prefill. q and out: contiguous bf16 [total_q, Hq, D];
    cu_q: int32 [B + 1] query-row offsets; seq_lens: int32 [B] keys in the
    cache (new tokens included); max_q_len: host int, the largest q length.
    pd_prefill_strided takes token rows of a wider buffer instead.
    crosscheck: call pd_prefill_crosscheck (the mma.sync kernel)."""
    if q.dim() != 3 or out.dim() != 3:
        raise ValueError("q and out must be bf16 [total_q, num_q_heads, head_dim]")
    T, hq, d = q.shape
    if tuple(out.shape) != (T, hq, d):
        raise ValueError("out must have q's shape")
    B = int(seq_lens.shape[0])
    if tuple(cu_q.shape) != (B + 1,):
        raise ValueError("cu_q must be int32 [num_seqs + 1]")
    dev = q.device
    fn = "pd_prefill_crosscheck" if crosscheck else "pd_prefill"
    rc = getattr(_lib, fn)(
        _dev(q, "q", torch.bfloat16, dev), 0, _dev(cu_q, "cu_q", torch.int32, dev),
        _dev(k_cache, "k_cache", None, dev), _dev(v_cache, "v_cache", None, dev),
        _dev(block_tables, "block_tables", torch.int32, dev),
        _dev(seq_lens, "seq_lens", torch.int32, dev), _dev(out, "out", torch.bfloat16, dev), 0,
        B, int(max_q_len), hq, num_kv_heads, d, block_size, block_tables.shape[1], num_blocks,
        float(scale), int(bool(causal)), int(sliding_window), _dtype_code(kv_dtype),
        float(k_scale), float(v_scale), _stream(stream))
    _check(fn, rc)
    return out


def pd_prefill_strided(q_rows, cu_q, k_cache, v_cache, block_tables, seq_lens, out_rows, *,
                       num_q_heads, head_dim, max_q_len, num_kv_heads, block_size, num_blocks,
                       scale, causal=True, sliding_window=0, kv_dtype=PD_KV_BF16, k_scale=1.0,
                       v_scale=1.0, stream=None, crosscheck=False):
    """pd_prefill with token rows of a wider buffer: q_rows / out_rows are
    contiguous bf16 [total_q, row] tensors holding each token's Hq * D
    values in the first Hq * D of its row (fused QKV rows, padded outputs)."""
    T, stride = _strided_rows(q_rows, num_q_heads, head_dim, "q_rows")
    To, ostride = _strided_rows(out_rows, num_q_heads, head_dim, "out_rows")
    if To != T:
        raise ValueError("q_rows and out_rows have different numbers of rows")
    B = int(seq_lens.shape[0])
    dev = q_rows.device
    fn = "pd_prefill_crosscheck" if crosscheck else "pd_prefill"
    rc = getattr(_lib, fn)(
        _dev(q_rows, "q_rows", torch.bfloat16, dev), stride, _dev(cu_q, "cu_q", torch.int32, dev),
        _dev(k_cache, "k_cache", None, dev), _dev(v_cache, "v_cache", None, dev),
        _dev(block_tables, "block_tables", torch.int32, dev),
        _dev(seq_lens, "seq_lens", torch.int32, dev),
        _dev(out_rows, "out_rows", torch.bfloat16, dev), ostride, B, int(max_q_len),
        num_q_heads, num_kv_heads, head_dim, block_size, block_tables.shape[1], num_blocks,
        float(scale), int(bool(causal)), int(sliding_window), _dtype_code(kv_dtype),
        float(k_scale), float(v_scale), _stream(stream))
    _check(fn, rc)
    return out_rows
