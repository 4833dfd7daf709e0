"""libpd.so loads and exports exactly the entry points include/pd.h declares,
and its host-only logic (sizes, split planning, argument validation) behaves
as documented. CPU only: nothing here launches a kernel."""
import ctypes
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "pd.h")


@pytest.fixture(scope="module")
def pdlib():
    from paged_kv_split_gb300 import build
    path = build.build()
    L = ctypes.CDLL(path)
    return path, L


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pd_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pd_reshape_and_cache", "pd_decode", "pd_decode_partial",
                     "pd_decode_combine", "pd_absmax_bf16", "pd_decode_workspace_bytes",
                     "pd_cache_bytes", "pd_choose_num_splits", "pd_status_string"):
        assert required in names


def test_exports_match_header(pdlib):
    path, _ = pdlib
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = sorted({m.group(1) for m in re.finditer(r"\sT\s+(pd_[a-z0-9_]+)$", out, re.M)})
    assert exported == declared_functions()


def test_cache_and_workspace_sizes(pdlib):
    _, L = pdlib
    L.pd_cache_bytes.restype = ctypes.c_size_t
    L.pd_cache_bytes.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.c_int32]
    L.pd_decode_workspace_bytes.restype = ctypes.c_size_t
    L.pd_decode_workspace_bytes.argtypes = [ctypes.c_int32] * 4
    import oracle
    orc = oracle.get()
    for dt in (0, 1, 2):
        for bs in (16, 32):
            for h, d in ((2, 64), (8, 128), (4, 256), (2, 512), (1, 64)):
                assert L.pd_cache_bytes(dt, 37, bs, h, d) == orc.cache_bytes(dt, 37, bs, h, d)
    assert L.pd_cache_bytes(9, 1, 16, 1, 64) == 0
    ws = L.pd_decode_workspace_bytes(32, 32, 128, 8)
    assert ws >= 32 * 32 * 8 * (128 + 2) * 4


def test_split_planner(pdlib):
    _, L = pdlib
    L.pd_plan_num_splits.argtypes = [ctypes.c_int32] * 8
    plan = L.pd_plan_num_splits
    # (num_seqs, kv heads, max pages, block size, window, head_dim, dtype, SMs):
    # about one wave of resident CTAs at the maximum length
    one = plan(4, 8, 1024, 32, 0, 128, 0, 152)
    assert 8 <= one <= 32
    assert plan(1, 8, 1024, 32, 0, 128, 0, 152) > one          # fewer units, more splits
    assert plan(64, 8, 1024, 32, 0, 128, 0, 152) == 1          # enough units already
    assert plan(1, 1, 1, 16, 0, 128, 0, 152) == 1               # one page, one split
    assert plan(1, 4, 1024, 16, 64, 128, 0, 152) <= 5           # a window bounds the pages
    assert plan(1, 8, 10, 16, 0, 128, 0, 0) < 0
    assert plan(1, 8, 10, 16, 0, 128, 7, 152) < 0


def test_split_planner_for_lengths(pdlib):
    import numpy as np
    _, L = pdlib
    f = L.pd_plan_num_splits_for_lengths
    f.argtypes = [ctypes.c_void_p] + [ctypes.c_int32] * 9
    lens = np.full(4, 32768, np.int32)
    S = f(lens.ctypes.data, 4, 32, 8, 1024, 32, 0, 128, 0, 152)
    # uniform long sequences: fill one wave of CTAs without a second, partial one
    assert S * 4 * 8 <= 152 * 4 and S >= 8
    # one long sequence among short ones is cut so that its pieces are no
    # longer than about a wave's share of the whole batch's pages
    mixed = np.array([32768] + [512] * 31, np.int32)
    s_mixed = f(mixed.ctypes.data, 32, 32, 8, 1024, 32, 0, 128, 0, 152)
    chunk = -(-1024 // s_mixed)
    total_pages = (1024 + 31 * 16) * 8
    assert chunk * 8 <= 2 * total_pages / (152 * 3) * 8 + 16
    assert f(lens.ctypes.data, 4, 30, 8, 1024, 32, 0, 128, 0, 152) < 0   # 30 % 8 != 0
    assert f(None, 0, 32, 8, 1024, 32, 0, 128, 0, 152) == 1


def test_status_strings(pdlib):
    _, L = pdlib
    L.pd_status_string.restype = ctypes.c_char_p
    assert L.pd_status_string(0) == b"PD_OK"
    for s in (1, 2, 3, 4):
        assert L.pd_status_string(s).startswith(b"PD_ERR_")
    assert L.pd_status_string(77) == b"unknown pd status"


def _decode_partial(L, **kw):
    args = dict(q=0x1000, k=0x2000, v=0x3000, bt=0x4000, lens=0x5000, B=2, Hq=8, Hkv=2, D=128,
                bs=16, mbs=4, nb=8, scale=0.1, S=2, W=0, dt=0, ks=1.0, vs=1.0, ws=0x6000,
                ws_bytes=1 << 20)
    args.update(kw)
    f = L.pd_decode_partial
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    f.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, f32, i32, i32, i32, f32, f32, P,
                  ctypes.c_size_t, P]
    a = args
    return f(a["q"], a["k"], a["v"], a["bt"], a["lens"], a["B"], a["Hq"], a["Hkv"], a["D"],
             a["bs"], a["mbs"], a["nb"], a["scale"], a["S"], a["W"], a["dt"], a["ks"], a["vs"],
             a["ws"], a["ws_bytes"], None)


def test_validation_rejects_before_any_launch(pdlib):
    """Every case below is refused on the host (the pointers are never touched)."""
    _, L = pdlib
    assert _decode_partial(L, Hq=6, Hkv=4) == 1            # GQA ratio not integral
    assert _decode_partial(L, Hq=34, Hkv=2) == 2           # group of 17 > 16
    assert _decode_partial(L, D=96) == 2                   # head_dim not built
    assert _decode_partial(L, bs=8) == 2                   # block size not built
    assert _decode_partial(L, dt=5) == 2                   # unknown cache form
    assert _decode_partial(L, S=0) == 1                    # partial needs S >= 1
    assert _decode_partial(L, S=2000) == 1                 # too many splits
    assert _decode_partial(L, W=-1) == 1                   # negative window
    assert _decode_partial(L, q=0x1004) == 1               # misaligned pointer
    assert _decode_partial(L, k=0) == 1                    # null pointer
    assert _decode_partial(L, dt=1, ks=0.0) == 1           # FP8 needs a positive scale
    assert _decode_partial(L, dt=1, vs=float("nan")) == 1
    assert _decode_partial(L, ws_bytes=100) == 3           # workspace too small


def test_reshape_and_cache_validation(pdlib):
    _, L = pdlib
    f = L.pd_reshape_and_cache
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    f.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64, i32, f32, f32, P]
    ok = dict(k=0x1000, v=0x2000, kc=0x3000, vc=0x4000, sl=0x5000, T=4, H=2, D=64, bs=16, nb=4,
              dt=0, ks=1.0, vs=1.0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["k"], a["v"], a["kc"], a["vc"], a["sl"], a["T"], a["H"], a["D"], a["bs"],
                 a["nb"], a["dt"], a["ks"], a["vs"], None)
    assert call(T=0) == 0                                   # nothing to do, no launch
    assert call(D=48) == 2
    assert call(bs=64) == 2
    assert call(T=-1) == 1
    assert call(kc=0x3001) == 1
    assert call(dt=1, ks=-1.0) == 1
    assert call(nb=0) == 1


def test_prefill_validation(pdlib):
    """pd_prefill refuses bad shapes on the host; the pointers are never touched
    (every call here must fail a check: a valid one would launch on them)."""
    _, L = pdlib
    f = L.pd_prefill
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    f.argtypes = [P, i64, P, P, P, P, P, P, i64, i32, i32, i32, i32, i32, i32, i32, i64, f32,
                  i32, i32, i32, f32, f32, P]
    ok = dict(q=0x1000, qs=0, cu=0x2000, kc=0x3000, vc=0x4000, bt=0x5000, sl=0x6000, o=0x7000,
              os=0, B=2, mq=16, Hq=8, Hkv=2, D=128, bs=16, mbs=8, nb=32, sc=0.088, causal=1, W=0,
              dt=0, ks=1.0, vs=1.0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["qs"], a["cu"], a["kc"], a["vc"], a["bt"], a["sl"], a["o"], a["os"],
                 a["B"], a["mq"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["mbs"], a["nb"], a["sc"],
                 a["causal"], a["W"], a["dt"], a["ks"], a["vs"], None)
    assert call(B=0) == 0                 # nothing to do, no launch
    assert call(mq=0) == 0
    assert call(dt=7) == 2                # unknown cache form
    assert call(dt=1, ks=0.0) == 1        # FP8 cache: scales must be positive and finite
    assert call(dt=1, vs=float("nan")) == 1
    assert call(D=512) == 2               # head_dim 512: not built for prefill
    assert call(D=96) == 2
    assert call(bs=8) == 2
    assert call(Hq=34, Hkv=2) == 2        # group of 17 > 16
    assert call(Hq=6, Hkv=4) == 1         # GQA ratio not integral
    assert call(mq=-1) == 1
    assert call(W=-1) == 1
    assert call(qs=100) == 1              # stride shorter than a token's heads
    assert call(os=1028) == 1             # stride not a multiple of 8 elements
    assert call(q=0x1004) == 1            # misaligned pointer
    assert call(cu=0) == 1                # null pointer
    assert call(sc=float("inf")) == 1


def _decode_entry(L, name, **kw):
    """pd_decode (workspace arguments) or pd_decode_static_ws (none) with
    placeholder pointers: only argument checks may run."""
    args = dict(q=0x1000, k=0x2000, v=0x3000, bt=0x4000, lens=0x5000, out=0x7000, B=2, Hq=8,
                Hkv=2, D=128, bs=16, mbs=4, nb=8, scale=0.1, S=0, W=0, dt=0, ks=1.0, vs=1.0)
    args.update(kw)
    a = args
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    head = [a["q"], a["k"], a["v"], a["bt"], a["lens"], a["out"], a["B"], a["Hq"], a["Hkv"],
            a["D"], a["bs"], a["mbs"], a["nb"], a["scale"], a["S"], a["W"], a["dt"], a["ks"],
            a["vs"]]
    types = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, f32, i32, i32, i32, f32, f32]
    f = getattr(L, name)
    if name == "pd_decode_static_ws":
        f.argtypes = types + [P]
        return f(*head, None)
    f.argtypes = types + [P, ctypes.c_size_t, P]
    return f(*head, 0x6000, 1 << 20, None)


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), 2),                  # head_dim not built: refused before choosing S
    (dict(D=96, B=70000), 1),         # too many sequences comes first
    (dict(Hq=34, Hkv=2), 2),          # group of 17
    (dict(Hq=6, Hkv=4), 1),           # GQA ratio not integral
    (dict(dt=7), 2),                  # unknown cache form
    (dict(S=5000), 1),                # split count out of range
    (dict(dt=1, ks=0.0), 1),          # FP8 needs a positive scale
    (dict(out=0x7004), 1),            # misaligned output
    (dict(scale=float("inf")), 1),
])
def test_static_workspace_answers_like_pd_decode(pdlib, kw, code):
    """pd_decode_static_ws runs pd_decode's own checks in pd_decode's order,
    before any CUDA call, so a malformed request gets the same status from
    both (here on a host without a GPU)."""
    _, L = pdlib
    assert _decode_entry(L, "pd_decode", **kw) == code
    assert _decode_entry(L, "pd_decode_static_ws", **kw) == code
    assert _decode_entry(L, "pd_decode_crosscheck", **kw) == code


def test_fp8_scale_matches_oracle(pdlib):
    """pd_fp8_scale (host) against oracle_fp8_scale, bit for bit: special
    values and 200k random absmax values over the whole float range."""
    import numpy as np
    import oracle
    from paged_kv_split_gb300 import inputs
    _, L = pdlib
    L.pd_fp8_scale.argtypes, L.pd_fp8_scale.restype = [ctypes.c_float], ctypes.c_float
    orc = oracle.get()
    special = [0.0, -0.0, float("nan"), float("inf"), 1e-45, 1.1754942e-38, 448.0, 1.0, 3.0e38,
               -5.0, 6.0, 2.0 ** -9]
    rnd = inputs.uniform_int(71, 200000, 0, 0x7F7FFFFF).astype(np.uint32).view(np.float32)
    for x in special + [float(v) for v in rnd]:
        got = np.float32(L.pd_fp8_scale(x))
        want = np.float32(orc.fp8_scale(x))
        assert got.view(np.uint32) == want.view(np.uint32), (x, got, want)
