"""Decode benchmark: paged split-KV decode attention on GB300.

One step = one decode (partial kernel + log-sum-exp combine) over the whole
batch of the Llama-3-8B-shaped workload (32 sequences, 32 q / 8 kv heads,
head_dim 128, block_size 16, lengths uniform in [1024, 4096], BF16 cache, pages
shuffled across the pool), inputs resident in HBM. The schedule comes from the
host-held lengths: pd_prefer_balanced picks between pd_decode with the
length-aware split count and pd_decode_balanced with a host plan. Reported
value: KV-read GB/s = algorithmic bytes / step time (us/step alongside); e2e:
the same through the C ABI from pinned host inputs, planning included.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pd|reference]
                    [--workload llama8b|long_b4_32k|...] [--splits S]
                    [--schedule auto|split|balanced]

The prefill_* workloads time pd_prefill (paged chunked prefill over the same
cache) instead: value = attention TFLOP/s (4 * head_dim per query row, q head
and key seen), roofline against the measured bf16 tensor peak.

With torchrun (N > 1) every rank decodes its own independent batch (seeded by
rank, replicas only: no data is exchanged); the barrier and max-over-ranks
timing use torch.distributed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode µs/step and KV-read HBM GB/s (% of GB300 peak) at 1 GPU"
ELEM_BYTES = {0: 2.0, 1: 1.0, 2: 0.5625}
DTYPE_NAME = {0: "bf16", 1: "fp8_e4m3", 2: "nvfp4"}
PARTIAL_KERNEL_SRC = ["paged_kv_split_gb300/csrc/decode_mma.cu",
                      "paged_kv_split_gb300/csrc/decode_balanced.cu",
                      "paged_kv_split_gb300/csrc/mma_tile.cuh",
                      "paged_kv_split_gb300/csrc/mma_common.cuh",
                      "paged_kv_split_gb300/csrc/pd_common.cuh"]


def workload(name: str, rank: int = 0):
    from paged_kv_split_gb300 import inputs as I
    seed = 1000 * rank
    table = {
        "llama8b": lambda: I.llama8b(seed=seed),
        "long_b1_32k": lambda: I.long_context(1, 32768, seed=seed),
        "long_b4_32k": lambda: I.long_context(4, 32768, seed=seed),
        "long_b4_8k": lambda: I.long_context(4, 8192, seed=seed),
        "wide_d512": lambda: I.wide_head(seed=seed),
        "window_d256": lambda: I.sliding(seed=seed),
        "quant_fp8": lambda: I.quantised(1, seed=seed),
        "quant_nvfp4": lambda: I.quantised(2, seed=seed),
        # the llama8b batch with quantised caches (same shapes, same lengths)
        "llama8b_fp8": lambda: _with_dtype(I.llama8b(seed=seed), 1),
        "llama8b_nvfp4": lambda: _with_dtype(I.llama8b(seed=seed), 2),
        # paged (chunked) prefill over the same BF16 cache (pd_prefill)
        "prefill_chunked": lambda: I.prefill_chunked(seed=seed),
        "prefill_long": lambda: I.prefill_chunked(seed=seed, num_seqs=16, chunk=256,
                                                  max_context=7936),
    }
    return table[name]()


PREFILL_METRIC = "prefill µs/step and attention TFLOP/s (% of GB300 bf16 peak) at 1 GPU"


def prefill_flops(case, rows=None) -> float:
    """4 * D per (query row, q head, key seen): the two contractions Q K^T and
    P V, causal (query i of a sequence sees L - q_len + i + 1 keys), within the
    window. rows: optional (sequence, first row, last row + 1) sample."""
    cu = case.extra["cu_q"]
    W = case.sliding_window
    total = 0
    spans = rows or [(b, 0, int(cu[b + 1] - cu[b])) for b in range(case.num_seqs)]
    for b, i0, i1 in spans:
        L, ql = int(case.seq_lens[b]), int(cu[b + 1] - cu[b])
        seen = L - ql + np.arange(i0, i1, dtype=np.int64) + 1
        if W > 0:
            seen = np.minimum(seen, W)
        total += int(seen.sum())
    return 4.0 * case.head_dim * case.num_q_heads * total


def prefill_config(name, case, world):
    """The `config` of a prefill line, from the workload alone (both arms)."""
    return {"workload": name, "num_seqs": case.num_seqs,
            "query_rows": int(case.extra["cu_q"][-1]), "num_q_heads": case.num_q_heads,
            "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim,
            "block_size": case.block_size, "kv_dtype": "bf16", "causal": True,
            "max_q_len": int(case.extra["q_lens"].max()), "keys_max": int(case.seq_lens.max()),
            "flops_per_step": prefill_flops(case), "l2": L2_POLICY,
            "parallelism": f"replicas x{world}"}


def _with_dtype(case, kv_dtype):
    case.kv_dtype = kv_dtype
    case.name = f"{case.name}_{DTYPE_NAME[kv_dtype]}"
    return case


def algorithmic_bytes(case, kv_dtype) -> dict:
    """KV bytes read over the window + q + out + block-table entries touched."""
    L = case.seq_lens.astype(np.int64)
    W = case.sliding_window
    lo = np.where((W > 0) & (L > W), L - W, 0)
    keys = int((L - lo).sum())
    bs = case.block_size
    pages = int(np.where(L > lo, (L - 1) // bs - lo // bs + 1, 0).sum())
    kv = keys * case.num_kv_heads * 2 * case.head_dim * ELEM_BYTES[kv_dtype]
    q = case.num_seqs * case.num_q_heads * case.head_dim * 2
    return {"kv": kv, "q": q, "out": q, "table": 4 * pages, "total": kv + 2 * q + 4 * pages,
            "keys": keys}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in PARTIAL_KERNEL_SRC:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name: str):
    """Per-launch DRAM bytes of the partial kernel from a committed ncu
    summary, if it was captured from the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload_name)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms in the background."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.samples = []
        self.proc = None
        self.thread = None
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "50"]
            if gpu_uuid:
                cmd += ["-i", gpu_uuid]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        win = [s for t, s in self.samples if t0 <= t <= t1]
        if not win:  # a very short timed region: take the nearest samples after it
            win = [s for t, s in self.samples if t > t1][:2]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in win if num(s[0]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in win:
            for k, name in enumerate(names):
                if len(s) > 4 + k and s[4 + k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(win[0][1]) if len(win[0]) > 1 else None,
                "reasons": sorted(reasons), "samples": len(win)}


def dist_init(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce_over_ranks(x: float, world: int, op) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    # the reduction's tensor lives where the process group's backend wants it
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(x: float, world: int) -> float:
    import torch.distributed as dist
    return _reduce_over_ranks(x, world, dist.ReduceOp.MAX if world > 1 else None)


def sum_over_ranks(x: float, world: int) -> float:
    import torch.distributed as dist
    return _reduce_over_ranks(x, world, dist.ReduceOp.SUM if world > 1 else None)


def job_throughput(ms_step_local: float, bytes_local: float, world: int):
    """Whole-job figures of a replicas run: the slowest rank's ms per step and
    the bytes all ranks moved per step, divided (GB/s)."""
    ms_step = max_over_ranks(ms_step_local, world)
    total_bytes = sum_over_ranks(bytes_local, world)
    return ms_step, total_bytes, total_bytes / (ms_step * 1e-3) / 1e9


# ---------------------------------------------------------------------------
def time_oracle(case, kv_dtype, kc_host, vc_host, ks, vs, budget_s: float):
    """The oracle as it stands, single-threaded, on a bounded sample (the first
    k sequences of the batch, k grown until one call takes ~budget_s)."""
    import oracle
    orc = oracle.get()
    k = 1
    while True:
        t = time.perf_counter()
        orc.decode(case.q[:k], kc_host, vc_host, case.block_tables[:k], case.seq_lens[:k],
                   case.num_kv_heads, case.block_size, case.num_blocks, case.scale,
                   case.sliding_window, kv_dtype, ks, vs)
        dt = time.perf_counter() - t
        if dt >= budget_s or k >= case.num_seqs:
            break
        k = min(case.num_seqs, max(k + 1, int(k * budget_s / max(dt, 1e-3))))
    # median of three calls on the chosen sample
    times = [dt]
    for _ in range(2):
        t = time.perf_counter()
        orc.decode(case.q[:k], kc_host, vc_host, case.block_tables[:k], case.seq_lens[:k],
                   case.num_kv_heads, case.block_size, case.num_blocks, case.scale,
                   case.sliding_window, kv_dtype, ks, vs)
        times.append(time.perf_counter() - t)
    dt = statistics.median(times)
    sub = type(case)(**{**case.__dict__})
    sub.seq_lens = case.seq_lens[:k]
    sub.num_seqs = k
    sub.q = case.q[:k]
    ab = algorithmic_bytes(sub, kv_dtype)
    return k, dt, ab


def cpu_description() -> dict:
    """Host CPU model and core count (the oracle baseline runs on one core)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return {"nproc": os.cpu_count(), "model": model or platform.processor() or platform.machine()}


def build_device_state(case, kv_dtype, replicas, dev):
    import torch
    from paged_kv_split_gb300 import binding as pd

    def bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    key, value = bf16(case.key), bf16(case.value)
    slots = torch.from_numpy(case.slot_mapping).to(dev)
    ks = vs = 1.0
    if kv_dtype == 1:
        ks, vs = pd.fp8_calibrate(key, value)
    caches = []
    for _ in range(replicas):
        kc = pd.empty_cache(kv_dtype, case.num_blocks, case.block_size, case.num_kv_heads,
                            case.head_dim, dev)
        vc = torch.empty_like(kc)
        kc.zero_()
        vc.zero_()
        pd.pd_reshape_and_cache(key, value, kc, vc, slots, num_blocks=case.num_blocks,
                                block_size=case.block_size, kv_dtype=kv_dtype, k_scale=ks,
                                v_scale=vs)
        caches.append((kc, vc))
    del key, value
    return caches, ks, vs


def workload_config(case, kv_dtype, world: int) -> dict:
    """The `config` object of a decode line: the workload itself, computed from
    its seeded shapes alone, so that both arms (the GPU path and the oracle)
    print the same dict."""
    ab = algorithmic_bytes(case, kv_dtype)
    return {"workload": None, "num_seqs": case.num_seqs,
            "num_q_heads": case.num_q_heads, "num_kv_heads": case.num_kv_heads,
            "head_dim": case.head_dim, "block_size": case.block_size,
            "kv_dtype": DTYPE_NAME[kv_dtype], "sliding_window": case.sliding_window,
            "keys_per_step": ab["keys"], "algorithmic_bytes_per_step": int(ab["total"]),
            "l2": L2_POLICY, "parallelism": f"replicas x{world}"}


L2_POLICY = ("inputs larger than L2: the GPU arm rotates cache replicas whose K/V together "
             "exceed 3x the L2, so no step reads K/V left in L2 by the previous one")
NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s HBM3e figure the target is stated against


def queue_ahead(steps: int) -> None:
    """Hold the stream in a short device-side spin (torch's sleep kernel)
    while the host enqueues the timed launches, so that a short timed region
    measures back-to-back device execution, not host launch latency; it runs
    before the start event and is not part of the timing."""
    import torch
    seconds = min(0.05, 0.002 + 60e-6 * steps)
    torch.cuda._sleep(int(seconds * 2.0e9))


def timed_region(stream, n, body, queue=True):
    """Device time (ms) of n calls of body(i), CUDA events on `stream`."""
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if queue:
        queue_ahead(n)
    start.record(stream)
    for i in range(n):
        body(i)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


class DecodeSetup:
    """Device state and the decode calls of one workload: cache replicas
    (together more than 3x the L2, rotated per step), the schedule the host
    lengths choose, and closures for a full step and its two kernels."""

    def __init__(self, args, case, dev, schedule="auto", splits=0):
        import torch
        from paged_kv_split_gb300 import binding as pd
        self.case, self.dev = case, dev
        kv_dtype = self.kv_dtype = case.kv_dtype
        self.ab = algorithmic_bytes(case, kv_dtype)
        self.cache_bytes = pd.pd_cache_bytes(kv_dtype, case.num_blocks, case.block_size,
                                             case.num_kv_heads, case.head_dim)
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.replicas = max(2, math.ceil(3 * self.l2 / max(2 * self.cache_bytes, 1)))
        self.caches, ks, vs = build_device_state(case, kv_dtype, self.replicas, dev)
        self.ks, self.vs = ks, vs
        q = self.q = torch.from_numpy(case.q.view(np.int16)).to(dev).view(torch.bfloat16)
        bt = self.bt = torch.from_numpy(case.block_tables).to(dev)
        lens = self.lens = torch.from_numpy(case.seq_lens).to(dev)
        out = self.out = torch.empty_like(q)
        B, hq, D = case.q.shape
        mbs = case.max_blocks_per_seq
        sms = self.sms = torch.cuda.get_device_properties(dev).multi_processor_count
        self.stream = torch.cuda.current_stream(dev)
        G = hq // case.num_kv_heads
        kw = self.kw = dict(num_kv_heads=case.num_kv_heads, block_size=case.block_size,
                            num_blocks=case.num_blocks, scale=case.scale,
                            sliding_window=case.sliding_window, kv_dtype=kv_dtype, k_scale=ks,
                            v_scale=vs)
        # the host holds the batch's lengths (as a serving scheduler does): the
        # schedule (split-KV with the length-aware split count, or the balanced
        # plan) is chosen and planned from them
        if schedule == "auto":
            schedule = "balanced" if (not splits and pd.pd_prefer_balanced(
                case.seq_lens, num_q_heads=hq, num_kv_heads=case.num_kv_heads,
                max_blocks_per_seq=mbs, block_size=case.block_size, head_dim=D,
                sliding_window=case.sliding_window, kv_dtype=kv_dtype, num_sms=sms)) else "split"
        self.schedule = schedule
        if schedule == "balanced":
            def make_plan(out_buf=None):
                return pd.pd_balanced_plan(case.seq_lens, num_q_heads=hq,
                                           num_kv_heads=case.num_kv_heads, head_dim=D,
                                           block_size=case.block_size, max_blocks_per_seq=mbs,
                                           sliding_window=case.sliding_window,
                                           kv_dtype=kv_dtype, num_sms=sms, out=out_buf)
            self.make_plan = make_plan
            plan = self.plan = make_plan()
            plan_d = self.plan_d = plan.to(dev)
            ws = torch.zeros(max(plan.workspace_bytes, 16), dtype=torch.uint8, device=dev)
            self.sched = {"schedule": "balanced (host plan)", "plan_ctas": plan.num_ctas,
                          "plan_pieces": plan.num_pieces}
            self.ws_traffic = 2 * plan.num_pieces * G * (D + 2) * 4

            def decode(kc, vc, q_, bt_, lens_, out_, plan_dev=None):
                pd.pd_decode_balanced(q_, kc, vc, bt_, plan_d if plan_dev is None else plan_dev,
                                      plan, out_, workspace=ws, **kw)

            def partial_only(kc, vc):
                pd.pd_decode_balanced_partial(q, kc, vc, bt, plan_d, plan, out, workspace=ws,
                                              **kw)

            def combine_only(kc, vc):
                pd.pd_decode_balanced_combine(q, kc, vc, bt, plan_d, plan, out, workspace=ws,
                                              **kw)
        else:
            S = splits or pd.pd_plan_num_splits_for_lengths(
                case.seq_lens, hq, case.num_kv_heads, mbs, case.block_size, case.sliding_window,
                D, kv_dtype, sms)
            ws = torch.empty(pd.pd_decode_workspace_bytes(B, hq, D, S), dtype=torch.uint8,
                             device=dev)
            self.sched = {"schedule": "split-KV", "num_splits": S,
                          "split_planner": "given" if splits else "seq_lens"}
            self.ws_traffic = 2 * B * hq * S * (D + 2) * 4

            def decode(kc, vc, q_, bt_, lens_, out_, plan_dev=None):
                pd.pd_decode(q_, kc, vc, bt_, lens_, out_, workspace=ws, num_splits=S, **kw)

            def partial_only(kc, vc):
                pd.pd_decode_partial(q, kc, vc, bt, lens, ws, num_splits=S, **kw)

            def combine_only(kc, vc):
                pd.pd_decode_combine(ws, lens, out, block_size=case.block_size,
                                     max_blocks_per_seq=mbs, num_splits=S,
                                     sliding_window=case.sliding_window)
        self.decode, self.partial_only, self.combine_only = decode, partial_only, combine_only

    def step(self, i):
        # one decode step = the partial kernel, then the combine launched as its
        # programmatic dependent, on the next cache replica
        kc, vc = self.caches[i % self.replicas]
        self.decode(kc, vc, self.q, self.bt, self.lens, self.out)

    def partial_ms(self, n):
        """Mean device time of the partial kernel alone (events around each
        launch, the combine launched after each, queued ahead)."""
        import torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        queue_ahead(2 * n)
        for i in range(n):
            kc, vc = self.caches[i % self.replicas]
            evs[i][0].record(self.stream)
            self.partial_only(kc, vc)
            evs[i][1].record(self.stream)
            self.combine_only(kc, vc)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    def roofline(self, part_ms, peak, peak_kind, workload_name=None):
        partial_bytes = self.ab["kv"] + self.ab["q"] + self.ab["table"]
        achieved = partial_bytes / (part_ms * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": "partial (" + self.sched["schedule"] + ")",
                "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_kind,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": recorded_traffic(workload_name) if workload_name else None,
                "algorithmic_bytes_per_launch": int(partial_bytes),
                "partial_us_per_launch": round(part_ms * 1e3, 2)}


def measure_workload(args, name, dev, steps=200, warmup=10):
    """A compact figure for one more workload (the `workloads` object of the
    default line): device-timed steps with L2 kept cold, the partial kernel's
    roofline fraction, the schedule and the clocks. No CPU baseline, no e2e."""
    import torch
    case = workload(name, 0)
    st = DecodeSetup(args, case, dev)
    for i in range(warmup):
        st.step(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid(dev))
    time.sleep(0.2)
    w0 = time.time()
    ms = timed_region(st.stream, steps, st.step) / steps
    w1 = time.time()
    time.sleep(0.1)
    sampler.stop()
    peak, kind = measured_peaks()
    part = st.partial_ms(min(steps, 100))
    gbs = st.ab["total"] / (ms * 1e-3) / 1e9
    r = st.roofline(part, peak, kind, name)
    out = {"us_per_step": round(ms * 1e3, 2), "value": round(gbs, 1), "unit": "GB/s",
           "frac": round(gbs / peak, 4), "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
           "partial_frac": r["frac"], "partial_us": r["partial_us_per_launch"],
           "partial_traffic": r["traffic"], "partial_algorithmic_bytes": r["algorithmic_bytes_per_launch"],
           "kv_dtype": DTYPE_NAME[case.kv_dtype], "steps": steps, **st.sched,
           "clocks": sampler.summary(w0, w1)}
    del st
    torch.cuda.empty_cache()
    return out


def gpu_uuid(dev):
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None


EXTRA_WORKLOADS = ["long_b4_32k", "long_b4_8k", "long_b1_32k", "wide_d512", "window_d256",
                   "quant_fp8", "quant_nvfp4"]


def run_pd(args, rank, world, local):
    import torch
    from paged_kv_split_gb300 import binding as pd

    dev = torch.device("cuda", local if world > 1 else 0)
    case = workload(args.workload, rank)
    kv_dtype = case.kv_dtype
    st = DecodeSetup(args, case, dev, args.schedule, args.splits)
    ab = st.ab
    B, hq, D = case.q.shape
    stream = st.stream
    replicas, caches = st.replicas, st.caches
    q, bt, lens, out = st.q, st.bt, st.lens, st.out
    decode, step = st.decode, st.step

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(gpu_uuid(dev))
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    w0 = time.time()
    total_ms = timed_region(stream, args.steps, step)
    w1 = time.time()
    barrier(world)
    time.sleep(0.1)
    sampler.stop()
    clocks = sampler.summary(w0, w1)
    # the partial kernel's own duration (events around each launch)
    n_inst = min(args.steps, 500)
    part_ms = st.partial_ms(n_inst)

    # per-step spread of the whole decode step (events around each pd_decode:
    # the event between steps also ends the programmatic overlap of the next
    # step's partial grid with this step's combine)
    n_dist = min(args.steps, 500)
    evd = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_dist)]
    queue_ahead(n_dist)
    for i in range(n_dist):
        evd[i][0].record(stream)
        step(i)
        evd[i][1].record(stream)
    torch.cuda.synchronize(dev)
    step_us = np.array([a.elapsed_time(b) * 1e3 for a, b in evd])
    spread = {f"p{p}": round(float(np.percentile(step_us, p)), 2) for p in (10, 50, 90)}

    # hot L2, labelled as such: one cache replica every step, so its K/V stays
    # in L2 as far as it fits (the headline rotates replicas past L2)
    n_hot = min(args.steps, 1000)
    for _ in range(3):
        kc, vc = caches[0]
        decode(kc, vc, q, bt, lens, out)
    torch.cuda.synchronize(dev)

    def hot_step(i):
        kc, vc = caches[0]
        decode(kc, vc, q, bt, lens, out)
    hot_us = timed_region(stream, n_hot, hot_step) * 1e3 / n_hot

    # the same step captured in CUDA graphs (one per cache replica), replayed in rotation
    def timed_replays(graphs, n):
        for i in range(3):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize(dev)
        return timed_region(stream, n, lambda i: graphs[i % len(graphs)].replay()) * 1e3 / n

    n_graph = min(args.steps, 2000)
    graphs = []
    for rep_i in range(replicas):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(rep_i)
        graphs.append(g)
    graph_us = timed_replays(graphs, n_graph)

    # a serving step: write one new token per sequence (its K and V), then
    # decode, both in one graph; the write lands on each sequence's last slot
    L = case.seq_lens.astype(np.int64)
    last_slot = (case.block_tables[np.arange(B), np.maximum(L - 1, 0) // case.block_size]
                 .astype(np.int64) * case.block_size + np.maximum(L - 1, 0) % case.block_size)
    from paged_kv_split_gb300 import inputs as I
    new_k = torch.from_numpy(I.normal_bf16(77, (B, case.num_kv_heads, D)).view(np.int16)).to(
        dev).view(torch.bfloat16)
    new_v = torch.from_numpy(I.normal_bf16(78, (B, case.num_kv_heads, D)).view(np.int16)).to(
        dev).view(torch.bfloat16)
    slots_new = torch.from_numpy(np.where(L > 0, last_slot, -1).astype(np.int32)).to(dev)
    graphs_w = []
    for rep_i in range(replicas):
        kc, vc = caches[rep_i]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            pd.pd_reshape_and_cache(new_k, new_v, kc, vc, slots_new, num_blocks=case.num_blocks,
                                    block_size=case.block_size, kv_dtype=kv_dtype,
                                    k_scale=st.ks, v_scale=st.vs)
            decode(kc, vc, q, bt, lens, out)
        graphs_w.append(g)
    graph_w_us = timed_replays(graphs_w, n_graph)
    del graphs, graphs_w

    ms_step_local = total_ms / args.steps
    ms_step, total_bytes, value = job_throughput(ms_step_local, ab["total"], world)

    # roofline of the dominant kernel (the split-KV partial)
    peak, peak_kind = measured_peaks()
    roofline = st.roofline(part_ms, peak, peak_kind, args.workload)
    roofline["timed_launches"] = n_inst

    # e2e: through the C ABI from pinned host memory, copies inside the timing.
    # Each step's inputs (q, block table, lengths and, for the balanced
    # schedule, the plan) sit in one pinned staging buffer and cross in one
    # copy; the output comes back every step.
    balanced = st.schedule == "balanced"
    out_ref = out.clone()  # the device-timed steps' output, to check the e2e one against
    parts = [("q", q.numel() * 2), ("bt", bt.numel() * 4), ("lens", lens.numel() * 4)]
    if balanced:
        parts.append(("plan", pd.balanced_plan_buffer(B, case.num_kv_heads, st.sms).numel() * 4))
    offs, h2d = {}, 0
    for name, nb in parts:  # 256-byte aligned segments
        offs[name] = (h2d, nb)
        h2d += (nb + 255) // 256 * 256
    stage_h = [torch.zeros(h2d, dtype=torch.uint8).pin_memory() for _ in range(2)]
    for s in stage_h:
        for name, arr in (("q", case.q), ("bt", case.block_tables), ("lens", case.seq_lens)):
            o, nb = offs[name]
            s[o:o + nb].copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)))
    stage_d = torch.empty(h2d, dtype=torch.uint8, device=dev)

    def seg(buf, name, dtype):
        o, nb = offs[name]
        return buf[o:o + nb].view(dtype)

    q_d = seg(stage_d, "q", torch.bfloat16).view(q.shape)
    bt_d = seg(stage_d, "bt", torch.int32).view(bt.shape)
    lens_d = seg(stage_d, "lens", torch.int32)
    out_h = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(10, min(args.steps, 200))
    if balanced:
        # step i copies one staging buffer while the host plans step i + 1
        # into the other
        plan_h = [seg(s, "plan", torch.int32) for s in stage_h]
        plan_dd = seg(stage_d, "plan", torch.int32)
        st.make_plan(plan_h[0])

    def e2e_step(i):
        kc, vc = caches[i % replicas]
        stage_d.copy_(stage_h[i % 2], non_blocking=True)
        if balanced:
            decode(kc, vc, q_d, bt_d, lens_d, out, plan_dev=plan_dd)
        else:
            decode(kc, vc, q_d, bt_d, lens_d, out)
        out_h.copy_(out, non_blocking=True)
        if balanced:
            # the scheduler plans every step (lengths change as tokens arrive);
            # the next step's lengths are known now (one more token each), so
            # its plan is built while the device runs this step
            st.make_plan(plan_h[(i + 1) % 2])
        stream.synchronize()

    for i in range(3):
        e2e_step(i)
    barrier(world)
    t = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    e2e_s = max_over_ranks((time.perf_counter() - t) / e2e_steps, world)
    same = bool(torch.equal(out_h.view(torch.int16), out_ref.cpu().view(torch.int16)))
    d2h = out_h.numel() * 2
    e2e = {"value": round(total_bytes / e2e_s / 1e9, 1), "unit": "GB/s",
           "us_per_step": round(e2e_s * 1e6, 2), "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h),
           "output_equals_device_timed": same}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        kc, vc = caches[0]
        k, dt, sab = time_oracle(case, kv_dtype, kc.cpu().numpy(), vc.cpu().numpy(), st.ks,
                                 st.vs, args.cpu_budget)
        cpu = {"value": round(sab["total"] / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle", "us_per_step_sample": round(dt * 1e6, 1),
               "host": cpu_description(), "timing": "median of 3 calls",
               "sample": f"first {k} of {case.num_seqs} sequences of the same batch "
                         f"({sab['keys']} keys), one single-threaded oracle_decode call"}
    sched, ws_traffic = st.sched, st.ws_traffic
    del st, caches
    torch.cuda.empty_cache()

    # the other configurations, compact (rank 0 of a one-GPU run; skipped with
    # --workloads none)
    extra = None
    if rank == 0 and world == 1 and args.workloads != "none":
        names = EXTRA_WORKLOADS if args.workloads == "all" else args.workloads.split(",")
        extra = {n: measure_workload(args, n, dev) for n in names if n != args.workload}

    if rank == 0:
        config = workload_config(case, kv_dtype, world)
        config["workload"] = args.workload
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "us_per_step": round(ms_step * 1e3, 2),
            "pct_of_hbm_peak": round(100 * value / peak, 2),
            "pct_of_nominal_8tbs": round(100 * value / NOMINAL_HBM_GBS, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE_NAME[kv_dtype], "data": "synthetic",
            "config": config,
            "schedule": {**sched, "workspace_bytes_per_step": int(ws_traffic),
                         "cache_replicas": replicas},
            "step_us": spread,
            "hot_l2": {"us_per_step": round(hot_us, 2),
                       "value": round(ab["total"] / (hot_us * 1e-6) / 1e9, 1), "unit": "GB/s",
                       "note": "one cache replica reused every step (K/V "
                               f"{2 * st_cache_mb(case, kv_dtype):.0f} MB): L2-warm, "
                               "not the headline"},
            "graph": {"us_per_step": round(graph_us, 2),
                      "value": round(ab["total"] / (graph_us * 1e-6) / 1e9, 1), "unit": "GB/s",
                      "note": "pd_decode captured in one CUDA graph per cache replica"},
            "graph_with_write": {"us_per_step": round(graph_w_us, 2),
                                 "tokens_written": int(B),
                                 "note": "pd_reshape_and_cache of one token per sequence, then "
                                         "pd_decode, captured in one CUDA graph"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": 2 * args.steps, "clocks": clocks,
            "workloads": extra,
        }
        print(json.dumps(line), flush=True)


def st_cache_mb(case, kv_dtype):
    from paged_kv_split_gb300 import binding as pd
    return pd.pd_cache_bytes(kv_dtype, case.num_blocks, case.block_size, case.num_kv_heads,
                             case.head_dim) / 1e6


def time_oracle_prefill(case, kc_host, vc_host, budget_s: float):
    """oracle_prefill as it stands, single-threaded, on a bounded sample: the
    last k query rows of the first sequence, k grown until a call takes about
    budget_s; median of three calls."""
    import oracle
    orc = oracle.get()
    ql = int(case.extra["cu_q"][1])

    def call(k):
        t = time.perf_counter()
        orc.prefill(case.q[ql - k:ql], np.array([0, k], np.int32), kc_host, vc_host,
                    case.block_tables[:1], case.seq_lens[:1], case.num_kv_heads,
                    case.block_size, case.num_blocks, case.scale, True, case.sliding_window)
        return time.perf_counter() - t
    k = 1
    while True:
        dt = call(k)
        if dt >= budget_s or k >= ql:
            break
        k = min(ql, max(k + 1, int(k * budget_s / max(dt, 1e-3))))
    dt = statistics.median([dt, call(k), call(k)])
    flops = prefill_flops(case, [(0, ql - k, ql)])
    return k, dt, flops


def run_prefill(args, rank, world, local):
    import torch
    from paged_kv_split_gb300 import binding as pd

    dev = torch.device("cuda", local if world > 1 else 0)
    case = workload(args.workload, rank)
    T, hq, D = case.q.shape
    cu = case.extra["cu_q"]
    max_q = int(case.extra["q_lens"].max())
    flops = prefill_flops(case)
    page_bytes = pd.pd_page_bytes(0, case.block_size, case.num_kv_heads, D)
    cache_bytes = case.num_blocks * page_bytes
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    replicas = max(2, math.ceil(3 * l2 / max(2 * cache_bytes, 1)))
    caches, _, _ = build_device_state(case, 0, replicas, dev)
    q = torch.from_numpy(case.q.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty_like(q)
    cu_d = torch.from_numpy(cu).to(dev)
    bt = torch.from_numpy(case.block_tables).to(dev)
    lens = torch.from_numpy(case.seq_lens).to(dev)
    kw = dict(max_q_len=max_q, num_kv_heads=case.num_kv_heads, block_size=case.block_size,
              num_blocks=case.num_blocks, scale=case.scale, causal=True,
              sliding_window=case.sliding_window,
              crosscheck=args.prefill_kernel == "mma_sync")

    def step(i):
        kc, vc = caches[i % replicas]
        pd.pd_prefill(q, cu_d, kc, vc, bt, lens, out, **kw)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    time.sleep(0.3)  # first samples before the timed region
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0 = time.time()
    ms_local = timed_region(stream, args.steps, step) / args.steps
    t1 = time.time()
    barrier(world)
    ms_step = max_over_ranks(ms_local, world)
    total_flops = sum_over_ranks(flops, world)
    tflops = total_flops / (ms_step * 1e-3) / 1e12
    clocks = sampler.summary(t0, t1)
    sampler.stop()

    # e2e through the C ABI: q, cu_q and lengths from pinned host memory, the
    # output read back, every step
    q_h = torch.from_numpy(case.q.view(np.int16)).pin_memory()
    cu_h = torch.from_numpy(cu).pin_memory()
    lens_h = torch.from_numpy(case.seq_lens).pin_memory()
    out_h = torch.empty(q_h.shape, dtype=torch.int16).pin_memory()
    q_e = torch.empty_like(q)
    cu_e, lens_e = torch.empty_like(cu_d), torch.empty_like(lens)

    def e2e_step(i):
        q_e.view(torch.int16).copy_(q_h, non_blocking=True)
        cu_e.copy_(cu_h, non_blocking=True)
        lens_e.copy_(lens_h, non_blocking=True)
        kc, vc = caches[i % replicas]
        pd.pd_prefill(q_e, cu_e, kc, vc, bt, lens_e, out, **kw)
        out_h.copy_(out.view(torch.int16), non_blocking=True)

    n_e2e = max(3, min(args.steps, 200))
    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(n_e2e):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world)
    h2d = q_h.numel() * 2 + cu_h.numel() * 4 + lens_h.numel() * 4
    d2h = out_h.numel() * 2
    if rank != 0:
        return
    peak_t = None
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            peak_t, peak_src = float(json.load(f)["bf16_tflops"]), "measured (bf16 burst)"
    if peak_t is None:
        peak_t, peak_src = 1900.0, "fallback"
    achieved = flops / (ms_local * 1e-3) / 1e12
    line = {
        "metric": PREFILL_METRIC, "value": round(tflops, 1), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "us_per_step": round(ms_step * 1e3, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": prefill_config(args.workload, case, world),
        "cache_replicas": replicas,
        "roofline": {"bound": "tensor",
                     "kernel": ("prefill_mma_kernel (mma.sync bf16, pd_prefill_crosscheck)"
                                if args.prefill_kernel == "mma_sync"
                                else "prefill_pair_kernel (tcgen05 bf16, two query tiles per "
                                     "CTA, TMEM accumulators)" if D <= 128
                                else "prefill_umma_kernel (tcgen05 bf16, TMEM accumulators)"),
                     "achieved": round(achieved, 1), "peak": peak_t, "peak_source": peak_src,
                     "unit": "TFLOP/s", "frac": round(achieved / peak_t, 4), "traffic": None},
        "e2e": {"value": round(total_flops / (ms_e2e * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                "us_per_step": round(ms_e2e * 1e3, 1), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        kc, vc = caches[0]
        k, dt, sflops = time_oracle_prefill(case, kc.cpu().numpy(), vc.cpu().numpy(),
                                            args.cpu_budget / 3)
        line["cpu_baseline"] = {
            "value": round(sflops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
            "kind": "oracle", "us_per_step_sample": round(dt * 1e6, 1),
            "host": cpu_description(), "timing": "median of 3 calls",
            "sample": f"last {k} of {int(cu[1])} query rows of sequence 0, one "
                      f"single-threaded oracle_prefill call"}
    print(json.dumps(line), flush=True)


def run_reference_prefill(args, case):
    """The reference arm for a prefill workload: oracle_prefill on host cores."""
    import oracle
    orc = oracle.get()
    n = orc.cache_bytes(0, case.num_blocks, case.block_size, case.num_kv_heads, case.head_dim)
    kc = np.zeros(n, np.uint8)
    vc = np.zeros(n, np.uint8)
    orc.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping, case.num_kv_heads,
                          case.head_dim, case.block_size, case.num_blocks, 0)
    per_step = min(2.0, 150.0 / max(args.steps + args.warmup, 1))
    k, _, sflops = time_oracle_prefill(case, kc, vc, per_step)
    ql = int(case.extra["cu_q"][1])
    times = []
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        orc.prefill(case.q[ql - k:ql], np.array([0, k], np.int32), kc, vc,
                    case.block_tables[:1], case.seq_lens[:1], case.num_kv_heads,
                    case.block_size, case.num_blocks, case.scale, True, case.sliding_window)
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    s = sum(times) / len(times)
    value = sflops / s / 1e12
    sample = (f"last {k} of {ql} query rows of sequence 0 per step, single-threaded "
              f"oracle_prefill")
    print(json.dumps({
        "impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": prefill_config(args.workload, case, 1),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": 1,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_reference(args, rank, world):
    """The oracle as it stands, timed on host cores, on a bounded sample."""
    if rank != 0:
        return
    case = workload(args.workload, 0)
    if args.workload.startswith("prefill_"):
        run_reference_prefill(args, case)
        return
    kv_dtype = case.kv_dtype
    import oracle
    orc = oracle.get()
    ks = vs = 1.0
    if kv_dtype == 1:
        ks = orc.fp8_scale(orc.absmax_bf16(case.key))
        vs = orc.fp8_scale(orc.absmax_bf16(case.value))
    n = orc.cache_bytes(kv_dtype, case.num_blocks, case.block_size, case.num_kv_heads,
                        case.head_dim)
    kc = np.zeros(n, np.uint8)
    vc = np.zeros(n, np.uint8)
    orc.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping, case.num_kv_heads,
                          case.head_dim, case.block_size, case.num_blocks, kv_dtype, ks, vs)
    per_step = min(2.0, 150.0 / max(args.steps + args.warmup, 1))
    k, _, sab = time_oracle(case, kv_dtype, kc, vc, ks, vs, per_step)
    times = []
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        orc.decode(case.q[:k], kc, vc, case.block_tables[:k], case.seq_lens[:k],
                   case.num_kv_heads, case.block_size, case.num_blocks, case.scale,
                   case.sliding_window, kv_dtype, ks, vs)
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    s = sum(times) / len(times)
    value = sab["total"] / s / 1e9
    sample = (f"first {k} of {case.num_seqs} sequences ({sab['keys']} keys) per step, "
              f"single-threaded oracle_decode")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_NAME[kv_dtype], "data": "synthetic",
        "config": {**workload_config(case, kv_dtype, world), "workload": args.workload},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pd", choices=["pd", "reference"])
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--schedule", default="auto", choices=["auto", "split", "balanced"])
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workloads", default="all",
                    help="the other decode configurations measured compactly into the line's "
                         "`workloads` object: all, none, or a comma-separated list")
    ap.add_argument("--prefill-kernel", default="tcgen05", choices=["tcgen05", "mma_sync"])
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    from paged_kv_split_gb300 import build as pd_build
    pd_build.build()
    rank, world, local = dist_init(args)
    try:
        if args.workload.startswith("prefill_"):
            run_prefill(args, rank, world, local)
        else:
            run_pd(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
