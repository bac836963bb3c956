"""Benchmark: paged decode attention on GB300 through the C ABI.

One step = one pass of the hot path over one batch: the cache write of every
sequence's new token followed by decode attention over the paged KV cache, as
the library's one call for it (pa_attention_varlen on decode tokens: the write,
then the split-context decode as the write's programmatic dependent, then its
merge kernel); the same step as the two calls pa_cache_write + pa_decode is
timed beside it.
Default workload: the Llama-3-8B-shaped decode layer (256 sequences, 32 query /
8 KV heads, head_size 128, block_size 16, lengths U{512..4096}).

Printed (rank 0, one JSON line): KV bytes read per second over the timed
steps (device time, inputs resident in HBM), seqs/s, the decode kernel's
roofline against the measured HBM copy bandwidth, an end-to-end figure with the
step's inputs copied from pinned host memory and the output copied back, SM
clocks sampled during the timed region, and the CPU oracle timed on a bounded
sample of the same workload.

Multi-GPU: the path needs no exchange (sequences are independent), so each rank
runs its own replica of the workload (weak scaling); timing is the max over
ranks.  ``--impl reference`` times the CPU fp64 oracle instead.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-attn decode: achieved KV-read GB/s (% of HBM peak) and seqs/s"
UNIT = "GB/s"
DEFAULT_WORKLOAD = 2


# ----------------------------------------------------------------------------- helpers

def kv_read_bytes(seq_lens, num_kv_heads: int, head_size: int) -> int:
    """Token-granular K+V bytes decode reads: sum_s 2*L_s*Hkv*D*2."""
    return int(sum(int(L) for L in seq_lens)) * 2 * num_kv_heads * head_size * 2


def decode_algorithmic_bytes(b, elem_bytes: int = 2) -> int:
    """KV read + q read + out write + tables and lengths read, per decode launch."""
    kv = kv_read_bytes(b.seq_lens.tolist(), b.num_kv_heads, b.head_size) * elem_bytes // 2
    qo = 2 * b.q.numel() * 2
    nblk = sum(-(-int(L) // b.block_size) for L in b.seq_lens.tolist())
    return kv + qo + nblk * 4 + b.num_seqs * 4


def cascade_algorithmic_bytes(b, shared_len: int, kv_elem_bytes: int = 2) -> int:
    """Bytes a shared-prefix decode must move: the shared tokens' K+V once, each
    sequence's own tokens, q, out and the tables; the prefix partials stay in L2.
    kv_elem_bytes: 2 for a bf16 pool, 1 for FP8."""
    own = [int(L) - shared_len for L in b.seq_lens.tolist()]
    kv = kv_read_bytes([shared_len] + own, b.num_kv_heads, b.head_size) * kv_elem_bytes // 2
    qo = 2 * b.q.numel() * 2
    nblk = shared_len // b.block_size + sum(-(-L // b.block_size) for L in own)
    return kv + qo + nblk * 4 + b.num_seqs * 4


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def profile_traffic(name: str):
    """DRAM bytes per launch from a committed ncu summary, if its kernel sources are unchanged."""
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    srcs = fields.get("source", "").split(",")
    want = fields.get("source_sha256", "").split(",")
    if len(srcs) != len(want):
        return None
    for name, sha in zip(srcs, want):
        src = os.path.join(ROOT, "paged_kv_cache_287_gb300", "csrc", name.strip())
        if not name.strip() or not os.path.exists(src):
            return None
        with open(src, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != sha.strip():
                return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Samples SM clock, power and clock-event reasons through NVML (read only)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: torch.device):
        self.ok = False
        self.samples = []
        self.max_mhz = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(device)
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            if self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) != 0:
                if self.nvml.nvmlDeviceGetHandleByIndex_v2(device.index or 0,
                                                           ctypes.byref(self.h)) != 0:
                    return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self._reasons_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) \
                or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _poll(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        pw = ctypes.c_uint()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                self._reasons_fn(self.h, ctypes.byref(rs))
                self.nvml.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw))
                self.samples.append((int(clk.value), int(rs.value), pw.value / 1000.0))
            time.sleep(0.002)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._poll, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "source": "nvml" if self.ok else "unavailable"}
        reasons = set()
        for _, r, _ in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "power_w_max": max(s[2] for s in self.samples),
                "samples": len(self.samples), "source": "nvml"}


def rejected_clocks(c) -> bool:
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(c.get("reasons", [])):
        return True
    if c.get("sm_mhz") and c.get("sm_max_mhz") and not c["reasons"]:
        return c["sm_mhz"] < 0.6 * c["sm_max_mhz"]
    return False


def median_launch_ms(fn, stream, runs: int = 50, flush=None) -> float:
    """Median device time of `runs` calls of fn(), each bracketed by its own pair
    of CUDA events on `stream` (the stream fn launches on); flush(), untimed, runs
    before each call when given (an L2 flush between runs)."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(runs)]
    torch.cuda.synchronize()
    for e0, e1 in evs:
        if flush is not None:
            flush()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)


def back_to_back_ms(fn, stream, n: int = 20, runs: int = 10) -> float:
    """Device time per call of a short kernel: n calls back to back between one
    pair of CUDA events, queued behind a bounded sleep kernel (about 100 us) so
    that the host's submission stays ahead of the GPU; the median over runs."""
    ts = []
    for _ in range(runs):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda._sleep(200000)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) / n)
    return statistics.median(ts)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_oracle_rate(n: int, budget_s: float = 12.0, seed=None, first: int = 64,
                    threads: int = 0):
    """Time the oracle (cache write + attention) on the first sequences of workload n.

    Sequences are processed one at a time, cycling over the sample, until about
    budget_s seconds of wall time are spent; threads = 0 uses every host core.
    Returns (GB/s of KV read, seqs/s, sequences timed, sample size, threads).
    """
    import numpy as np

    import oracle
    from paged_kv_cache_287_gb300.workloads import config_spec, sample_of_config

    k = min(len(config_spec(n)["seq_lens"]), first)
    b = sample_of_config(n, k, device="cpu", seed=seed)
    lib = oracle.load()
    threads = threads or oracle.max_threads(lib)
    lens = b.seq_lens.tolist()
    pool = oracle._u16(b.kv_cache).copy()
    done_bytes = 0
    done = 0
    spent = 0.0
    while spent < budget_s:
        s = done % k
        one = slice(s, s + 1)
        r0, r1 = int(b.cu_q_lens[s]), int(b.cu_q_lens[s + 1])
        t = time.perf_counter()
        oracle.cache_write(pool, b.k_new[r0:r1], b.v_new[r0:r1], b.slot_mapping[r0:r1], lib=lib,
                           inplace=True)
        oracle.attention(b.q[r0:r1], np.array([0, r1 - r0], np.int32), pool,
                         b.block_tables[one], b.seq_lens[one], b.num_heads, b.scale,
                         threads=threads, lib=lib)
        spent += time.perf_counter() - t
        done_bytes += kv_read_bytes(lens[s:s + 1], b.num_kv_heads, b.head_size)
        done += 1
    return done_bytes / spent / 1e9, done / spent, done, k, threads


def cpu_mixed_step_ms(b, stride: int = 8, threads: int = 0):
    """The oracle's time for one step of a flattened mixed batch (cache write of
    every new token + fp64 attention of every chunk row and decode token),
    estimated from a timed sample: the whole cache write, then attention of every
    stride-th row, scaled by causally visible (query, key) pairs.  Returns
    (ms per step, sampled rows, all rows, threads)."""
    import numpy as np

    import oracle

    lib = oracle.load()
    threads = threads or oracle.max_threads(lib)
    cu = b.cu_q_lens.tolist()
    lens = b.seq_lens.tolist()
    vis = []  # visible keys of every query row
    for s in range(b.num_seqs):
        ql = cu[s + 1] - cu[s]
        vis += [lens[s] - ql + i + 1 for i in range(ql)]
    rows = np.arange(0, len(vis), stride, dtype=np.int32)
    pool = oracle._u16(b.kv_cache).copy()
    t = time.perf_counter()
    oracle.cache_write(pool, b.k_new, b.v_new, b.slot_mapping, lib=lib, inplace=True)
    tw = time.perf_counter() - t
    t = time.perf_counter()
    oracle.attention(b.q, b.cu_q_lens, pool, b.block_tables, b.seq_lens, b.num_heads, b.scale,
                     rows=rows, threads=threads, lib=lib)
    ta = time.perf_counter() - t
    work = sum(vis[r] for r in rows.tolist())
    return (tw + ta * sum(vis) / work) * 1e3, len(rows), len(vis), threads


# ----------------------------------------------------------------------------- arms

def run_reference(args, world, rank):
    """The oracle as it stands, on the host cores: each step a bounded sample."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    from paged_kv_cache_287_gb300.workloads import CONFIG_NAMES, config_spec, sample_of_config

    n = args.workload
    spec = config_spec(n)
    if n == 4:
        # The mixed step's own metric: the oracle's time per step, each timed
        # step a sample of rows scaled to the whole step.
        from paged_kv_cache_287_gb300.workloads import make_config
        b = make_config(4, device="cpu")
        for _ in range(args.warmup):
            cpu_mixed_step_ms(b, stride=64)
        est, t0 = [], time.perf_counter()
        for _ in range(args.steps):
            ms, nrows, allrows, threads = cpu_mixed_step_ms(b, stride=64)
            est.append(ms)
        el = time.perf_counter() - t0
        value = sum(est) / len(est)
        sample = (f"each step: the cache write of all {int(b.cu_q_lens[-1])} new tokens and "
                  f"fp64 attention of every 64th of the {allrows} query rows ({nrows} rows), "
                  f"scaled to the whole step by causally visible (query, key) pairs")
        print(json.dumps({
            "impl": "reference", "metric": "mixed chunked-prefill + decode step",
            "value": value, "unit": "ms", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": value, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(4),
            "cpu_baseline": {"value": value, "unit": "ms", "cores": threads, "kind": "oracle",
                             "sample": sample, "wall_s": el},
            "e2e": {"value": value, "unit": "ms", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}), flush=True)
        return
    per_step = 2
    b = sample_of_config(n, per_step, device="cpu")
    lib = oracle.load()
    threads = oracle.max_threads(lib)
    kv = kv_read_bytes(b.seq_lens.tolist(), b.num_kv_heads, b.head_size)

    pool = oracle._u16(b.kv_cache).copy()

    def step():
        oracle.cache_write(pool, b.k_new, b.v_new, b.slot_mapping, lib=lib, inplace=True)
        oracle.attention(b.q, b.cu_q_lens, pool, b.block_tables, b.seq_lens, b.num_heads,
                         b.scale, lib=lib)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t
    value = kv * args.steps / el / 1e9
    sample = (f"first {per_step} of {len(spec['seq_lens'])} sequences of {CONFIG_NAMES[n]} "
              f"per step (cache write + fp64 attention, all heads)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(n),
        "seqs_per_s": per_step * args.steps / el,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def workload_config(n: int, first: int = 0):
    from paged_kv_cache_287_gb300.workloads import CONFIG_NAMES, config_spec
    s = config_spec(n)
    if first:
        s["seq_lens"] = s["seq_lens"][:first]
    return {"workload": CONFIG_NAMES[n] + (f"[:{first}]" if first else ""),
            "num_seqs": len(s["seq_lens"]),
            "num_heads": s["num_heads"], "num_kv_heads": s["num_kv_heads"],
            "head_size": s["head_size"], "block_size": s["block_size"],
            "seq_len_mean": sum(s["seq_lens"]) / len(s["seq_lens"]),
            "seq_len_max": max(s["seq_lens"]),
            "l2": "inputs larger than L2 (KV pool >> 129 MB); no flush",
            "parallelism": "replicas (one independent batch per GPU)"}


def by_workload(args, dev, stream) -> dict:
    """The other workloads of the set, measured in the same run as the headline.

    Each figure is the median of at least 50 individually event-timed calls
    (after warm-up) with the SM clocks sampled over those calls; pools larger
    than L2 need no flush, and the prefix-sharing workload (whose shared prefix
    and part of the own tokens fit in L2) is timed both cold (L2 flushed by
    writing 512 MB before every call, untimed) and warm (back to back).
    Workload 1 is launch-bound, so its figure is per step, eager and replayed
    from a CUDA graph of 20 steps.  Key "_launches": this library's kernels
    launched in these timed calls."""
    from paged_kv_cache_287_gb300 import binding
    from paged_kv_cache_287_gb300.workloads import (CONFIG_NAMES, FP8_K_SCALE, FP8_V_SCALE,
                                                    fp8_pool_of, make_config)
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        pk = json.load(f)
    hbm, tfl = float(pk["hbm_gbs"]), float(pk["bf16_tflops"])
    runs = max(50, args.median_runs)
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    launches = 0
    sc = (FP8_K_SCALE, FP8_V_SCALE)

    def timed(fn, kernels, flushed=False, warm=5):
        nonlocal launches
        for _ in range(warm):
            fn()
        with ClockSampler(dev) as clk:
            ms = median_launch_ms(fn, stream, runs, (lambda: flush_buf.zero_()) if flushed else None)
        binding.pa_error_check(stream)
        launches += kernels * runs
        return ms, clk.summary()

    def hbm_roof(alg, ms, traffic_file=None):
        a = alg / (ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": a, "peak": hbm, "unit": "GB/s", "frac": a / hbm,
                "traffic": profile_traffic(traffic_file) if traffic_file else None,
                "algorithmic_bytes_per_launch": alg, "launch_ms": ms,
                "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)"}

    def ws_for(b, n=None):
        return torch.empty(binding.pa_decode_workspace_bytes(
            b.num_seqs if n is None else n, b.num_heads, b.num_kv_heads, b.head_size),
            dtype=torch.uint8, device=dev)

    res = {}
    # 1: launch-bound tiny decode step (cache write + decode), eager and graphed.
    b = make_config(1, device=dev)
    out, ws = torch.empty_like(b.q), ws_for(b)
    max_len = b.max_seq_len  # a host value, read once (the property syncs the device)

    def step1(st=stream):
        binding.pa_cache_write(b.kv_cache, b.k_new, b.v_new, b.slot_mapping, st)
        binding.pa_decode(out, b.q, b.kv_cache, b.block_tables, b.seq_lens, max_len,
                          b.scale, ws, st)

    per_step = 1 + binding.pa_decode_cascade_kernels(b.num_seqs, b.num_heads, b.num_kv_heads,
                                                     b.head_size, b.block_size, max_len, 0)
    eager2, clk2 = timed(step1, per_step)
    # The same step as one call: pa_attention_varlen on a batch of decode tokens
    # only (no chunks) writes the new tokens, then decodes.
    wsv = torch.empty(binding.pa_attention_varlen_workspace_bytes(
        b.num_seqs, 0, b.num_heads, b.num_kv_heads, b.head_size), dtype=torch.uint8, device=dev)
    cu0 = b.cu_q_lens[:1].contiguous()

    def step1u(st=stream):
        binding.pa_attention_varlen(out, b.q, b.k_new, b.v_new, b.slot_mapping, cu0, 0, 0, 0,
                                    b.kv_cache, b.block_tables, b.seq_lens, max_len, b.scale,
                                    wsv, st)

    eager, clk = timed(step1u, per_step)
    # The same call as a C caller makes it: the argument struct filled once, one
    # foreign call per step (no Python-side checks or marshalling).
    L = binding.lib()
    cbuf = ctypes.create_string_buffer(L.pa_varlen_args_bytes())
    binding.VARLEN_ARGS.pack_into(
        cbuf, 0, out.data_ptr(), b.q.data_ptr(), b.k_new.data_ptr(), b.v_new.data_ptr(),
        b.slot_mapping.data_ptr(), cu0.data_ptr(), b.kv_cache.data_ptr(),
        b.block_tables.data_ptr(), b.seq_lens.data_ptr(), wsv.data_ptr(), wsv.numel(),
        stream.cuda_stream, b.num_seqs, 0, 0, 0, b.kv_cache.shape[0], b.block_size,
        b.num_heads, b.num_kv_heads, b.head_size, b.block_tables.shape[1], max_len, 0,
        b.scale, 1.0, 1.0)
    caddr = ctypes.addressof(cbuf)

    def step1c():
        if L.pa_attention_varlen_packed(caddr):
            raise RuntimeError("pa_attention_varlen_packed failed")

    eager_c, clk_c = timed(step1c, per_step)
    graph, cap = torch.cuda.CUDAGraph(), torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(graph, stream=cap):
        for _ in range(20):
            step1u(cap)
    torch.cuda.synchronize(dev)
    replay, clk_g = timed(graph.replay, 20 * per_step)
    res[1] = {"workload": CONFIG_NAMES[1], "value": b.num_seqs / (eager / 1e3),
              "unit": "seqs/s", "ms_per_step": eager,
              "step": "pa_attention_varlen (cache write, then decode: one call, two launches), eager",
              "two_calls": {"value": b.num_seqs / (eager2 / 1e3), "unit": "seqs/s",
                            "ms_per_step": eager2, "step": "pa_cache_write + pa_decode, eager",
                            "clocks": clk2},
              "c_abi": {"value": b.num_seqs / (eager_c / 1e3), "unit": "seqs/s",
                        "ms_per_step": eager_c,
                        "step": "pa_attention_varlen_packed with the argument struct filled "
                                "once (a C caller's cost: no Python-side checks), eager",
                        "clocks": clk_c},
              "graph": {"value": b.num_seqs / (replay / 20 / 1e3), "unit": "seqs/s",
                        "ms_per_step": replay / 20, "steps_per_replay": 20,
                        "step": "the one-call step, 20 captured in one CUDA graph",
                        "clocks": clk_g},
              "roofline": {"bound": "launch", "frac": None,
                           "note": "264 KB of KV: launch latency, not HBM, bounds the step"},
              "clocks": clk}
    del b, out, ws, wsv, graph

    # 2 (FP8 pool) and 3: decode of the Llama-3-8B batch and of the long skewed one.
    for n in (2, 3):
        b = make_config(n, device=dev)
        out, ws = torch.empty_like(b.q), ws_for(b)
        max_len = b.max_seq_len
        entry = {"workload": CONFIG_NAMES[n]}
        if n == 3:
            binding.pa_cache_write(b.kv_cache, b.k_new, b.v_new, b.slot_mapping, stream)
            ms, clk = timed(lambda: binding.pa_decode(out, b.q, b.kv_cache, b.block_tables,
                                                      b.seq_lens, max_len, b.scale, ws,
                                                      stream), 2)
            entry.update({"value": kv_read_bytes(b.seq_lens.tolist(), b.num_kv_heads,
                                                 b.head_size) / (ms / 1e3) / 1e9,
                          "unit": "GB/s", "ms_per_step": ms,
                          "seqs_per_s": b.num_seqs / (ms / 1e3), "kernel": "pa_decode",
                          "roofline": hbm_roof(decode_algorithmic_bytes(b), ms,
                                               f"decode_{b.name}.traffic.txt"), "clocks": clk})
        pool8 = fp8_pool_of(b)
        b.kv_cache = torch.empty(0, device=dev)
        torch.cuda.empty_cache()
        binding.pa_cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, *sc, stream)
        ms, clk = timed(lambda: binding.pa_decode_fp8(out, b.q, pool8, b.block_tables,
                                                      b.seq_lens, max_len, b.scale, *sc,
                                                      ws, stream), 2)
        entry["fp8"] = {"value": kv_read_bytes(b.seq_lens.tolist(), b.num_kv_heads,
                                               b.head_size) / 2 / (ms / 1e3) / 1e9,
                        "unit": "GB/s", "ms_per_step": ms, "seqs_per_s": b.num_seqs / (ms / 1e3),
                        "kernel": "pa_decode_fp8",
                        "roofline": hbm_roof(decode_algorithmic_bytes(b, 1), ms,
                                             f"decode_fp8_{b.name}.traffic.txt"), "clocks": clk}
        res[n] = entry
        del b, out, ws, pool8
        torch.cuda.empty_cache()

    # 4: the mixed step through the one call, and its prefill alone.
    b = make_config(4, device=dev)
    n_pre = int((b.q_lens > 1).sum())
    r_pre = int(b.cu_q_lens[n_pre])
    cu_pre = b.cu_q_lens[:n_pre + 1].contiguous()
    max_q, max_dec = int(b.q_lens[:n_pre].max()), int(b.seq_lens[n_pre:].max())
    out_all = torch.empty_like(b.q)
    out_pre = torch.empty_like(b.q[:r_pre])
    ws = torch.empty(binding.pa_attention_varlen_workspace_bytes(
        b.num_seqs, n_pre, b.num_heads, b.num_kv_heads, b.head_size), dtype=torch.uint8,
        device=dev)
    flops = prefill_flops(b, 0, n_pre)
    entry = {"workload": CONFIG_NAMES[4]}
    for kind in ("bf16", "fp8"):
        pool = fp8_pool_of(b) if kind == "fp8" else b.kv_cache
        kw = {"kv_scales": sc} if kind == "fp8" else {}
        step_ms, clk = timed(lambda: binding.pa_attention_varlen(
            out_all, b.q, b.k_new, b.v_new, b.slot_mapping, cu_pre, n_pre, r_pre, max_q, pool,
            b.block_tables, b.seq_lens, max_dec, b.scale, ws, stream, **kw), 3)
        if kind == "fp8":
            pre = lambda: binding.pa_prefill_chunk_fp8(out_pre, b.q[:r_pre], cu_pre, max_q, pool,
                                                       b.block_tables[:n_pre],
                                                       b.seq_lens[:n_pre], b.scale, *sc, stream)
        else:
            pre = lambda: binding.pa_prefill_chunk(out_pre, b.q[:r_pre], cu_pre, max_q, pool,
                                                   b.block_tables[:n_pre], b.seq_lens[:n_pre],
                                                   b.scale, stream)
        pre_ms, clk_p = timed(pre, 1)
        tf = flops / (pre_ms / 1e3) / 1e12
        e = {"value": step_ms, "unit": "ms", "higher_is_better": False, "ms_per_step": step_ms,
             "step": "pa_attention_varlen" + ("_fp8" if kind == "fp8" else "") +
                     ": cache write (its extra block splits the SMs), then chunked prefill "
                     "and decode side by side in one launch, then the decode's merge",
             "prefill": {"tflops": tf, "launch_ms": pre_ms, "flops_per_launch": flops,
                         "clocks": clk_p},
             "roofline": {"bound": "tensor", "achieved": tf, "peak": tfl, "unit": "TFLOP/s",
                          "frac": tf / tfl, "kernel": "pa_prefill_chunk" +
                          ("_fp8" if kind == "fp8" else ""),
                          "traffic": profile_traffic(
                              f"prefill{'_fp8' if kind == 'fp8' else ''}_{b.name}.traffic.txt"),
                          "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops)"},
             "clocks": clk}
        if kind == "fp8":
            entry["fp8"] = e
        else:
            entry.update(e)
        del pool
    res[4] = entry
    del b, out_all, out_pre, ws
    torch.cuda.empty_cache()

    # 5: prefix-shared decode, plain and cascade (bf16 and FP8 pools), cold and warm.
    b = make_config(5, device=dev)
    shared = b.shared_prefix_blocks * b.block_size
    max_len = b.max_seq_len
    out = torch.empty_like(b.q)
    ws = torch.empty(binding.pa_decode_cascade_workspace_bytes(
        b.num_seqs, b.num_heads, b.num_kv_heads, b.head_size, shared), dtype=torch.uint8,
        device=dev)
    binding.pa_cache_write(b.kv_cache, b.k_new, b.v_new, b.slot_mapping, stream)
    plain_ms, clk = timed(lambda: binding.pa_decode(out, b.q, b.kv_cache, b.block_tables,
                                                    b.seq_lens, max_len, b.scale, ws,
                                                    stream), 2, flushed=True)
    logical = kv_read_bytes(b.seq_lens.tolist(), b.num_kv_heads, b.head_size)
    entry = {"workload": CONFIG_NAMES[5],
             "plain_decode": {"value": logical / (plain_ms / 1e3) / 1e9, "unit": "GB/s (logical)",
                              "ms_per_step": plain_ms, "seqs_per_s": b.num_seqs / (plain_ms / 1e3),
                              "timing": "cold (L2 flushed before each call)", "clocks": clk}}
    pool8 = fp8_pool_of(b)
    binding.pa_cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, *sc, stream)
    for kind, pool in (("bf16", b.kv_cache), ("fp8", pool8)):
        kw = {"kv_scales": sc} if kind == "fp8" else {}
        call = lambda: binding.pa_decode_cascade(out, b.q, pool, b.block_tables, b.seq_lens,
                                                 max_len, shared, b.scale, ws, stream, **kw)
        alg = cascade_algorithmic_bytes(b, shared, 1 if kind == "fp8" else 2)
        e = {}
        for timing in ("cold", "warm"):
            ms, clk = timed(call, 2, flushed=timing == "cold")
            e[timing] = {"value": alg / (ms / 1e3) / 1e9, "unit": "GB/s (unique bytes)",
                         "ms_per_step": ms, "seqs_per_s": b.num_seqs / (ms / 1e3),
                         "roofline": hbm_roof(alg, ms, f"cascade{'_fp8' if kind == 'fp8' else ''}"
                                                       f"_{b.name}.traffic.txt"), "clocks": clk}
        c = dict(e["cold"], kernel="pa_decode_cascade" + ("_fp8" if kind == "fp8" else ""),
                 timing="cold (L2 flushed by writing 512 MB before each call)", warm=e["warm"])
        entry["cascade" if kind == "bf16" else "cascade_fp8"] = c
    entry.update({k: entry["cascade"][k] for k in ("value", "unit", "ms_per_step", "roofline",
                                                   "clocks")})
    res[5] = entry
    res["_launches"] = launches
    return res


def run_ours(args, world, rank, local):
    from paged_kv_cache_287_gb300 import binding
    from paged_kv_cache_287_gb300.workloads import make_config

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device (the library has no CPU path)")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    n = args.workload
    if n == 4:
        return run_mixed(args, world, rank, local)
    seed = None if rank == 0 else 287 + n + 7919 * rank
    if args.seqs:
        from paged_kv_cache_287_gb300.workloads import sample_of_config
        b = sample_of_config(n, args.seqs, device=dev, seed=seed)
    else:
        b = make_config(n, device=dev, seed=seed)
    binding.lib()
    stream = torch.cuda.current_stream(dev)
    out = torch.empty_like(b.q)
    fp8 = args.kv == "fp8"
    pool = b.kv_cache
    if fp8:
        from paged_kv_cache_287_gb300.workloads import FP8_K_SCALE, FP8_V_SCALE, fp8_pool_of
        pool = fp8_pool_of(b)
        b.kv_cache = torch.empty(0, device=dev)  # the bf16 pool is not read
        torch.cuda.empty_cache()
    shared = b.shared_prefix_blocks * b.block_size if args.cascade else 0
    if args.cascade and not shared:
        raise SystemExit("--cascade needs a workload whose sequences share a prefix (5)")
    if args.cascade:
        nbytes = binding.pa_decode_cascade_workspace_bytes(b.num_seqs, b.num_heads,
                                                           b.num_kv_heads, b.head_size, shared)
    else:
        nbytes = binding.pa_decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads,
                                                   b.head_size)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    max_len = b.max_seq_len

    def attend(q, tables, lens, st, dst=None):
        dst = out if dst is None else dst
        if args.cascade and fp8:
            binding.pa_decode_cascade_fp8(dst, q, pool, tables, lens, max_len, shared, b.scale,
                                          FP8_K_SCALE, FP8_V_SCALE, ws, st)
        elif args.cascade:
            binding.pa_decode_cascade(dst, q, pool, tables, lens, max_len, shared, b.scale,
                                      ws, st)
        elif fp8:
            binding.pa_decode_fp8(dst, q, pool, tables, lens, max_len, b.scale, FP8_K_SCALE,
                                  FP8_V_SCALE, ws, st)
        else:
            binding.pa_decode(dst, q, pool, tables, lens, max_len, b.scale, ws, st)

    def write(k_new, v_new, slots, st):
        if fp8:
            binding.pa_cache_write_fp8(pool, k_new, v_new, slots, FP8_K_SCALE, FP8_V_SCALE, st)
        else:
            binding.pa_cache_write(pool, k_new, v_new, slots, st)

    cu0 = b.cu_q_lens[:1].contiguous()  # no chunks: decode tokens only

    def one_call(k_new, v_new, slots, q, tables, lens, st, dst=None):
        """The step through the library's one call: the cache write, then the
        decode as a programmatic dependent of the write (its set-up overlaps it)."""
        dst = out if dst is None else dst
        kw = {"kv_scales": (FP8_K_SCALE, FP8_V_SCALE)} if fp8 else {}
        binding.pa_attention_varlen(dst, q, k_new, v_new, slots, cu0, 0, 0, 0, pool, tables,
                                    lens, max_len, b.scale, ws, st, **kw)

    def step(st=None, calls=None):
        """One step: write the new tokens, then decode.  The shared-prefix decode
        has no one-call form, so it (and calls == 2) runs the two calls."""
        st = stream if st is None else st
        if args.cascade or calls == 2:
            write(b.k_new, b.v_new, b.slot_mapping, st)
            attend(b.q, b.block_tables, b.seq_lens, st)
        else:
            one_call(b.k_new, b.v_new, b.slot_mapping, b.q, b.block_tables, b.seq_lens, st)

    for _ in range(max(args.warmup, 3)):
        step()
    binding.pa_error_check(stream)
    graph = None
    per_graph = max(1, args.graph_steps) if args.graph else 1
    if args.steps % per_graph:
        raise SystemExit("--steps must be a multiple of --graph-steps")
    if args.graph:
        # per_graph captured steps (cache write + decode kernels each) per replay;
        # several steps per replay take the host's launch of the graph off the
        # per-step time of a launch-bound workload.
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(per_graph):
                step(st=cap)
        torch.cuda.synchronize(dev)

    def timed(calls=None):
        """K steps (graph replays) between one pair of events on the stream."""
        n_rep = args.steps // per_graph if graph is not None else args.steps
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        sampler = ClockSampler(dev) if rank == 0 else None
        if sampler:
            sampler.__enter__()
        start.record(stream)
        for i in range(n_rep):
            if graph is not None:
                graph.replay()
            else:
                step(calls=calls)
        stop.record(stream)
        torch.cuda.synchronize(dev)
        if sampler:
            sampler.__exit__(None, None, None)
        barrier(world)
        return start.elapsed_time(stop), (sampler.summary() if sampler else {})

    total_ms, clocks = timed()
    if rank == 0 and rejected_clocks(clocks):
        total_ms, clocks = timed()
        clocks["remeasured"] = True
    binding.pa_error_check(stream)
    total_ms = max_over_ranks(total_ms, world, dev)
    # The same steps as the two separate calls (eager only), for comparison.
    two_calls_ms = None
    if graph is None and not args.cascade:
        for _ in range(3):
            step(calls=2)
        two_calls_ms = max_over_ranks(timed(calls=2)[0], world, dev)
    # The attention call alone: the median of individually event-timed launches
    # (the roofline's duration); the cache write's device time back to back.
    runs = max(50, args.median_runs)
    decode_med_ms = median_launch_ms(
        lambda: attend(b.q, b.block_tables, b.seq_lens, stream), stream, runs)
    write_ms = back_to_back_ms(lambda: write(b.k_new, b.v_new, b.slot_mapping, stream), stream)
    decode_ms = decode_med_ms

    # End to end: every step's inputs from pinned host memory, its output back to
    # pinned host memory.  Two buffer sets and one stream per copy direction:
    # step i+1's inputs are copied in, and step i-1's output out, while step i
    # computes (what a serving loop does with the copy engines).  One stream for
    # both directions would queue step i+1's inputs behind step i's output copy,
    # which waits for step i's kernels.
    # A step's inputs travel as one staging buffer (typed views into it), so each
    # step issues one host-to-device copy.
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "seq_lens")
    offs, total = {}, 0
    for k in names:
        t = getattr(b, k)
        offs[k] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256

    def views(buf):
        v = {}
        for k in names:
            t = getattr(b, k)
            nbytes = t.numel() * t.element_size()
            v[k] = buf[offs[k]:offs[k] + nbytes].view(t.dtype).view(t.shape)
        return v

    host_buf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for k, v in views(host_buf).items():
        v.copy_(getattr(b, k).to("cpu"))
    dev_buf = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    dev_in = [views(x) for x in dev_buf]
    dev_out = [torch.empty_like(out) for _ in range(2)]
    out_host = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(getattr(b, k).numel() * getattr(b, k).element_size() for k in names)
    d2h = out_host[0].numel() * out_host[0].element_size()
    copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    free = [torch.cuda.Event() for _ in range(2)]      # buffer set's last output copied out
    landed = [torch.cuda.Event() for _ in range(2)]    # buffer set's inputs copied in
    done = [torch.cuda.Event() for _ in range(2)]      # buffer set's step computed
    for e in free:
        e.record(copy_out)

    def e2e_step(i):
        p = i % 2
        # The buffer set is free once its previous output has been copied out
        # (which also orders this copy after that step's kernels read it).
        copy_in.wait_event(free[p])
        with torch.cuda.stream(copy_in):
            dev_buf[p].copy_(host_buf, non_blocking=True)
        landed[p].record(copy_in)
        stream.wait_event(landed[p])
        x = dev_in[p]
        if args.cascade:
            write(x["k_new"], x["v_new"], x["slot_mapping"], stream)
            attend(x["q"], x["block_tables"], x["seq_lens"], stream, dst=dev_out[p])
        else:
            one_call(x["k_new"], x["v_new"], x["slot_mapping"], x["q"], x["block_tables"],
                     x["seq_lens"], stream, dst=dev_out[p])
        done[p].record(stream)
        copy_out.wait_event(done[p])
        with torch.cuda.stream(copy_out):
            out_host[p].copy_(dev_out[p], non_blocking=True)
        free[p].record(copy_out)

    for i in range(max(args.warmup, 3)):
        e2e_step(i)
    barrier(world)
    torch.cuda.synchronize(dev)
    n_e2e = max(args.steps, args.e2e_steps)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    barrier(world)

    if rank != 0:
        return
    kv = kv_read_bytes(b.seq_lens.tolist(), b.num_kv_heads, b.head_size) // (2 if fp8 else 1)
    value = world * kv * args.steps / (total_ms / 1e3) / 1e9
    seqs_s = world * b.num_seqs * args.steps / (total_ms / 1e3)
    peak, peak_src = measured_peaks()
    alg = cascade_algorithmic_bytes(b, shared, 1 if fp8 else 2) if args.cascade else \
        decode_algorithmic_bytes(b, 1 if fp8 else 2)
    achieved = alg / (decode_med_ms / 1e3) / 1e9
    # Kernels of one attention call (the cache write is one more per step).
    attn_kernels = 2
    if args.cascade:
        attn_kernels = binding.pa_decode_cascade_kernels(b.num_seqs, b.num_heads, b.num_kv_heads,
                                                         b.head_size, b.block_size, max_len,
                                                         shared, fp8)
        kernel = (f"pa_decode_cascade{'_fp8' if fp8 else ''} ("
                  + ("prefix pass beside the own tokens' decode in one launch, then the merge "
                     "kernel" if attn_kernels == 2 else
                     "prefix pass, own tokens' decode, merge kernel") + ")")
        traffic_file = f"cascade{'_fp8' if fp8 else ''}_{b.name}.traffic.txt"
    elif fp8:
        kernel = "pa_decode_fp8 (split-context kernel + merge kernel)"
        traffic_file = f"decode_fp8_{b.name}.traffic.txt"
    else:
        kernel = "pa_decode (split-context kernel + merge kernel)"
        traffic_file = f"decode_{b.name}.traffic.txt"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16" if fp8 else "bf16",
        "data": "synthetic",
        "config": dict(workload_config(n, args.seqs),
                       launch=(f"cuda-graph, {per_graph} steps per replay" if graph else "eager"),
                       kv_cache="fp8-e4m3 (per-tensor k/v scale 1/64)" if fp8 else "bf16",
                       **({"cascade_shared_len": shared} if args.cascade else {})),
        "seqs_per_s": seqs_s,
        "hbm_frac_of_step": value / world / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profile_traffic(traffic_file),
                     "kernel": kernel,
                     "algorithmic_bytes_per_launch": alg, "launch_ms": decode_med_ms,
                     "launch_ms_how": f"median of {runs} individually event-timed launches",
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s"},
        "step": ("pa_cache_write, then " + kernel if args.cascade else
                 "pa_attention_varlen on the decode tokens: the cache write, then the decode "
                 "as its programmatic dependent (one call)"),
        "kernels_ms": {"pa_cache_write": write_ms, "pa_decode": decode_ms},
        "kernels_ms_how": "the write: 20 launches back to back per pair of events; the "
                          "decode: median of individually event-timed launches",
        **({"two_calls": {"ms_per_step": two_calls_ms / args.steps,
                          "value": world * kv * args.steps / (two_calls_ms / 1e3) / 1e9,
                          "step": "pa_cache_write + pa_decode"
                                  + ("_fp8" if fp8 else "") + ", two calls"}}
           if two_calls_ms is not None else {}),
        "e2e": {"value": world * kv * n_e2e / e2e_s / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
                "note": "KV pool resident in HBM (the cache); every step's inputs copied in "
                        "from pinned host memory and its output copied out, on one stream per "
                        "copy direction overlapping the neighbouring steps' kernels (two "
                        "buffer sets); host wall clock over all steps"},
        "clocks": clocks,
        "gpu_launches": (1 + attn_kernels) * args.steps,
    }
    if world == 1 and not args.no_cpu_baseline and not fp8:
        gbs, sps, done, k, threads = cpu_oracle_rate(n)
        gbs1, sps1, done1, _, _ = cpu_oracle_rate(n, budget_s=4.0, threads=1)
        line["cpu_baseline"] = {"value": gbs, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "seqs_per_s": sps,
                                "sample": f"{done} sequence-steps cycling over the first {k} "
                                          f"sequences of {b.name} (cache write + fp64 "
                                          f"attention, all heads, one sequence per call)",
                                "single_thread": {"value": gbs1, "unit": UNIT, "cores": 1,
                                                  "seqs_per_s": sps1,
                                                  "sample": f"{done1} sequence-steps, same "
                                                            f"sample, one thread"}}
    if (world == 1 and n == DEFAULT_WORKLOAD and not args.seqs and not args.graph
            and not args.cascade and not fp8 and not args.no_by_workload):
        # Every other workload of the set, measured in the same run on the same GPU.
        line["by_workload"] = by_workload(args, dev, stream)
        line["gpu_launches_by_workload"] = line["by_workload"].pop("_launches")
    print(json.dumps(line), flush=True)


def prefill_flops(b, lo: int, hi: int) -> int:
    """4*Hq*D per causally visible (query, key) pair: q_len*ctx + q_len*(q_len+1)/2."""
    pairs = 0
    for s in range(lo, hi):
        ql = int(b.q_lens[s])
        ctx = int(b.seq_lens[s]) - ql
        pairs += ql * ctx + ql * (ql + 1) // 2
    return 4 * b.num_heads * b.head_size * pairs


def run_mixed(args, world, rank, local):
    """Workload 4: write all new tokens, then chunked prefill of the 8 chunks and
    decode of the 248 sequences.  value = one step through the unified call;
    the three separate calls are timed per kernel alongside."""
    from paged_kv_cache_287_gb300 import binding
    from paged_kv_cache_287_gb300.workloads import make_config

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    b = make_config(4, device=dev)
    stream = torch.cuda.current_stream(dev)
    n_pre = int((b.q_lens > 1).sum())
    r_pre = int(b.cu_q_lens[n_pre])
    q_pre, q_dec = b.q[:r_pre], b.q[r_pre:]
    out_pre, out_dec = torch.empty_like(q_pre), torch.empty_like(q_dec)
    cu_pre = b.cu_q_lens[:n_pre + 1].contiguous()
    bt_pre, bt_dec = b.block_tables[:n_pre], b.block_tables[n_pre:]
    sl_pre, sl_dec = b.seq_lens[:n_pre], b.seq_lens[n_pre:]
    max_q = int(b.q_lens[:n_pre].max())
    max_dec = int(sl_dec.max())
    ws = torch.empty(binding.pa_decode_workspace_bytes(b.num_seqs - n_pre, b.num_heads,
                                                       b.num_kv_heads, b.head_size),
                     dtype=torch.uint8, device=dev)

    fp8 = args.kv == "fp8"
    if fp8:
        from paged_kv_cache_287_gb300.workloads import FP8_K_SCALE, FP8_V_SCALE, fp8_pool_of
        pool8 = fp8_pool_of(b)

    def step(ev=None):
        if ev: ev[0].record(stream)
        if fp8:
            binding.pa_cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, FP8_K_SCALE,
                                       FP8_V_SCALE, stream)
        else:
            binding.pa_cache_write(b.kv_cache, b.k_new, b.v_new, b.slot_mapping, stream)
        if ev: ev[1].record(stream)
        if fp8:
            binding.pa_prefill_chunk_fp8(out_pre, q_pre, cu_pre, max_q, pool8, bt_pre, sl_pre,
                                         b.scale, FP8_K_SCALE, FP8_V_SCALE, stream)
        else:
            binding.pa_prefill_chunk(out_pre, q_pre, cu_pre, max_q, b.kv_cache, bt_pre, sl_pre,
                                     b.scale, stream)
        if ev: ev[2].record(stream)
        if fp8:
            binding.pa_decode_fp8(out_dec, q_dec, pool8, bt_dec, sl_dec, max_dec, b.scale,
                                  FP8_K_SCALE, FP8_V_SCALE, ws, stream)
        else:
            binding.pa_decode(out_dec, q_dec, b.kv_cache, bt_dec, sl_dec, max_dec, b.scale, ws,
                              stream)
        if ev: ev[3].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    binding.pa_error_check(stream)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    with ClockSampler(dev) as sampler:
        for i in range(args.steps):
            step(evs[i])
        torch.cuda.synchronize(dev)
    binding.pa_error_check(stream)
    ms = [sum(e[j].elapsed_time(e[j + 1]) for e in evs) / args.steps for j in range(3)]

    def prefill_only():
        if fp8:
            binding.pa_prefill_chunk_fp8(out_pre, q_pre, cu_pre, max_q, pool8, bt_pre, sl_pre,
                                         b.scale, FP8_K_SCALE, FP8_V_SCALE, stream)
        else:
            binding.pa_prefill_chunk(out_pre, q_pre, cu_pre, max_q, b.kv_cache, bt_pre, sl_pre,
                                     b.scale, stream)

    # The tensor-bound kernel's roofline duration: the median of individually
    # event-timed launches.
    runs = max(50, args.median_runs)
    pre_med_ms = median_launch_ms(prefill_only, stream, runs)

    def write_only():
        if fp8:
            binding.pa_cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, FP8_K_SCALE,
                                       FP8_V_SCALE, stream)
        else:
            binding.pa_cache_write(b.kv_cache, b.k_new, b.v_new, b.slot_mapping, stream)

    write_b2b_ms = back_to_back_ms(write_only, stream)

    # The same step through the one unified call (write, chunks, decode tokens).
    out_all = torch.empty_like(b.q)
    ws_all = torch.empty(binding.pa_attention_varlen_workspace_bytes(
        b.num_seqs, n_pre, b.num_heads, b.num_kv_heads, b.head_size), dtype=torch.uint8,
        device=dev)

    def unified():
        if fp8:
            binding.pa_attention_varlen(out_all, b.q, b.k_new, b.v_new, b.slot_mapping, cu_pre,
                                        n_pre, r_pre, max_q, pool8, b.block_tables, b.seq_lens,
                                        max_dec, b.scale, ws_all, stream,
                                        kv_scales=(FP8_K_SCALE, FP8_V_SCALE))
        else:
            binding.pa_attention_varlen(out_all, b.q, b.k_new, b.v_new, b.slot_mapping, cu_pre,
                                        n_pre, r_pre, max_q, b.kv_cache, b.block_tables,
                                        b.seq_lens, max_dec, b.scale, ws_all, stream)

    for _ in range(max(args.warmup, 3)):
        unified()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(args.steps):
        unified()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    binding.pa_error_check(stream)
    unified_ms = e0.elapsed_time(e1) / args.steps
    unified_med_ms = median_launch_ms(unified, stream, runs)

    # End to end through the unified call: every step's inputs (q, new K/V, slots,
    # chunk offsets, tables, lengths) from pinned host memory in one staging
    # buffer, its output back, one stream per copy direction and two buffer sets,
    # as the decode workloads' leg; the pool stays resident.
    names = ("q", "k_new", "v_new", "slot_mapping", "cu_q_lens", "block_tables", "seq_lens")
    offs, total = {}, 0
    for k in names:
        t = getattr(b, k)
        offs[k] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256

    def views(buf):
        v = {}
        for k in names:
            t = getattr(b, k)
            v[k] = buf[offs[k]:offs[k] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        return v

    host_buf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for k, v in views(host_buf).items():
        v.copy_(getattr(b, k).to("cpu"))
    dev_buf = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    dev_in = [views(x) for x in dev_buf]
    dev_out = [torch.empty_like(b.q) for _ in range(2)]
    out_host = [torch.empty(b.q.shape, dtype=b.q.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(getattr(b, k).numel() * getattr(b, k).element_size() for k in names)
    d2h = out_host[0].numel() * out_host[0].element_size()
    copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    free = [torch.cuda.Event() for _ in range(2)]
    landed = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    for e in free:
        e.record(copy_out)

    def e2e_step(i):
        p = i % 2
        x = dev_in[p]
        copy_in.wait_event(free[p])
        with torch.cuda.stream(copy_in):
            dev_buf[p].copy_(host_buf, non_blocking=True)
        landed[p].record(copy_in)
        stream.wait_event(landed[p])
        cu = x["cu_q_lens"][:n_pre + 1]
        if fp8:
            binding.pa_attention_varlen(dev_out[p], x["q"], x["k_new"], x["v_new"],
                                        x["slot_mapping"], cu, n_pre, r_pre, max_q, pool8,
                                        x["block_tables"], x["seq_lens"], max_dec, b.scale,
                                        ws_all, stream, kv_scales=(FP8_K_SCALE, FP8_V_SCALE))
        else:
            binding.pa_attention_varlen(dev_out[p], x["q"], x["k_new"], x["v_new"],
                                        x["slot_mapping"], cu, n_pre, r_pre, max_q, b.kv_cache,
                                        x["block_tables"], x["seq_lens"], max_dec, b.scale,
                                        ws_all, stream)
        done[p].record(stream)
        copy_out.wait_event(done[p])
        with torch.cuda.stream(copy_out):
            out_host[p].copy_(dev_out[p], non_blocking=True)
        free[p].record(copy_out)

    for i in range(max(args.warmup, 3)):
        e2e_step(i)
    barrier(world)
    torch.cuda.synchronize(dev)
    n_e2e = max(args.steps, args.e2e_steps)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(time.perf_counter() - t0, world, dev) * 1e3 / n_e2e
    binding.pa_error_check(stream)
    barrier(world)
    if rank != 0:
        return
    flops = prefill_flops(b, 0, n_pre)
    kv_dec = kv_read_bytes(sl_dec.tolist(), b.num_kv_heads, b.head_size)
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        pk = json.load(f)
    pre_tflops = flops / (pre_med_ms / 1e3) / 1e12
    # bf16 rows read, pool bytes written (one byte per element in an FP8 pool)
    wbytes = 2 * b.k_new.numel() * (2 + (1 if fp8 else 2))
    line = {"metric": "mixed chunked-prefill + decode step",
            "value": unified_ms, "unit": "ms", "ms_per_step": unified_ms,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "dtype": "f16" if fp8 else "bf16", "data": "synthetic",
            "config": dict(workload_config(4),
                           kv_cache="fp8-e4m3 (per-tensor k/v scale 1/64)" if fp8 else "bf16"),
            "step": "pa_attention_varlen: cache write (one extra block of its launch chooses "
                    "the decode SMs), then chunked prefill and decode side by side in one "
                    "launch, then the decode's merge"
                    + ("; FP8 pool" if fp8 else ""),
            "kernels_ms": {"pa_cache_write": ms[0], "pa_prefill_chunk": ms[1], "pa_decode": ms[2]},
            "sequential_step_ms": sum(ms),
            "unified_ms_median": unified_med_ms,
            "prefill": {"tflops": pre_tflops, "flops_per_launch": flops,
                        "launch_ms_median": pre_med_ms,
                        "peak_tflops": pk["bf16_tflops"],
                        "frac": flops / (ms[1] / 1e3) / 1e12 / pk["bf16_tflops"]},
            "decode": {"kv_gbs": kv_dec / (2 if fp8 else 1) / (ms[2] / 1e3) / 1e9,
                       "frac": kv_dec / (2 if fp8 else 1) / (ms[2] / 1e3) / 1e9 / pk["hbm_gbs"]},
            # In the step (after the decode's 2 GB stream, L2 clean; the event
            # clock's step is about 2 us) and back to back (20 launches per event
            # pair): device time of one launch.
            "cache_write": {"gbs": wbytes / (ms[0] / 1e3) / 1e9,
                            "back_to_back_us": write_b2b_ms * 1e3,
                            "gbs_back_to_back": wbytes / (write_b2b_ms / 1e3) / 1e9,
                            "frac_back_to_back": wbytes / (write_b2b_ms / 1e3) / 1e9 /
                                                 pk["hbm_gbs"],
                            "bytes_per_launch": wbytes},
            # The tensor-bound kernel of the step, timed alone in the separate calls
            # (so against the burst bf16 peak; its f16 MMAs run at the same rate).
            "roofline": {"bound": "tensor", "achieved": pre_tflops,
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": pre_tflops / pk["bf16_tflops"],
                         "traffic": profile_traffic(
                             f"prefill{'_fp8' if fp8 else ''}_{b.name}.traffic.txt"),
                         "kernel": f"pa_prefill_chunk{'_fp8' if fp8 else ''}",
                         "algorithmic_flops_per_launch": flops, "launch_ms": pre_med_ms,
                         "launch_ms_how": f"median of {runs} individually event-timed launches",
                         "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops)"},
            "e2e": {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": n_e2e,
                    "note": "the unified call with every step's inputs copied in from pinned "
                            "host memory and its output copied out, one stream per copy "
                            "direction, two buffer sets; the KV pool resident; host wall "
                            "clock over all steps"},
            "clocks": sampler.summary(), "gpu_launches": 3 * args.steps,
            "unified_gpu_launches_per_step": 3}
    if world == 1 and not args.no_cpu_baseline and not fp8:
        est, nrows, allrows, threads = cpu_mixed_step_ms(
            type(b)(**{**b.__dict__, **{k: getattr(b, k).cpu()
                                          for k, v in b.__dict__.items()
                                          if isinstance(v, torch.Tensor)}}), stride=16)
        line["cpu_baseline"] = {"value": est, "unit": "ms", "cores": threads, "kind": "oracle",
                                "sample": f"the cache write of all new tokens and fp64 "
                                          f"attention of every 16th of the {allrows} query "
                                          f"rows ({nrows} rows), scaled to the whole step by "
                                          f"causally visible (query, key) pairs"}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="replay one CUDA-graph-captured step per timed step")
    ap.add_argument("--graph-steps", type=int, default=1,
                    help="with --graph: steps captured in one graph (replayed steps/N times)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="KV-cache element type of the decode workloads")
    ap.add_argument("--cascade", action="store_true",
                    help="shared-prefix decode (pa_decode_cascade) on a prefix-sharing workload")
    ap.add_argument("--seqs", type=int, default=0,
                    help="profile only the first N sequences of the workload (not a bench line)")
    ap.add_argument("--median-runs", type=int, default=50,
                    help="individually timed launches behind each median (at least 50)")
    ap.add_argument("--e2e-steps", type=int, default=300,
                    help="steps of the end-to-end leg (at least --steps)")
    ap.add_argument("--no-by-workload", action="store_true",
                    help="default workload only: skip the other workloads' figures")
    args = ap.parse_args(argv)
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
