"""Benchmark of one paged-decode step on GB300.

A step is the whole hot path over one batch: pa_reshape_and_cache (write each
sequence's newest K/V through its slot) then pa_decode (paged attention, with
split-context partitions joined by log-sum-exp when the workload uses them).

Default workload: the Llama-3-70B-shaped continuous-batching decode batch (256
sequences, 64 query / 8 KV heads, head_dim 128, block_size 32, context lengths
lognormal with median 1024 clipped to [1, 16384], fp16, 2048-token partitions),
the largest of the decode batches.  Measured in the same run and reported
under `extra_workloads`: the Llama-3-8B-shaped GQA batch (64 sequences, 32/8
heads, block_size 16, context lengths U[512,4096], fp16) and the 70B batch in
bf16.  Inputs are seeded synthetic data resident in HBM; the KV bytes read per
step (0.6-1.8 GB) exceed the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  `value` is KV GB/s: algorithmic bytes per step
(K and V of exactly the context tokens, q in and out, the block-table entries
and context lengths read, the scattered rows) over the device time per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--dtype fp16|bf16] [--impl ours|reference] [--extra NAME:DTYPE]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-decode KV GB/s (fraction of GB300 HBM peak); decode tokens/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
# layers of the model each batch is shaped after (Llama-3-8B: 32, Llama-3-70B: 80)
MODEL_LAYERS = {"llama3_8b_gqa": 32, "shared_prefix_cow": 32, "long_context": 32,
                "llama3_70b_cb": 80}
DEFAULT_WORKLOAD = "llama3_70b_cb"
# the other decode targets measured beside the default line, in the same run
DEFAULT_EXTRAS = ("llama3_8b_gqa:fp16", "llama3_70b_cb:bf16", "shared_prefix_cow:shared",
                  "shared_prefix_cow", "llama3_70b_cb:e4m3", "llama3_8b_gqa:e4m3")
DECODE_SOURCES = ("pa_decode.cu", "pa_device.cuh", "pa_tile.cuh")


def algorithmic_bytes(w) -> dict:
    """Bytes the step must move at minimum.  Decode: K and V rows of the ctx
    tokens of every (sequence, KV head), the query read and the output
    written, the block-table entries the sequences reach and the context
    lengths.  Scatter: the new K/V rows read and written and the slots."""
    import numpy as np
    s = w.elem_bytes  # cached element: 2 (fp16/bf16) or 1 (FP8)
    ctx = w.context_lens.numpy().astype(np.int64)
    kv = int(2 * ctx.sum() * w.num_kv_heads * w.head_dim * s)
    qo = 2 * w.num_seqs * w.num_q_heads * w.head_dim * 2
    tables = int(4 * ((ctx + w.block_size - 1) // w.block_size).sum() + 4 * w.num_seqs)
    T = int((w.slot_mapping.numpy() >= 0).sum())
    # K and V rows: 16-bit values read, cached elements written
    scatter = 2 * T * w.num_kv_heads * w.head_dim * (2 + s) + 8 * w.num_seqs
    out = {"kv": kv, "qo": qo, "tables": tables, "decode": kv + qo + tables,
           "scatter": scatter, "step": kv + qo + tables + scatter}
    if w.group_start is not None:
        # K/V rows of distinct physical slots: a row that several sequences
        # reach through shared blocks counts once (what a decode that reads
        # each shared block once per group must move)
        bt = w.block_tables.numpy()
        used = {}
        for i, c in enumerate(ctx):
            for lb in range(int((c + w.block_size - 1) // w.block_size)):
                b = int(bt[i, lb])
                used[b] = max(used.get(b, 0), int(min(w.block_size, c - lb * w.block_size)))
        kv_u = 2 * sum(used.values()) * w.num_kv_heads * w.head_dim * s
        out.update({"kv_unique": kv_u, "decode_unique": kv_u + qo + tables,
                    "step_unique": kv_u + qo + tables + scatter})
    return out


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """K and V of one token over all layers: 2 * layers * kv_heads * d * bytes."""
    return 2 * n_layers * n_kv_heads * head_dim * elem_bytes


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(x, pre=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, f"{pre}{k}.")
                else:
                    flat[pre[:-1]] = x
            walk(d)
            for key in ("hbm_gbs", "hbm.gbs", "hbm_gbs_burst", "hbm.burst_gbs"):
                if isinstance(flat.get(key), (int, float)):
                    return float(flat[key]), f"measured (MEASURED_PEAKS.json {key})"
            for k, v in flat.items():
                if "hbm" in k.lower() and isinstance(v, (int, float)) and v > 100:
                    return float(v), f"measured (MEASURED_PEAKS.json {k})"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


def decode_source_hash() -> str:
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        h.update(open(os.path.join(ROOT, "pagedattention_kv_cache_attention_gb300", "csrc", f),
                      "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, partition_size: int):
    """Per-launch DRAM bytes of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel source at the same
    split-context partition size."""
    path = os.path.join(ROOT, "profiles", f"pa_decode_kernel_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_src = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    m_ps = re.search(r"partition_size:\s*([0-9]+)", text)
    if not m_src or not m_tr or not m_ps or m_src.group(1) != decode_source_hash():
        return None
    if int(m_ps.group(1)) != int(partition_size):
        return None
    return int(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) >= 9:
                rows.append(p)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def max_over_ranks(x: float, dist, device) -> float:
    """Largest value of x over all ranks (every rank gets it)."""
    import torch
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, bytes_per_step: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank moves bytes_per_step per step (replicas);
    ms_per_step is the slowest rank's."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def shape_overrides(args) -> dict:
    """Workload keyword overrides from the command line (dtype and head shape)."""
    kw = {}
    if args.dtype:
        kw["dtype"] = args.dtype
    if args.head_dim:
        kw["head_dim"] = args.head_dim
    if args.q_heads:
        kw["num_q_heads"] = args.q_heads
    if args.kv_heads:
        kw["num_kv_heads"] = args.kv_heads
    return kw


def make_workload(args):
    import workloads
    kw = shape_overrides(args)
    if args.partition_size is not None:
        kw["partition_size"] = args.partition_size
    w = workloads.make(args.workload, seed=args.seed, **kw)
    if getattr(args, "kv_dtype", None) == "e4m3":
        w = workloads.to_fp8(w)
    return w


def cpu_model() -> str:
    """Name of the host CPU (lscpu's model name, else /proc/cpuinfo, else the
    machine type)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine() or "unknown"


def cpu_oracle_run(w, budget_s: float, threads: int = 0):
    """Time the oracle (scatter + fp64 decode) on a bounded sample: the first
    n sequences, n grown until one run takes a good part of the budget; when
    the whole batch is quicker than that, the run is repeated until about two
    thirds of the budget is spent.  ``threads`` = 0 uses every core this
    process may run on.
    Returns (GB/s, threads used, sample description, seconds, n)."""
    import numpy as np
    import torch

    import oracle
    fp8 = w.kv_dtype == "e4m3"
    if fp8:
        kh, vh = w.k_cache.numpy().copy(), w.v_cache.numpy().copy()
    else:
        kh = w.k_cache.view(torch.int16).numpy().view(np.uint16).copy()
        vh = w.v_cache.view(torch.int16).numpy().view(np.uint16).copy()
    # an explicit count every time: the oracle's OpenMP thread count persists
    # from one call to the next
    cores = threads if threads > 0 else len(os.sched_getaffinity(0))

    def one_run(n):
        sub = slice(0, n)
        t0 = time.perf_counter()
        if fp8:
            oracle.reshape_and_cache_fp8(w.key[sub], w.value[sub], kh, vh, w.slot_mapping[sub],
                                         w.dtype, w.k_scale, w.v_scale)
        else:
            oracle.reshape_and_cache(w.key[sub], w.value[sub], kh, vh, w.slot_mapping[sub])
        oracle.decode(w.query[sub], kh, vh, w.block_tables[sub], w.context_lens[sub], w.scale,
                      w.dtype, partition_size=w.partition_size, threads=cores,
                      kv_dtype="e4m3" if fp8 else None, k_scale=w.k_scale, v_scale=w.v_scale)
        return time.perf_counter() - t0

    n = min(w.num_seqs, 4)
    while True:
        dt = one_run(n)
        if n >= w.num_seqs or dt > budget_s / 4:
            break
        n = min(w.num_seqs, max(n + 1, int(n * min(8.0, (budget_s / 3) / max(dt, 1e-3)))))
    total, runs = dt, 1
    while n >= w.num_seqs and total < budget_s * 2 / 3 and runs < 1000:
        total += one_run(n)
        runs += 1
    ctx = w.context_lens.numpy()[:n].astype(np.int64)
    s = w.elem_bytes
    byts = (2 * ctx.sum() * w.num_kv_heads * w.head_dim * s
            + 2 * n * w.num_q_heads * w.head_dim * 2
            + 4 * ((ctx + w.block_size - 1) // w.block_size).sum() + 4 * n
            + 2 * n * w.num_kv_heads * w.head_dim * (2 + s) + 8 * n)
    sample = (f"first {n} of {w.num_seqs} sequences of {w.name} (all {w.num_q_heads} query heads, "
              f"{int(ctx.sum())} context tokens), scatter + fp64 decode, {runs} run(s) in "
              f"{total:.2f} s on {cores} thread(s)")
    return byts * runs / total / 1e9, cores, sample, total, n


def cpu_baseline(w, budget_s: float) -> dict:
    """The oracle timed on every host core and on one core (about two thirds
    and one third of the budget), with the CPU model."""
    v, cores, sample, _, _ = cpu_oracle_run(w, budget_s * 2 / 3)
    v1, _, sample1, _, _ = cpu_oracle_run(w, budget_s / 3, threads=1)
    return {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": sample, "value_1core": round(v1, 4), "sample_1core": sample1,
            "cpu_model": cpu_model()}


def run_reference(args):
    """The oracle as the reference arm, timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = make_workload(args)
    budget = 20.0 / max(1, args.steps + args.warmup)
    vals = []
    for i in range(args.warmup + args.steps):
        v, cores, sample, dt, n = cpu_oracle_run(w, max(budget, 2.0))
        if i >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic, seeded (numpy/torch CPU generators)",
        "config": {"workload": w.name, "batch": w.num_seqs, "q_heads": w.num_q_heads,
                   "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "block_size": w.block_size, "num_blocks": w.num_blocks,
                   "context_tokens": int(w.context_lens.sum()),
                   "max_context_len": w.max_context_len, "partition_size": w.partition_size,
                   "kv_dtype": w.kv_dtype or w.dtype},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_cpu_table(args):
    """The oracle on every workload at all host cores and at one core (a
    reported baseline, not a target): one JSON line per workload."""
    import workloads
    for name in workloads.NAMES:
        w = workloads.make(name, seed=args.seed)
        v, cores, sample, _, _ = cpu_oracle_run(w, args.cpu_budget * 2 / 3)
        v1, _, sample1, _, _ = cpu_oracle_run(w, args.cpu_budget / 3, threads=1)
        print(json.dumps({"op": "cpu_table", "workload": name, "dtype": w.dtype, "unit": "GB/s",
                          "all_cores": {"value": round(v, 4), "cores": cores, "sample": sample},
                          "one_core": {"value": round(v1, 4), "sample": sample1},
                          "cpu_model": cpu_model()}), flush=True)
    return 0


class Step:
    """One workload resident on the device and the calls of its decode step:
    pa_reshape_and_cache of the new tokens, then pa_decode (or their FP8
    forms, or pa_decode_shared_prefix when `shared`) with a zero-filled
    workspace allocated once."""

    def __init__(self, pa, w, dev, shared=False):
        import torch
        self.pa, self.w, self.dev = pa, w, dev
        self.fp8 = w.kv_dtype == "e4m3"
        if shared and w.group_start is None:
            raise ValueError("the shared-prefix decode needs a workload with prefix groups")
        self.shared = shared
        if shared:
            self.gs, self.pl = w.group_start.to(dev), w.prefix_lens.to(dev)
        self.kc, self.vc = w.k_cache.to(dev), w.v_cache.to(dev)
        self.key, self.value = w.key.to(dev), w.value.to(dev)
        self.sm = w.slot_mapping.to(dev)
        self.q = w.query.to(dev)
        self.bt = w.block_tables.to(dev)
        self.cl = w.context_lens.to(dev)
        self.out = torch.empty_like(self.q)
        self.maxctx = w.max_context_len
        self.ps = w.partition_size
        self.nparts = pa.pa_decode_num_partitions(self.maxctx, self.ps)
        self.ws = pa.new_decode_workspace(w.num_seqs, w.num_q_heads, w.head_dim, self.maxctx,
                                          self.ps, device=dev)

    def scatter(self, k_new, v_new, slots, st):
        w, pa = self.w, self.pa
        if self.fp8:
            pa.pa_reshape_and_cache_fp8(k_new, v_new, self.kc, self.vc, slots, w.k_scale,
                                        w.v_scale, stream=st)
        else:
            pa.pa_reshape_and_cache(k_new, v_new, self.kc, self.vc, slots, stream=st)

    def decode(self, qq, tables, lens, st, out=None, groups=None):
        """groups: (group_start, prefix_lens) on the device for the
        shared-prefix call (default: the resident copies)."""
        w, pa = self.w, self.pa
        out = self.out if out is None else out
        if self.fp8 and self.shared:
            gs, pl = groups if groups is not None else (self.gs, self.pl)
            pa.pa_decode_shared_prefix_fp8(out, qq, self.kc, self.vc, tables, lens, gs, pl,
                                           w.max_group_size, w.scale, w.k_scale, w.v_scale,
                                           self.maxctx, self.ps, workspace=self.ws, stream=st)
        elif self.fp8:
            pa.pa_decode_fp8(out, qq, self.kc, self.vc, tables, lens, w.scale, w.k_scale,
                             w.v_scale, self.maxctx, self.ps, workspace=self.ws, stream=st)
        elif self.shared:
            gs, pl = groups if groups is not None else (self.gs, self.pl)
            pa.pa_decode_shared_prefix(out, qq, self.kc, self.vc, tables, lens, gs, pl,
                                       w.max_group_size, w.scale, self.maxctx, self.ps,
                                       workspace=self.ws, stream=st)
        else:
            pa.pa_decode(out, qq, self.kc, self.vc, tables, lens, w.scale, self.maxctx,
                         self.ps, workspace=self.ws, stream=st)

    def step(self, st):
        self.scatter(self.key, self.value, self.sm, st)
        self.decode(self.q, self.bt, self.cl, st)

    def launches_per_step(self) -> int:
        """Kernels one step launches: the scatter, the decode kernel, the
        reduce kernel when the join does not run inside the decode kernel, and
        the shared-prefix kernel before the decode when sharing applies."""
        fused = self.nparts <= 32 and self.w.num_seqs * self.w.num_kv_heads <= 65536
        return (2 + (1 if self.nparts > 1 and not fused else 0)
                + (1 if self.shared and self.nparts > 1 else 0))


def time_steps(fn, K: int, stream, dev) -> float:
    """Mean ms of K back-to-back calls of fn, CUDA events only at the ends (an
    event between kernels drains the GPU and hides the launch overlap)."""
    import torch
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(K):
        fn()
    stop.record(stream)
    torch.cuda.synchronize(dev)
    return start.elapsed_time(stop) / K


def time_each(fn, K: int, stream, dev) -> float:
    """Mean ms of K calls of fn, each bracketed by CUDA events on the stream."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for i in range(K):
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def measure_extra(pa, spec: str, args, dev, stream, peak: float) -> dict:
    """Step and decode-call figures of another workload ("name:flag:..." with
    flags fp16 / bf16 for the query and cache type, e4m3 for FP8 caches,
    shared for the shared-prefix call), in the same run and on the same stream
    as the main line."""
    import torch

    import workloads
    name, *flags = spec.split(":")
    dtype = next((f for f in flags if f in ("fp16", "bf16")), None)
    shared = "shared" in flags
    w = workloads.make(name, seed=args.seed, **({"dtype": dtype} if dtype else {}))
    if "e4m3" in flags:
        w = workloads.to_fp8(w)
    ab = algorithmic_bytes(w)
    s = Step(pa, w, dev, shared=shared)
    for _ in range(args.warmup):
        s.step(stream)
    torch.cuda.synchronize(dev)
    ms = time_steps(lambda: s.step(stream), args.steps, stream, dev)
    dms = time_each(lambda: s.decode(s.q, s.bt, s.cl, stream), args.steps, stream, dev)
    if pa.pa_device_errors(stream) != 0:
        raise RuntimeError(f"device error bits raised on {spec}")
    dec_gbs = ab["decode"] / (dms * 1e-3) / 1e9
    res = {"workload": w.name, "dtype": w.dtype, "kv_dtype": w.kv_dtype or w.dtype,
           "batch": w.num_seqs,
           "partition_size": w.partition_size, "partitions": s.nparts,
           "ms_per_step": round(ms, 5),
           "value": round(ab["step"] / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "hbm_fraction": round(ab["step"] / (ms * 1e-3) / 1e9 / peak, 4),
           "decode_ms": round(dms, 5), "decode_gbs": round(dec_gbs, 2),
           "roofline_frac": round(dec_gbs / peak, 4),
           "decode_tokens_per_s": round(w.num_seqs / (ms * 1e-3), 1),
           "gpu_launches_per_step": s.launches_per_step()}
    if "kv_unique" in ab:
        # bytes of distinct slots (a shared prefix counted once per group)
        res["decode"] = (("pa_decode_shared_prefix" if shared else "pa_decode")
                         + ("_fp8" if s.fp8 else ""))
        res["unique"] = {"step_gbs": round(ab["step_unique"] / (ms * 1e-3) / 1e9, 2),
                         "hbm_fraction": round(ab["step_unique"] / (ms * 1e-3) / 1e9 / peak, 4),
                         "decode_gbs": round(ab["decode_unique"] / (dms * 1e-3) / 1e9, 2),
                         "roofline_frac": round(ab["decode_unique"] / (dms * 1e-3) / 1e9 / peak,
                                                4)}
    del s
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import numpy as np
    import torch

    import pagedattention_kv_cache_attention_gb300 as pa

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    w = make_workload(args)
    ab = algorithmic_bytes(w)
    stream = torch.cuda.current_stream(dev)
    S = Step(pa, w, dev, shared=args.shared_prefix)
    fp8 = S.fp8

    K = args.steps
    # the clock sampler starts first, so that the warm-up steps run right
    # before the timed region (no idle gap for the GPU to drop its clocks in)
    with ClockSampler(dev.index) as clk:
        for _ in range(args.warmup):
            S.step(stream)
        torch.cuda.synchronize(dev)
        if pa.pa_device_errors(stream) != 0:
            raise RuntimeError("device error bits raised during warm-up")
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        # timed region: K back-to-back steps, events only at its two ends
        step_ms = time_steps(lambda: S.step(stream), K, stream, dev)
    if dist:
        dist.barrier()
    ms_per_step = max_over_ranks(step_ms, dist, dev)
    if pa.pa_device_errors(stream) != 0:
        raise RuntimeError("device error bits raised during the timed steps")

    # the dominant kernel's own duration: the same K decode calls, each
    # bracketed by CUDA events on the launch stream
    decode_ms = time_each(lambda: S.decode(S.q, S.bt, S.cl, stream), K, stream, dev)

    # spread of the step time: 10 blocks of 5 back-to-back steps (events only
    # at block ends), and single steps after an L2 flush (a 2x-L2 memset, then
    # the step between events) -- neither enters `value`
    def pct(xs, f):
        xs = sorted(xs)
        return xs[min(len(xs) - 1, max(0, int(round(f * (len(xs) - 1)))))]

    blocks = [time_steps(lambda: S.step(stream), 5, stream, dev) for _ in range(10)]
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    flushed = []
    for _ in range(20):
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            flush.zero_()
        f0.record(stream)
        S.step(stream)
        f1.record(stream)
        torch.cuda.synchronize(dev)
        flushed.append(f0.elapsed_time(f1))
    del flush
    step_stats = {
        "blocks_of_5_ms": {"median": round(statistics.median(blocks), 5),
                           "p10": round(pct(blocks, 0.1), 5), "p90": round(pct(blocks, 0.9), 5)},
        "l2_flushed_ms": {"median": round(statistics.median(flushed), 5),
                          "p10": round(pct(flushed, 0.1), 5), "p90": round(pct(flushed, 0.9), 5)},
    }
    if pa.pa_device_errors(stream) != 0:
        raise RuntimeError("device error bits raised during the spread measurement")

    # the same step replayed from a CUDA graph (no host work per step)
    graph_ms = None
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(2):
                S.step(side)
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            S.step(torch.cuda.current_stream(dev))
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
        graph_ms = time_steps(graph.replay, K, stream, dev)
        del graph
    except RuntimeError as e:  # capture unsupported: report without the graph figure
        print(f"graph replay skipped: {e}", file=sys.stderr)
    if pa.pa_device_errors(stream) != 0:
        raise RuntimeError("device error bits raised during the decode / graph timing")

    # end to end through the public API with host buffers: per step, the
    # step's inputs go host -> device in one copy from a pinned staging buffer
    # (each input in its own 256-byte-aligned segment, as a serving loop would
    # stage them), then the step, then the output back to pinned host memory
    segs = (("q", w.query), ("key", w.key), ("value", w.value), ("sm", w.slot_mapping),
            ("bt", w.block_tables), ("cl", w.context_lens))
    if S.shared:  # the shared-prefix call also takes the step's group description
        segs += (("gs", w.group_start), ("pl", w.prefix_lens))
    offs, total = {}, 0
    for n, t in segs:
        offs[n] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    hstage = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    dstage = torch.empty(total, dtype=torch.uint8, device=dev)

    def seg_view(buf, n, t):
        nbytes = t.numel() * t.element_size()
        return buf[offs[n]:offs[n] + nbytes].view(t.dtype).view(t.shape)

    for n, t in segs:
        seg_view(hstage, n, t).copy_(t)
    dviews = [seg_view(dstage, n, t) for n, t in segs]
    dq, dkey, dval, dsm, dbt, dcl = dviews[:6]
    dgroups = tuple(dviews[6:8]) if S.shared else None
    hout = torch.empty(S.out.shape, dtype=S.out.dtype, pin_memory=True)
    h2d = total
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        dstage.copy_(hstage, non_blocking=True)
        S.scatter(dkey, dval, dsm, stream)
        S.decode(dq, dbt, dcl, stream, groups=dgroups)
        hout.copy_(S.out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_serial_ms = max_over_ranks(time_steps(e2e_step, K, stream, dev), dist, dev)

    # the same, pipelined as a serving loop runs it: two device staging
    # buffers and two outputs; on one copy stream step k's inputs go in while
    # step k - 1 computes, on another step k - 1's output comes back.  Every
    # step still moves all of its inputs in and its output out inside the
    # timed region.
    in_stream, out_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dstage2 = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    views2 = [tuple(seg_view(dstage2[b], n, t) for n, t in segs) for b in range(2)]
    out2 = [torch.empty_like(S.out) for _ in range(2)]
    hout2 = [torch.empty(S.out.shape, dtype=S.out.dtype, pin_memory=True) for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def pipelined(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(in_stream)
        for k in range(steps):
            b = k % 2
            if k >= 2:
                in_stream.wait_event(ev_done[b])      # buffer b's previous step has finished
            with torch.cuda.stream(in_stream):
                dstage2[b].copy_(hstage, non_blocking=True)
            ev_in[b].record(in_stream)
            stream.wait_event(ev_in[b])
            if k >= 2:
                stream.wait_event(ev_out[b])          # out2[b] has been read back
            q_, key_, val_, sm_, bt_, cl_ = views2[b][:6]
            S.scatter(key_, val_, sm_, stream)
            S.decode(q_, bt_, cl_, stream, out=out2[b],
                     groups=tuple(views2[b][6:8]) if S.shared else None)
            ev_done[b].record(stream)
            out_stream.wait_event(ev_done[b])
            with torch.cuda.stream(out_stream):
                hout2[b].copy_(out2[b], non_blocking=True)
            ev_out[b].record(out_stream)
        e1.record(out_stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps

    pipelined(max(2, args.warmup))
    e2e_ms = max_over_ranks(pipelined(K), dist, dev)

    peak, peak_src = hbm_peak()
    # the shared-prefix decode must move each shared row once: its roofline
    # counts distinct slots
    achieved = ab["decode_unique" if S.shared else "decode"] / (decode_ms * 1e-3) / 1e9
    value_gbs = job_throughput(world, ab["step"], ms_per_step)
    clocks = clk.summary()

    # the other decode targets, measured in the same run (rank 0, one GPU)
    extras = []
    if rank == 0 and world == 1:
        for spec in (args.extra or []):
            extras.append(measure_extra(pa, spec, args, dev, stream, peak))

    line = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu = cpu_baseline(w, args.cpu_budget)
        line = {
            "metric": METRIC,
            "value": round(value_gbs, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("f16" if w.dtype == "fp16" else "bf16") + ("+e4m3 kv" if fp8 else ""),
            "data": "synthetic: seeded N(0,1) KV pool, queries and new tokens; NaN in every "
                    "slot no sequence owns",
            "config": {"workload": w.name, "batch": w.num_seqs, "q_heads": w.num_q_heads,
                       "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                       "block_size": w.block_size, "num_blocks": w.num_blocks,
                       "context_tokens": int(w.context_lens.sum()),
                       "max_context_len": S.maxctx, "partition_size": S.ps,
                       "partitions": S.nparts, "kv_dtype": w.kv_dtype or w.dtype,
                       "accumulate": "f32",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": f"no flush: inputs larger than L2 ({ab['kv'] / 1e6:.0f} MB of KV "
                             f"read per step vs {L2_BYTES / 2**20:.0f} MiB L2)"},
            "decode_tokens_per_s": round(world * w.num_seqs / (ms_per_step * 1e-3), 1),
            # one attention layer per step; the full model has n_layers of them
            # (attention only: no projections or MLPs counted)
            "attention_only_full_model_tokens_per_s": {
                "layers": MODEL_LAYERS.get(w.name),
                "value": (round(world * w.num_seqs / (ms_per_step * 1e-3) / MODEL_LAYERS[w.name], 1)
                          if w.name in MODEL_LAYERS else None)},
            "graph_replay": None if graph_ms is None else {
                "ms_per_step": round(graph_ms, 5),
                "value": round(world * ab["step"] / (graph_ms * 1e-3) / 1e9, 2), "unit": "GB/s"},
            "hbm_fraction": round(value_gbs / world / peak, 4),
            "step_stats": step_stats,
            "bytes_per_step": ab,
            "unique": None if "kv_unique" not in ab else {
                "step_gbs": round(job_throughput(world, ab["step_unique"], ms_per_step), 2),
                "hbm_fraction": round(job_throughput(world, ab["step_unique"], ms_per_step)
                                      / world / peak, 4),
                "decode": ("pa_decode_shared_prefix" if S.shared else "pa_decode")
                          + ("_fp8" if fp8 else "")},
            "roofline": {"bound": "hbm",
                         "kernel": ("pa_decode_shared_prefix call (shared-prefix kernel + decode "
                                    "kernel; the LSE join runs in the latter), bytes of distinct "
                                    "slots" if S.shared else
                                    "pa_decode call (one decode kernel; the LSE join runs in it)"
                                    if S.launches_per_step() == 2 else
                                    "pa_decode call (decode kernel + LSE reduce kernel)")
                         + ", K event-bracketed calls after the timed steps",
                         "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         # the committed summaries profile the default launch of each
                         # workload (its own dtype and shape, 16-bit cache) and name
                         # the partition size they were taken at
                         "traffic": (profiled_traffic(w.name, S.ps) if not fp8 and not S.shared
                                     and not shape_overrides(args) else None),
                         "peak_source": peak_src,
                         "decode_ms": round(decode_ms, 5)},
            "cpu_baseline": cpu,
            # the faster of the two serving loops (both move every step's
            # inputs in and its output out inside the timed region)
            "e2e": {"value": round(job_throughput(world, ab["step"], min(e2e_ms, e2e_serial_ms)), 2),
                    "unit": "GB/s", "ms_per_step": round(min(e2e_ms, e2e_serial_ms), 5),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "mode": "pipelined" if e2e_ms <= e2e_serial_ms else "serial",
                    "pipelined": {"value": round(job_throughput(world, ab["step"], e2e_ms), 2),
                                  "ms_per_step": round(e2e_ms, 5),
                                  "mode": "step k's inputs copied in and step k-1's output copied "
                                          "out while step k-1 / k compute (two staging buffers, "
                                          "two copy streams)"},
                    "serial": {"value": round(job_throughput(world, ab["step"], e2e_serial_ms), 2),
                               "ms_per_step": round(e2e_serial_ms, 5),
                               "mode": "copy in, step, copy out, all on one stream"}},
            "gpu_launches": S.launches_per_step() * K,
            "clocks": clocks,
            "extra_workloads": extras,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_block_ops(args):
    """Bandwidth of the whole-block moves on the workload's pool: a
    copy-on-write fork of many blocks (pa_copy_blocks, both caches) and a swap
    of the first quarter of the sequences to a pinned host pool and back
    (pa_swap_blocks, both caches).  Bytes = blocks x block bytes x 2 (read and
    write) x 2 caches."""
    import numpy as np
    import torch

    import pagedattention_kv_cache_attention_gb300 as pa
    dev = torch.device("cuda", 0)
    w = make_workload(args)
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    block_bytes = kc[0].numel() * kc.element_size()
    rng = np.random.default_rng(args.seed)
    K = args.steps
    res = {}

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / K

    n = min(4096, w.num_blocks // 2)
    ids = rng.permutation(w.num_blocks)
    m = torch.from_numpy(np.stack([ids[:n], ids[n:2 * n]], 1).astype(np.int64)).to(dev)
    ms = timed(lambda: pa.pa_copy_blocks(kc, vc, m))
    res["copy_blocks"] = {"blocks": n, "ms": round(ms, 5),
                          "GBps": round(4 * n * block_bytes / (ms * 1e-3) / 1e9, 1)}
    nblk = w.blocks_used()
    victims = np.concatenate([w.block_tables[i, :int(nblk[i])].numpy()
                              for i in range(max(1, w.num_seqs // 4))]).astype(np.int64)
    nv = len(victims)
    hk = torch.empty((nv,) + tuple(kc.shape[1:]), dtype=kc.dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    out_m = torch.from_numpy(np.stack([victims, np.arange(nv)], 1)).to(dev)
    in_m = torch.from_numpy(np.stack([np.arange(nv), victims], 1)).to(dev)

    def swap_out():
        pa.pa_swap_blocks(kc, hk, out_m)
        pa.pa_swap_blocks(vc, hv, out_m)

    def swap_in():
        pa.pa_swap_blocks(hk, kc, in_m)
        pa.pa_swap_blocks(hv, vc, in_m)
    for nm, fn in (("swap_out", swap_out), ("swap_in", swap_in)):
        ms = timed(fn)
        res[nm] = {"blocks": nv, "ms": round(ms, 5),
                   "GBps": round(2 * nv * block_bytes / (ms * 1e-3) / 1e9, 1),
                   "note": "GB/s counts each byte once (one side is host memory)"}
    if pa.pa_device_errors() != 0:
        raise RuntimeError("device error bits raised")
    print(json.dumps({"op": "block_moves", "workload": w.name, "block_bytes": block_bytes,
                      "steps": K, "results": res}), flush=True)
    return 0


def prefill_flops(pw) -> int:
    """Useful FLOPs of causal chunked prefill: each (row, query head) attends to
    pos + 1 keys at 4 d FLOPs per key (QK^T and P.V)."""
    import numpy as np
    ctx = pw.context_lens.numpy().astype(np.int64)
    ql = pw.q_lens.numpy().astype(np.int64)
    # sum over t < q of (ctx - q + t + 1) = q (ctx - q + 1) + q (q - 1) / 2
    keys = (ql * (ctx - ql + 1) + ql * (ql - 1) // 2).sum()
    return int(4 * pw.head_dim * pw.num_q_heads * keys)


def run_prefill(args):
    """Chunked-prefill throughput: scatter of the chunk tokens then pa_prefill."""
    import torch

    import pagedattention_kv_cache_attention_gb300 as pa
    import workloads
    dev = torch.device("cuda", 0)
    pw = workloads.make_prefill(args.workload, seed=args.seed, chunk=args.chunk,
                                **shape_overrides(args))
    fp8 = args.kv_dtype == "e4m3"
    if fp8:
        pw = workloads.to_fp8(pw)
    kc, vc = pw.k_cache.to(dev), pw.v_cache.to(dev)
    key, value, sm = pw.key.to(dev), pw.value.to(dev), pw.slot_mapping.to(dev)
    q, qs = pw.query.to(dev), pw.query_start.to(dev)
    bt, cl = pw.block_tables.to(dev), pw.context_lens.to(dev)
    out = torch.empty_like(q)
    if fp8:
        pa.pa_reshape_and_cache_fp8(key, value, kc, vc, sm, pw.k_scale, pw.v_scale)
    else:
        pa.pa_reshape_and_cache(key, value, kc, vc, sm)

    def call():
        if fp8:
            pa.pa_prefill_fp8(out, q, qs, kc, vc, bt, cl, pw.scale, pw.k_scale, pw.v_scale,
                              pw.max_q_len)
        else:
            pa.pa_prefill(out, q, qs, kc, vc, bt, cl, pw.scale, pw.max_q_len)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    if pa.pa_device_errors() != 0:
        raise RuntimeError("device error bits raised")
    fl = prefill_flops(pw)
    print(json.dumps({"op": "prefill", "workload": pw.name, "chunk": args.chunk,
                      "seqs": pw.num_seqs, "total_q": pw.total_q, "dtype": pw.dtype,
                      "kv_dtype": pw.kv_dtype or pw.dtype,
                      "head_dim": pw.head_dim, "group": pw.num_q_heads // pw.num_kv_heads,
                      "ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 2),
                      "tokens_per_s": round(pw.total_q / (ms * 1e-3), 1)}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--dtype", choices=("fp16", "bf16"), default=None)
    ap.add_argument("--kv-dtype", choices=("same", "e4m3"), default="same",
                    help="e4m3: FP8 KV cache (16-bit queries)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--partition-size", type=int, default=None,
                    help="override the workload's split-context partition (tokens, 0 = none)")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of host time for the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", choices=("step", "blocks", "prefill", "cpu-table"), default="step",
                    help="step: the decode step (default); blocks: copy/swap block bandwidth; "
                         "prefill: chunked-prefill attention; cpu-table: the oracle on every "
                         "workload at all cores and one core")
    ap.add_argument("--extra", action="append", default=None, metavar="NAME[:DTYPE][:shared]",
                    help="another workload measured in the same run (repeatable); default: "
                         + ", ".join(DEFAULT_EXTRAS) + " beside the default workload")
    ap.add_argument("--no-extra", action="store_true", help="measure the main workload only")
    ap.add_argument("--shared-prefix", action="store_true",
                    help="decode with pa_decode_shared_prefix (workloads with prefix groups)")
    ap.add_argument("--chunk", type=int, default=512, help="prefill chunk (tokens)")
    ap.add_argument("--head-dim", type=int, default=None, help="override the workload's head_dim")
    ap.add_argument("--q-heads", type=int, default=None, help="override the query head count")
    ap.add_argument("--kv-heads", type=int, default=None, help="override the KV head count")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.no_extra:
        args.extra = []
    elif args.extra is None:
        plain = (args.workload == DEFAULT_WORKLOAD and not shape_overrides(args)
                 and args.partition_size is None and args.kv_dtype == "same"
                 and not args.shared_prefix)
        args.extra = list(DEFAULT_EXTRAS) if plain else []
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "cpu-table":
        return run_cpu_table(args)
    if args.op == "blocks":
        return run_block_ops(args)
    if args.op == "prefill":
        return run_prefill(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
