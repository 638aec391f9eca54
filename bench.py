"""Benchmark: one paged GQA decode step (per-CTA workqueue + split-KV decode +
LSE merge, by the engine a calibrated policy picks) on the batch-8 bimodal
fp16 workload (Hq=32, Hkv=8, d=128, page 16, lengths half U[512, 2048] and
half U[16384, 32768], pages scattered in a pool of 1.25x the pages used),
measured as KV HBM GB/s and tokens/s.  The `budget_step` object times the
whole budgeted step (query EMAs, page summaries, scoring, selection,
compaction, append, decode) on the batch-64 bf16 workload with per-sequence
page budgets; `multi_token` and `multi_token_t32` time 4 and 32 query tokens
per sequence.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload bimodal|uniform|zipf|bucket32k|bucket64k|bucket128k|tiny]

Prints one JSON line.  `value` is algorithmic bytes (valid K/V tokens + q +
block-table entries) per step / device time per step, with inputs resident in
HBM and L2 flushed between steps (a 512 MiB memset, then its first 256 MiB
read back so the lines left in L2 are clean; both outside the timed events).
`e2e` times the host-buffer entry point (q, block table and lengths copied
in, out and lse copied back, per step).  `roofline` reports the attention
kernel alone (events bracket it inside the call) against the measured HBM
copy bandwidth.  `cpu_baseline` times the CPU oracle on a bounded sample of
the same workload.  With --impl reference the CPU oracle is the measured arm.
Under torchrun (N > 1) every rank runs an independent replica (the step does
not shard), the max time over ranks is reported and `value` sums all ranks'
bytes.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_492_b300 import workloads as W  # noqa: E402

WORKLOADS = {
    "bimodal": W.bimodal,
    "bimodal_b4": W.bimodal_b4,
    "uniform": W.uniform_lengths,
    "zipf": W.zipf_lengths,
    "bucket32k": lambda: W.bucketed_long(32768),
    "bucket64k": lambda: W.bucketed_long(65536),
    "bucket128k": lambda: W.bucketed_long(131072),
    "tiny": lambda: W.tiny()["decode"],
}
METRIC = "paged GQA decode attention: KV HBM GB/s (% of B300 peak), tokens/s"
# The nominal HBM3e figure the targets are quoted against (~8 TB/s); the
# measured copy bandwidth (MEASURED_PEAKS.json) is what the roofline uses.
NOMINAL_HBM_GBS = 8000.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


def workload_config(x: W.DecodeInputs, name: str):
    return {"workload": name, "batch": x.B, "Hq": x.Hq, "Hkv": x.Hkv, "d": x.d,
            "page_size": x.page_size, "dtype": W.DTYPE_NAMES[x.dtype],
            "seq_lens": [int(v) for v in x.seq_lens], "num_pages": x.num_pages,
            "kv_bytes_per_step": x.kv_bytes(), "algorithmic_bytes_per_step": x.algorithmic_bytes(),
            "l2": L2_NOTE,
            "parallelism": "replicas (one independent decode per GPU)"}


L2_NOTE = ("flushed between steps: a 512 MiB memset, then its first 256 MiB read back, so L2 "
           "holds clean lines of the flush buffer (none of the inputs, no write-back pending); "
           "both outside the timed events")


class L2Flush:
    """The L2 flush between timed steps.  A 512 MiB memset alone leaves L2
    full of the memset's dirty lines, which the next kernel then writes back
    to HBM while it streams its own inputs; reading back the first half of the
    buffer (long since pushed out of L2 by the second half) replaces them with
    clean lines, so the timed step starts as ncu's cache control starts a
    kernel: no input in L2, no write-back pending.  `write_only` is the
    memset alone, kept for comparison."""

    def __init__(self, torch, dev, mib=512):
        self.torch = torch
        self.buf = torch.empty(mib << 20, dtype=torch.uint8, device=dev)
        self.half = self.buf[: (mib // 2) << 20].view(torch.float32)
        self.acc = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self, write_only=False):
        self.buf.zero_()
        if not write_only:
            self.torch.sum(self.half, dim=0, out=self.acc)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_sample(x: W.DecodeInputs, heads: int = 2):
    """A bounded sample of the workload for the CPU oracle: every sequence,
    the first `heads` KV heads (with their query heads)."""
    G = x.Hq // x.Hkv
    heads = min(heads, x.Hkv)
    y = W.DecodeInputs(name=x.name + "_sample", B=x.B, Hq=heads * G, Hkv=heads, d=x.d,
                       page_size=x.page_size, dtype=x.dtype, scale=x.scale,
                       q=np.ascontiguousarray(x.q[:, : heads * G]),
                       k_pool=np.ascontiguousarray(x.k_pool[:, :heads]),
                       v_pool=np.ascontiguousarray(x.v_pool[:, :heads]),
                       block_table=x.block_table, seq_lens=x.seq_lens)
    return y


def time_oracle(x: W.DecodeInputs, steps: int, warmup: int):
    from oracle import oracle as O

    cores = len(os.sched_getaffinity(0))
    y = oracle_sample(x)
    O.decode(y, nthreads=cores)  # build + page in
    for _ in range(max(0, warmup - 1)):
        O.decode(y, nthreads=cores)
    t = []
    for _ in range(steps):
        t0 = time.perf_counter()
        O.decode(y, nthreads=cores)
        t.append(time.perf_counter() - t0)
    sec = statistics.median(t)
    # the same sample on one host thread, once
    t0 = time.perf_counter()
    O.decode(y, nthreads=1)
    sec1 = time.perf_counter() - t0
    return {"value": y.algorithmic_bytes() / sec / 1e9, "unit": "GB/s", "cores": cores,
            "single_thread": {"value": y.algorithmic_bytes() / sec1 / 1e9, "unit": "GB/s",
                              "ms_per_step": sec1 * 1e3, "cores": 1},
            "kind": "oracle", "ms_per_step": sec * 1e3,
            "tokens_per_s": x.B / sec * (y.Hkv / x.Hkv),
            "sample": f"all {x.B} sequences, KV heads 0..{y.Hkv - 1} of {x.Hkv} "
                      f"({y.algorithmic_bytes() / 1e6:.1f} MB of K/V+q+table per step), "
                      f"fp64 C oracle, {steps} timed step(s), median {sec:.2f} s"}


def run_reference(args, x, name, rank, world):
    if rank != 0:
        return
    cpu = time_oracle(x, max(1, args.steps), min(args.warmup, 3))
    line = {"impl": "reference", "metric": METRIC, "value": cpu["value"], "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": cpu["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(x, name),
            "cpu_baseline": cpu,
            "e2e": {"value": cpu["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, x, name, rank, world):
    import torch
    import torch.distributed as dist

    from paged_kv_cache_492_b300 import kv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    def dev_bits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
            torch.float16 if x.dtype == W.F16 else torch.bfloat16)

    q = dev_bits(x.q)
    k = dev_bits(x.k_pool)
    v = dev_bits(x.v_pool)
    table = torch.from_numpy(x.block_table).to(dev)
    lens = torch.from_numpy(x.seq_lens).to(dev)
    out = torch.empty((x.B, x.Hq, x.d), dtype=torch.float32, device=dev)
    lse = torch.empty((x.B, x.Hq), dtype=torch.float32, device=dev)
    flush = L2Flush(torch, dev)

    # The engine: PersistentKV's adaptive policy among this library's own
    # variants (the fused kernel's split sizes and the tensor-core engine),
    # calibrated once for the workload before any timing, as a server would
    # on first sight of a batch shape.
    policy = kv.DecodePolicy()
    cands = policy.usable(x.B, x.Hq, x.Hkv, x.d, x.max_pages)
    ws_t = kv.alloc_workspace(policy.workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages), device=dev)
    best, us = kv.kv_decode_tune(q, k, v, table, lens, x.scale, out, lse, ws_t, cands, reps=7,
                                 flush=flush.buf)
    del ws_t
    pps = {"policy": best, "fused": 0, "tensor-core": kv.KV_DECODE_TENSOR_CORE}[args.engine]
    if pps not in cands:
        raise SystemExit(f"--engine {args.engine}: not available for this shape")
    tensor_core = pps == kv.KV_DECODE_TENSOR_CORE
    ws = kv.alloc_workspace(kv.kv_decode_hostio_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages,
                                                               16, pps), device=dev)

    # host-side copies for the end-to-end (host buffers) leg
    hq = torch.from_numpy(x.q.view(np.int16).copy()).view(q.dtype).pin_memory()
    ht = torch.from_numpy(x.block_table.copy()).pin_memory()
    hl = torch.from_numpy(x.seq_lens.copy()).pin_memory()
    ho = torch.empty((x.B, x.Hq, x.d), dtype=torch.float32).pin_memory()
    hls = torch.empty((x.B, x.Hq), dtype=torch.float32).pin_memory()

    decode = kv.prepare_decode(q, k, v, table, lens, x.scale, out, lse, ws, pages_per_split=pps,
                               stream=stream)

    def step():
        rc = decode()
        if rc:
            raise kv.KVError(rc, "kv_decode")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if kv.kv_get_status(ws) != 0:
        raise SystemExit("device error during warm-up")

    n = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    evk = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evk:  # materialise the events before handing them to the library
        a.record(stream)
        b.record(stream)
    # End to end through the host-buffer entry point (inputs copied in and
    # outputs delivered to pinned host memory every step, the host waits for
    # the result), measured before the clock sampler starts: nvidia-smi's
    # driver queries delay every host-side CUDA call by ~30 us while it runs
    # and for seconds after it stops, which a host-timed loop cannot separate
    # from the library's own cost (the device-timed loops are unaffected).
    hostio = kv.prepare_decode_hostio(hq, k, v, ht, hl, x.scale, ho, hls, ws,
                                      pages_per_split=pps, stream=stream)

    def e2e_loop(count):
        t = []
        for _ in range(count):
            flush()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            if hostio():
                raise SystemExit("kv_decode_hostio failed")
            stream.synchronize()
            t.append(time.perf_counter() - t0)
        return t

    e2e_loop(5)  # warm
    e2e_quiet = e2e_loop(max(20, n))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        # the step as a user runs it: no profiling hooks inside the timed region
        queue_ahead(torch, n)
        for i in range(n):
            flush()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        # the attention kernel alone (events recorded inside the call, around it)
        queue_ahead(torch, n)
        for i in range(n):
            flush()
            kv.kv_profile_next_decode(evk[i][0], evk[i][1])
            step()
        torch.cuda.synchronize()
        # the same steps after the memset alone (its dirty lines still in L2),
        # for comparison with the flush used above
        evd = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        queue_ahead(torch, n)
        for i in range(n):
            flush(write_only=True)
            evd[i][0].record(stream)
            step()
            evd[i][1].record(stream)
        torch.cuda.synchronize()
        # the same end-to-end loop while the clocks are sampled, for reference
        e2e_t = e2e_loop(max(3, n // 2))
    clocks = clk.summary()
    if kv.kv_get_status(ws) != 0:
        raise SystemExit("device error during the timed region")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kern_ms = [a.elapsed_time(b) for a, b in evk]
    t_step = sum(step_ms) / n / 1e3
    t_kern = sum(kern_ms) / n / 1e3
    t_e2e = statistics.median(e2e_t)
    t_e2e_q = statistics.median(e2e_quiet)
    t_step, t_e2e, t_kern, t_e2e_q = max_over_ranks([t_step, t_e2e, t_kern, t_e2e_q], world, dev)
    if rank != 0:
        return
    nbytes = x.algorithmic_bytes()
    peak, peak_kind = measured_peaks()
    value = whole_job_gbs(nbytes, t_step, world)
    achieved = nbytes / t_kern / 1e9
    engine = "tensor_core" if tensor_core else "fused"
    traffic = None
    prof = os.path.join(ROOT, "profiles", f"{engine}_{name}_traffic.txt")
    if os.path.exists(prof):
        with open(prof) as f:
            tj = dict(line.split(": ", 1) for line in f.read().splitlines() if ": " in line)
        if tj.get("kernel_source_hash") == kernel_hash(engine):  # null once the kernel changed
            traffic = float(tj["dram_bytes_per_launch"])
    tname = W.DTYPE_NAMES[x.dtype].upper()
    kernel = (f"mma_attend_kernel<{tname},{x.d}>" if tensor_core
              else f"decode_kernel<{x.d},{x.Hq // x.Hkv},{tname}>")
    h2d = x.q.nbytes + x.block_table.nbytes + x.seq_lens.nbytes
    d2h = x.B * x.Hq * x.d * 4 + x.B * x.Hq * 4
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": n,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3,
        "ms_per_step_median": statistics.median(step_ms), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": W.DTYPE_NAMES[x.dtype],
        "data": "synthetic", "config": workload_config(x, name),
        "tokens_per_s": world * x.B / t_step, "kv_tokens_per_s": world * float(x.seq_lens.sum()) / t_step,
        "pct_of_peak": 100.0 * (nbytes / t_step / 1e9) / peak,
        "pct_of_nominal_peak": 100.0 * (nbytes / t_step / 1e9) / NOMINAL_HBM_GBS,
        "device_ms_per_step_incl_flush": ev[0][0].elapsed_time(ev[-1][1]) / n,
        "ms_per_step_after_memset_only_flush": statistics.mean(
            a.elapsed_time(b) for a, b in evd),
        "e2e": {"value": world * nbytes / t_e2e_q / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e_q * 1e3,
                "ms_per_step_during_clock_sampling": t_e2e * 1e3,
                "note": "host-timed, median; measured before the clock sampler starts "
                        "(nvidia-smi delays host-side CUDA calls while it samples and for "
                        "seconds after)",
                "entry": "kv_decode_hostio (pinned host q/table/lens read by one copy kernel, "
                         "out/lse written in place by the decode kernels)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "kernel": kernel,
                     "units": f"{int(x.seq_lens.sum())} K/V tokens x {2 * x.Hkv * x.d * 2} B + q "
                              "+ table entries per launch",
                     "kernel_ms": t_kern * 1e3, "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})"},
        "gpu_launches": launches_per_step(x.B, tensor_core) * n,
        "gpu_launches_note": ("per step: the tensor-core attention kernel and the split merge "
                              "kernel" if tensor_core else
                              "per step: one decode kernel (workqueue slice, split-KV decode and "
                              "LSE merge fused)") + "; a page-offset pass is added above 1024 sequences",
        "clocks": clocks,
    }
    line["config"]["engine"] = ("tensor-core engine" if tensor_core else
                                f"fused decode kernel, pages_per_split={pps} (0 = automatic)")
    line["policy"] = {"candidates_pages_per_split": cands, "us": us, "best": best,
                      "chosen": pps,
                      "note": f"0 = automatic split rule, {kv.KV_DECODE_TENSOR_CORE} = tensor-core "
                              "engine; calibrated once before timing, L2 flushed before every "
                              "calibration call as in the timed steps"}
    if not args.no_budget:
        line["multi_token"] = measure_multi(x, dev, peak)
        line["multi_token_t32"] = measure_multi(x, dev, peak, T=32)
        line["budget_step"] = measure_budget(dev, peak, peak_kind, args.budget_steps,
                                             args.budget_warmup)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(x, 3, 1)
    print(json.dumps(line), flush=True)


def max_over_ranks(values, world, device):
    """Element-wise maximum of per-rank timings over all ranks (the slowest
    replica sets the job's time); identity for one rank."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist

    t = torch.tensor(values, device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_gbs(bytes_per_replica, t_step_max, world):
    """Whole-job throughput: every replica moves bytes_per_replica per step,
    the job's step takes the slowest replica's time."""
    return world * bytes_per_replica / t_step_max / 1e9


def queue_ahead(torch, steps, ms_per_step=0.5):
    """Hold the GPU in a bounded sleep kernel while the host enqueues the
    timed steps, so that each step's events bracket device work only: a host
    call delayed past the queued flush would otherwise leave the GPU idle
    between a step's start event and its first kernel.  The sleep runs before
    the first start event and is outside every timed interval."""
    torch.cuda._sleep(int(max(2.0, steps * ms_per_step) * 1e-3 * 2.1e9))


def launches_per_step(B, tensor_core=False):
    return (2 if tensor_core else 1) + (0 if B <= 1024 else 1)


def measure_budget(dev, peak, peak_kind, steps, warmup):
    """Whole budgeted decode step on the batch-64 bf16 workload: fit to the
    budgets, then `warmup` untimed and `steps` timed steps of EMA update,
    boundary compress-or-grow, append and decode.  Each step's bytes are the
    decode's algorithmic bytes over the resident tokens after the append."""
    import torch

    from paged_kv_cache_492_b300 import budget as BG
    from paged_kv_cache_492_b300 import kv

    t0 = time.perf_counter()
    c = W.budgeted_serving()
    x = c["decode"]
    assert warmup + steps <= c["steps"], "the workload is 128 steps long"
    tdt = torch.bfloat16 if x.dtype == W.BF16 else torch.float16

    def dev_bits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(tdt)

    k = dev_bits(x.k_pool)
    v = dev_bits(x.v_pool)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)  # noqa: E731
    cfg = BG.BudgetConfig(a_fast=c["a_fast"], a_slow=c["a_slow"], n_first=c["n_first"],
                          n_last=c["n_last"], delta=c["delta"])
    dec = BG.BudgetedDecoder(k, v, i32(x.block_table), i32(x.seq_lens), i32(x.free_list),
                             i32([x.free_top]), i32(c["budget"]), x.Hq, cfg)
    dec.summarize_pages(i32(np.arange(x.num_pages)))
    toks = [tuple(dev_bits(a) for a in W.step_tokens(c["seed"], t, x.B, x.Hq, x.Hkv, x.d, x.dtype))
            for t in range(warmup + steps)]
    q0 = dev_bits(W.step_tokens(c["seed"], 0, x.B, x.Hq, x.Hkv, x.d, x.dtype)[0])
    dec.fit(q0)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()
    # the decode engine for this batch, picked as for the decode-only leg
    engine, engine_us = dec.calibrate(q0, flush=flush.buf)
    eager_steps = 24
    split_steps = 24  # further graph-replayed steps with the decode timed apart
    gw = 2            # untimed steps that replay each graph once (its first launch uploads it)
    assert warmup + gw + steps + split_steps + eager_steps <= c["steps"], \
        "the workload is 128 steps long"
    toks += [tuple(dev_bits(a) for a in W.step_tokens(c["seed"], t, x.B, x.Hq, x.Hkv, x.d, x.dtype))
             for t in range(warmup + steps, warmup + gw + steps + split_steps + eager_steps)]
    for t in range(warmup):
        dec.step(*toks[t], t)
    dec.capture()  # the steady-state step as CUDA graphs (the step; budgeting and decode apart)
    # each step's token packed as the graphs' input buffer holds it (set-up,
    # outside the timed region): it arrives in one copy per step
    packed = [dec.pack_token(*tk) for tk in toks]
    dec.step_graphed_packed(packed[warmup])
    dec.step_graphed_packed(packed[warmup + 1], between=lambda: None)
    warmup += gw
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    evk = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(split_steps)]
    lens_after = []
    torch.cuda.synchronize()
    queue_ahead(torch, steps)
    for i in range(steps):
        t = warmup + i
        flush()
        ev[i][0].record(stream)
        dec.step_graphed_packed(packed[t])
        ev[i][1].record(stream)
        lens_after.append(dec.lens.clone())
    torch.cuda.synchronize()
    # the decode part alone, on the following steps (budgeting and decode
    # replayed as two graphs with events between them)
    split_lens = []
    queue_ahead(torch, split_steps)
    for i in range(split_steps):
        t = warmup + steps + i
        flush()
        dec.step_graphed_packed(packed[t], between=evk[i][0].record)
        evk[i][1].record(stream)
        split_lens.append(dec.lens.clone())
    torch.cuda.synchronize()
    split_bytes = []
    for L in split_lens:
        Lh = L.cpu().numpy().astype(np.int64)
        split_bytes.append(int(Lh.sum()) * 2 * x.Hkv * x.d * 2 + x.B * x.Hq * x.d * 2 +
                           4 * int((-(-Lh // x.page_size)).sum()))
    # the same step issued call by call from Python on the next steps (the
    # tokens passed straight to the calls: no copies into static buffers)
    eva = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(eager_steps)]
    queue_ahead(torch, eager_steps)
    for i in range(eager_steps):
        t = warmup + steps + split_steps + i
        flush()
        eva[i][0].record(stream)
        dec.step(*toks[t], t)
        eva[i][1].record(stream)
    torch.cuda.synchronize()
    eager_ms = [a.elapsed_time(b) for a, b in eva]
    st = [dec.status()]
    if any(st):
        raise SystemExit(f"device error in the budgeted step: {st}")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    dec_ms = [a.elapsed_time(b) for a, b in evk]
    nbytes = []
    for L in lens_after:
        Lh = L.cpu().numpy().astype(np.int64)
        npg = -(-Lh // x.page_size)
        nbytes.append(int(Lh.sum()) * 2 * x.Hkv * x.d * 2 + x.B * x.Hq * x.d * 2 + 4 * int(npg.sum()))
    tot_b = float(sum(nbytes))
    t_step = sum(step_ms) / 1e3
    t_dec = sum(dec_ms) / 1e3 * steps / split_steps  # scaled to the same number of steps
    dec_b = float(sum(split_bytes)) * steps / split_steps
    return {
        "workload": "budgeted_b64_bf16 (Hq=32, Hkv=8, d=128, L~U[2048,16384], budgets U[32,256])",
        "steps_timed": steps, "warmup_steps": warmup,
        "ms_per_step": t_step / steps * 1e3, "decode_ms_per_step": t_dec / steps * 1e3,
        "issue": "the step replayed as one CUDA graph; the token's q, k and v (packed at "
                 "set-up) copied into the graph's static input buffer (one copy) inside the "
                 f"timed region; the decode part timed apart on {split_steps} further steps "
                 "(two graphs, events between them)",
        "budgeting": "one kv_budget_step launch (EMA, marks, summaries, scores, selection, "
                     "grant, compaction, append)" if dec.fused_step else "separate calls",
        "decode_engine": {"chosen": engine, "us": {str(k): v for k, v in engine_us.items()},
                          "note": f"{kv.KV_DECODE_TENSOR_CORE} = tensor-core engine, 0 = fused "
                                  "kernel; calibrated on the fitted batch, L2 flushed"},
        "eager_ms_per_step": statistics.mean(eager_ms),
        "eager_note": f"mean of {eager_steps} further steps issued call by call from Python "
                      "with the tokens passed to the calls directly (no copies)",
        "step_gbs": tot_b / t_step / 1e9, "decode_gbs": dec_b / t_dec / 1e9,
        "decode_frac_of_peak": dec_b / t_dec / 1e9 / peak, "peak_gbs": peak,
        "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
        "tokens_per_s": x.B * steps / t_step,
        "resident_kv_bytes_per_step": tot_b / steps,
        "l2": L2_NOTE,
        "setup_s": setup_s,
    }


def measure_multi(x, dev, peak, T=4, steps=10):
    """kv_attend_multi on the same batch with T query tokens per sequence
    (causal), L2 flushed between steps.  Algorithmic bytes count every K/V
    token once; the tensor-core engine serves 64 / G tokens per pass over the
    pages, and `streamed_gbs` counts the bytes of every pass (each pass reads
    the tokens its queries can see)."""
    import torch

    from paged_kv_cache_492_b300 import kv

    tdt = torch.float16 if x.dtype == W.F16 else torch.bfloat16
    rng = np.random.default_rng(123)
    qm = torch.from_numpy(W.normal_bits(rng, (x.B, T, x.Hq, x.d), x.dtype).view(np.int16)).to(
        dev).view(tdt)
    k = torch.from_numpy(np.ascontiguousarray(x.k_pool).view(np.int16)).to(dev).view(tdt)
    v = torch.from_numpy(np.ascontiguousarray(x.v_pool).view(np.int16)).to(dev).view(tdt)
    table = torch.from_numpy(x.block_table).to(dev)
    lens = torch.from_numpy(x.seq_lens).to(dev)
    out = torch.empty((x.B, T, x.Hq, x.d), dtype=torch.float32, device=dev)
    lse = torch.empty((x.B, T, x.Hq), dtype=torch.float32, device=dev)
    ws = kv.alloc_workspace(kv.kv_attend_multi_workspace_size(x.B, T, x.Hq, x.Hkv, x.d,
                                                              x.max_pages), device=dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        kv.kv_attend_multi(qm, k, v, table, lens, x.scale, out, lse, ws)
    ms = []
    for _ in range(steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        kv.kv_attend_multi(qm, k, v, table, lens, x.scale, out, lse, ws)
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    if kv.kv_get_status(ws) != 0:
        raise SystemExit("device error in kv_attend_multi")
    t = statistics.median(ms) / 1e3
    algo = x.kv_bytes() + x.B * T * x.Hq * x.d * 2 + 4 * sum(-(-int(L) // 16) for L in x.seq_lens)
    plan = multi_pass_plan(T, x.Hq // x.Hkv)
    streamed, t0 = 0, 0
    for n in plan:
        shift = T - t0 - n
        streamed += int(np.maximum(x.seq_lens.astype(np.int64) - shift, 0).sum()) * 2 * x.Hkv * x.d * 2
        t0 += n
    passes = len(plan)
    return {"T": T, "ms_per_step": t * 1e3, "tokens_per_s": x.B * T / t,
            "algorithmic_gbs": algo / t / 1e9, "algorithmic_frac_of_peak": algo / t / 1e9 / peak,
            "streamed_gbs": streamed / t / 1e9, "passes": passes,
            "pass_tokens": plan,
            "note": "tensor-core engine: passes of at most 64 rows per KV head over the pages"}


def multi_pass_plan(T, G):
    """Query tokens per pass of kv_attend_multi (the library's rule): the
    fewest passes of at most 64 rows per KV head; where G divides 16 the
    ceil(T * G / 16) row blocks are dealt out evenly (larger shares first, the
    last pass taking the remaining tokens), otherwise full passes and the rest
    last."""
    most = max(1, 64 // G)
    passes = -(-T // most)
    tpb = 16 // G if 16 % G == 0 else 0
    blocks = -(-T // tpb) if tpb else 0
    plan, t0 = [], 0
    for p in range(passes):
        n = (blocks // passes + (1 if p < blocks % passes else 0)) * tpb if tpb else most
        n = min(n, T - t0)
        plan.append(n)
        t0 += n
    return plan


def kernel_hash(engine="fused"):
    import hashlib

    h = hashlib.sha256()
    for f in ("kv_mma.cu" if engine == "tensor_core" else "kv_decode.cu", "kv_common.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_492_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="bimodal", choices=list(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-budget", action="store_true", help="skip the budgeted-step leg")
    ap.add_argument("--budget-steps", type=int, default=64)
    ap.add_argument("--budget-warmup", type=int, default=8)
    ap.add_argument("--engine", default="policy", choices=["policy", "fused", "tensor-core"],
                    help="decode engine: the calibrated choice (default), the fused decode "
                         "kernel with the automatic split, or the tensor-core engine")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.init_process_group("nccl")
    x = WORKLOADS[args.workload]()
    if args.impl == "reference":
        run_reference(args, x, args.workload, rank, world)
    else:
        run_ours(args, x, args.workload, rank, world)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
