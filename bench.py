#!/usr/bin/env python3
"""Throughput of QSA gather-GQA sparse attention over a ragged, paged KV cache.

A step is one call of the whole hot path (row -> sequence lookup, selection
read, page translation, K/V gather, online softmax, split-K combine, output)
over one batch of the bf16 chunked-prefill workload: 4 sequences with
[512, 1024, 256, 2048] new rows on cached lengths [0, 4096, 16384, 8192], 64
query heads on 8 kv heads, head_dim 128, page 64, selection width 2048 (the
64 positions nearest each row plus distinct uniform picks of the rest).
Inputs are synthetic and seeded.  Each step attends 55.6 M (key, kv head)
pairs, 28.6 GB of algorithmic K/V bytes over a 133 MB cache, so most gathers
are L2 hits; the roofline line is therefore the tensor (flop) bound, with the
DRAM fraction beside it.  L2 is flushed before every timed step: a 2x-L2
buffer is written, then a second 2x-L2 buffer is read, so neither the
workload nor dirty flush lines sit in L2 when the timed call starts.
``--workload`` picks any other workload (bf16_decode, fp8_mixed, ...).

One JSON line on stdout (rank 0).  ``--impl reference`` times the float64 CPU
oracle on a bounded sample of the same workload instead, on every host core.
Under torchrun each rank runs its own replica (the op shards with no
exchange), timings are max-reduced and ``value`` is the aggregate over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse attn query-tokens/s per layer; effective HBM GB/s (% of GB300 peak)"
UNIT = "query-tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
NOMINAL_HBM_GBS = 8000.0
# Fixed costs of one call of the per-(row, kv head) kernel, measured on a
# GB300 with CUDA events and a per-CTA globaltimer trace of the long-context
# decode launch: an empty kernel of the same grid, the three dependent trips
# to memory before the first gathered byte (row search with counts and Q,
# the band's list entries, the page-table entries), and the cluster merge of
# split bands.  With the algorithmic bytes at the copy peak they give the
# floor a call of that kernel cannot beat.
EMPTY_LAUNCH_US = 4.1
DEPENDENT_TRIPS_US = 4.3
CLUSTER_MERGE_US = 1.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="bf16_chunked_prefill")
    ap.add_argument("--kernel", type=int, default=0, help="force 1 CUDA-core, 2 per-(row, kv head), 3 stream-K or 4 row-group kernel")
    ap.add_argument("--splits", type=int, default=0, help="kernel 2: force CTAs per (row, kv head)")
    ap.add_argument("--ctas", type=int, default=0, help="kernel 3: force the persistent grid size")
    ap.add_argument("--heads-per-unit", type=int, default=0, help="kernel 3: force the kv heads per unit")
    ap.add_argument("--tcgen05", type=int, default=0, help="kernel 2: 1 the tcgen05 consumer, -1 mma.sync")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle time budget of the CPU baseline")
    ap.add_argument("--cpu-threads", type=int, default=0, help="oracle threads (0: every core this process may use)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--min-warmup-s", type=float, default=1.0,
                    help="keep warming up at least this long (0 for profiler runs)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def measured_peaks() -> dict:
    """Roofline denominators: MEASURED_PEAKS.json (measured copy
    bandwidth and cuBLAS bf16 rates) when present, else the fallbacks."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk["bf16_tflops_sustained"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED, "source": "fallback"}


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def roofline(x, ms: float, kernel: str, traffic) -> dict:
    """The roofline entry of the dominant kernel.

    Algorithmic bytes: every attended K and V row once per (row, kv head),
    plus q, output, indices and counts.  Algorithmic flops: 4 * group *
    head_dim per attended (key, kv head) pair (q.K and p.V).  When the
    attended K/V bytes exceed twice the distinct K/V bytes the selections
    name, the repeats are L2 hits and HBM does not bound the call: the line
    is then the tensor bound (bf16 sustained rate; FP8 runs q.K at twice that
    rate and p.V at the f16 rate, so 4/3 of it), with the DRAM fraction (from
    the recorded traffic) beside it.  Otherwise it is the HBM bound."""
    pk = measured_peaks()
    t = ms / 1e3
    alg = x.algorithmic_bytes()
    eff_gbs = alg / t / 1e9
    dram = None
    if traffic:
        dram = {"achieved": traffic / t / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": traffic / t / 1e9 / pk["hbm_gbs"], "traffic": traffic}
    pairs = x.attended_pairs()
    kv_alg = pairs * 2 * x.head_dim * (1 if x.dtype == "e4m3" else 2 if x.dtype == "bf16" else 4)
    distinct = x.distinct_kv_bytes()
    reuse = kv_alg / distinct if distinct else 1.0
    common = {"kernel": kernel, "traffic": traffic, "algorithmic_bytes_per_launch": alg,
              "l2_reuse": reuse, "effective_gbs": eff_gbs, "dram": dram}
    if reuse >= 2.0 and x.dtype in ("bf16", "e4m3"):
        flops = 4 * x.group * x.head_dim * pairs
        peak = pk["bf16_tflops_sustained"] * (4.0 / 3.0 if x.dtype == "e4m3" else 1.0)
        ach = flops / t / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                "peak_source": f"{pk['source']} (MEASURED_PEAKS bf16_tflops_sustained"
                               f"{' x 4/3: fp8 q.K at 2x, p.V at 1x' if x.dtype == 'e4m3' else ''})",
                "flops_per_launch": flops, **common}
    return {"bound": "hbm", "achieved": eff_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": eff_gbs / pk["hbm_gbs"],
            "peak_source": f"{pk['source']} (MEASURED_PEAKS hbm_gbs copy)", **common}


def latency_floor(x, ms: float, splits: int) -> dict:
    """Floor of a per-(row, kv head) kernel call: launch + three dependent
    trips + the algorithmic bytes at the measured copy peak (+ the merge when
    bands are split), beside the measured time."""
    pk = measured_peaks()
    hbm_us = x.algorithmic_bytes() / (pk["hbm_gbs"] * 1e3)
    fixed = EMPTY_LAUNCH_US + DEPENDENT_TRIPS_US + (CLUSTER_MERGE_US if splits > 1 else 0.0)
    floor = fixed + hbm_us
    return {"floor_us": floor, "fixed_us": fixed, "bytes_at_copy_peak_us": hbm_us, "time_us": ms * 1e3,
            "frac_of_floor": floor / (ms * 1e3)}


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments, blank lines and runs of spaces
    (string and character literals kept), so comment and layout edits do not
    change the hash."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(" ".join(l.split()) for l in "".join(out).splitlines() if l.strip())


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (comments ignored): recorded ncu
    traffic is reported only while it matches."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "index_gathered_sparse_gb300", "csrc")
    for n in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, n), encoding="utf-8") as f:
            h.update(n.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current kernel sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        e = rec.get(workload)
        if e and e.get("kernel_hash") == kernel_source_hash():
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        cmd = ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.p = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def replica_spec(name: str, rank: int, world: int):
    """The workload one rank runs: every rank gets its own seeded batch."""
    from index_gathered_sparse_gb300 import workloads as wl

    spec = (wl.WORKLOADS.get(name) or wl.MSA_WORKLOADS.get(name) or wl.LATENT_WORKLOADS[name])()
    if world > 1:
        spec.seed += 100 * rank
    return spec


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of each rank's ``x`` (identity on one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(rows_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job query-tokens/s: every rank's rows over the slowest rank's step."""
    return world * rows_per_rank / (ms_per_step / 1e3)


def sample_rows(total_q: int):
    """A fixed spread of rows used by the CPU measurements."""
    import numpy as np

    order = np.random.default_rng(123).permutation(total_q)
    return order.astype(np.int64)


def is_block_sparse(x) -> bool:
    return getattr(x, "d_indices", None) is not None


def is_latent(x) -> bool:
    return getattr(x, "comp_indices", None) is not None


def oracle_fn(x):
    """The oracle function for ``x``: token lists, block lists or latent
    (window + compressed entries + sinks)."""
    import oracle

    if is_latent(x):
        return oracle.latent_attention
    return oracle.msa_attention if is_block_sparse(x) else oracle.sparse_attention


def cpu_oracle_rate(x, seconds: float, threads: int = 1):
    """Rows per second of the float64 oracle on this host: ``threads``
    threads each take the next sampled row until ``seconds`` have passed
    (the C oracle runs outside the interpreter lock, so the threads run on
    separate cores).  Returns (rate, rows done, elapsed seconds)."""
    import itertools
    from concurrent.futures import ThreadPoolExecutor

    run = oracle_fn(x)
    rows = sample_rows(x.total_q)
    ticket = itertools.count()
    t0 = time.perf_counter()
    stop = t0 + seconds

    def worker():
        done = 0
        while time.perf_counter() < stop:
            k = next(ticket) % rows.size
            run(x, rows[k:k + 1])
            done += 1
        return done

    with ThreadPoolExecutor(max_workers=threads) as ex:
        futs = [ex.submit(worker) for _ in range(threads)]
        done = sum(f.result() for f in futs)
    el = time.perf_counter() - t0
    return done / el, done, el


def cpu_baseline(x, seconds: float, threads: int) -> dict:
    """The oracle timed on the host cores: every core (the reported value)
    and one thread beside it, on sampled rows of the same workload."""
    one_s = max(1.0, seconds / 4)
    r1, n1, e1 = cpu_oracle_rate(x, one_s, 1)
    rn, nn, en = cpu_oracle_rate(x, max(1.0, seconds - one_s), threads)
    return {"value": rn, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{nn} query rows of {x.name} (all heads, full selections) in {en:.1f}s on {threads} "
                      f"threads; one thread: {n1} rows in {e1:.1f}s",
            "one_thread": {"value": r1, "unit": UNIT, "cores": 1}}


def run_reference(args, x, rank, world):
    """The reference arm: the float64 CPU oracle timed on every host core."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    if rank != 0:
        return
    oracle.build()
    run = oracle_fn(x)
    rows = sample_rows(x.total_q)
    threads = args.cpu_threads or host_cores()
    t0 = time.perf_counter()
    run(x, rows[:1])
    per_row = time.perf_counter() - t0
    # a step is about half a second of all-core work
    rows_per_step = max(threads, int(round(0.5 * threads / max(per_row, 1e-6))))
    k = 0
    ex = ThreadPoolExecutor(max_workers=threads)

    def step():
        nonlocal k
        sel = np.take(rows, np.arange(k, k + rows_per_step), mode="wrap")
        list(ex.map(lambda r: run(x, sel[r:r + 1]), range(sel.size)))
        k += rows_per_step

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    ex.shutdown()
    value = rows_per_step * args.steps / el
    sample = (f"{rows_per_step} query row(s) of the {x.name} workload per step (all heads, full selections), "
              f"one row per oracle call on {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy)", "config": workload_config(x),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(x) -> dict:
    if is_latent(x):
        cfg = workload_config(x.swa)
        cfg.update({"workload": x.name, "selection": "sliding window + listed compressed entries + per-head sinks",
                    "window": x.window, "num_comp": int(x.comp_indices.shape[1]), "num_kv_heads": 1,
                    "group": x.num_heads, "comp_page_size": x.comp.kv_shape[3],
                    "selection_width": x.window + int(x.comp_indices.shape[1])})
        return cfg
    cfg = {
        "workload": x.name, "batch": x.batch, "total_q": x.total_q, "num_q_heads": x.num_q_heads,
        "num_kv_heads": x.num_kv_heads, "group": x.group, "head_dim": x.head_dim, "page_size": x.kv_shape[3],
        "num_layers": x.kv_shape[2], "layer_idx": x.layer_idx, "selection_width": x.selection_width,
        "cache_dtype": x.dtype, "out_dtype": x.out_dtype,
        "l2": "flushed before every timed step (2x L2 buffer written, then a second 2x L2 buffer read)",
    }
    if is_block_sparse(x):
        cfg.update({"selection": "blocks (d_indices [num_kv_heads, total_q, topk])", "topk": x.topk,
                    "selection_width": x.topk * x.kv_shape[3]})
    return cfg


def run_compress(args, spec, rank, world, local):
    """Block-key compression (QSACompressKeysPaged) on the GPU or, for the
    reference arm, in the float64 oracle on one host core."""
    from index_gathered_sparse_gb300 import workloads as wl

    x = spec.build()
    metric, unit = "block-key compression rows/s; effective HBM GB/s", "block-key rows/s"
    rows = x.batch * x.max_blocks
    cfg = {"workload": x.name, "batch": x.batch, "max_blocks": x.max_blocks, "head_dim": x.head_dim,
           "ratio": x.ratio, "rotary_dim": x.rotary_dim, "page_size": x.cache.kv_shape[3], "dtype": x.dtype,
           "raw_keys": int(x.key_counts.clip(0).sum()),
           "l2": "flushed before every timed step (2x L2 buffer written, then a second 2x L2 buffer read)"}
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle

        oracle.build()
        oracle.compress_keys(x)
        t0 = time.perf_counter()
        for _ in range(max(1, min(args.steps, 3))):
            oracle.compress_keys(x)
        n = max(1, min(args.steps, 3))
        el = (time.perf_counter() - t0) / n
        line = {"impl": "reference", "metric": metric, "value": rows / el, "unit": unit, "n_gpus": world,
                "steps": n, "warmup": 1, "ms_per_step": el * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy)", "config": cfg,
                "cpu_baseline": {"value": rows / el, "unit": unit, "cores": 1, "kind": "oracle",
                                 "sample": f"the whole {x.name} call per step"},
                "e2e": {"value": rows / el, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    import torch

    from index_gathered_sparse_gb300 import binding as B
    from index_gathered_sparse_gb300 import build as libbuild

    libbuild.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    d = wl.to_torch_compress(x, dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(None)
    t0, n_warm = time.perf_counter(), 0
    while n_warm < max(3, args.warmup) or time.perf_counter() - t0 < args.min_warmup_s:
        flush_w.fill_(n_warm & 0xFF)
        flush_r.sum()
        B.qsa_compress_keys_paged(**d)
        n_warm += 1
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush_w.fill_(i & 0xFF)
        flush_r.sum()
        ev[i][0].record(stream)
        B.qsa_compress_keys_paged(**d)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    per_step = [a.elapsed_time(b) for a, b in ev]
    clocks = sampler.stop()
    ms = sum(per_step) / args.steps
    flags = B.qsa_read_device_status(clear=True)
    alg = x.algorithmic_bytes()
    pk = measured_peaks()
    peak, peak_src = pk["hbm_gbs"], pk["source"]
    achieved = alg / (ms / 1e3) / 1e9
    # end to end: counts and page table in from pinned memory, block keys back
    host = {k: d[k].cpu().pin_memory() for k in ("key_counts", "cache_lengths", "kv_lookup_table")}
    out_host = torch.empty(d["block_keys"].shape, dtype=d["block_keys"].dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(3, min(args.steps, 20))
    e0.record(stream)
    for _ in range(n_e2e):
        for k, t in host.items():
            d[k].copy_(t, non_blocking=True)
        B.qsa_compress_keys_paged(**d)
        out_host.copy_(d["block_keys"], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    te = e0.elapsed_time(e1) / n_e2e
    cpu = None
    if not args.no_cpu_baseline:
        import oracle

        oracle.build()
        t1 = time.perf_counter()
        oracle.compress_keys(x)
        el = time.perf_counter() - t1
        cpu = {"value": rows / el, "unit": unit, "cores": 1, "kind": "oracle",
               "sample": f"the whole {x.name} call ({rows} rows) in {el:.1f}s, one thread"}
    line = {
        "metric": metric, "value": rows / (ms / 1e3), "unit": unit, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": sorted(per_step)[len(per_step) // 2],
        "ms_per_step_min": min(per_step), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": x.dtype, "data": "synthetic (seeded numpy)", "config": cfg, "effective_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": recorded_traffic(x.name), "peak_source": f"{peak_src} (MEASURED_PEAKS hbm_gbs copy)",
                     "kernel": "qsa compress_kernel", "algorithmic_bytes_per_launch": alg},
        "cpu_baseline": cpu,
        "e2e": {"value": rows / (te / 1e3), "unit": unit,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host.values()),
                "d2h_bytes_per_step": out_host.numel() * out_host.element_size(), "steps": n_e2e},
        "gpu_launches": args.steps, "clocks": clocks, "device_status": flags,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    from index_gathered_sparse_gb300 import workloads as wl

    if args.workload in wl.COMPRESS_WORKLOADS:
        spec = wl.COMPRESS_WORKLOADS[args.workload]()
        if world > 1:
            spec.seed += 100 * rank
        run_compress(args, spec, rank, world, local)
        return
    import numpy as np  # noqa: F401

    from index_gathered_sparse_gb300 import workloads as wl

    spec = replica_spec(args.workload, rank, world)
    t_gen = time.perf_counter()
    x = spec.build()
    print(f"[bench] rank {rank}: built {x.name} in {time.perf_counter() - t_gen:.1f}s", file=sys.stderr)

    if args.impl == "reference":
        run_reference(args, x, rank, world)
        return

    import torch

    from index_gathered_sparse_gb300 import binding as B
    from index_gathered_sparse_gb300 import build as libbuild

    libbuild.build()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    blocks, latent = is_block_sparse(x), is_latent(x)
    d = wl.to_torch_latent(x, dev) if latent else wl.to_torch_msa(x, dev) if blocks else wl.to_torch(x, dev)
    code = {"f32": B.QSA_F32, "bf16": B.QSA_BF16, "e4m3": B.QSA_F8E4M3}[x.dtype]
    if latent:  # groups of up to 16 query heads on the one latent head
        lg = min(x.num_heads, 16)
        plan = B.qsa_plan(code, x.total_q, x.num_heads // lg, 128, x.window + x.comp_indices.shape[1], lg,
                          kernel=2, splits=args.splits)
    else:
        width = x.topk * x.kv_shape[3] if blocks else x.selection_width
        extents = {} if blocks else dict(batch=x.batch, page_size=x.kv_shape[3],
                                         max_prompt_length=x.max_prompt_length, max_cache_length=x.max_cache_length)
        plan = B.qsa_plan(code, x.total_q, x.num_kv_heads, x.head_dim, width, x.group,
                          kernel=2 if blocks else args.kernel, splits=args.splits, ctas=args.ctas, block_lists=blocks,
                          heads_per_unit=0 if blocks else args.heads_per_unit, tcgen05=args.tcgen05, **extents)
    B.qsa_reserve_workspace(plan["workspace_bytes"])
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    class _Flush:
        """Writes a 2xL2 buffer, then reads a second 2xL2 buffer, so L2 holds
        none of the workload and no dirty flush lines are written back inside
        the timed region."""

        def fill_(self, v):
            flush_w.fill_(v)
            flush_r.sum()

    flush_buf = _Flush()

    def call(dd=d):
        if latent:
            B.qsa_latent_attention_ragged_paged(**dd, splits=args.splits)
        elif blocks:
            B.qsa_msa_attention_ragged_paged(**dd, splits=args.splits, tcgen05=args.tcgen05)
        else:
            B.qsa_sparse_attention_ragged_paged(**dd, kernel=args.kernel, splits=args.splits, ctas=args.ctas,
                                                heads_per_unit=args.heads_per_unit, tcgen05=args.tcgen05)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    # warm-up: at least W steps and at least ~1 s so the clock samples see load
    t0 = time.perf_counter()
    n_warm = 0
    while n_warm < max(3, args.warmup) or time.perf_counter() - t0 < args.min_warmup_s:
        flush_buf.fill_(n_warm & 0xFF)
        call()
        n_warm += 1
        if n_warm % 64 == 0:
            torch.cuda.synchronize()
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush_buf.fill_(i & 0xFF)
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    barrier()
    per_step = [a.elapsed_time(b) for a, b in ev]  # ms
    clocks = sampler.stop()
    ms_per_step = max_over_ranks(sum(per_step), world, dev) / args.steps
    value = aggregate_rate(x.total_q, world, ms_per_step)

    flags = B.qsa_read_device_status(clear=True)
    if flags:
        print(f"[bench] warning: device status word {flags:#x}", file=sys.stderr)

    # ---- end to end: per-step inputs from pinned host memory, output back ----
    # Every step copies its inputs host -> device, calls the op and copies the
    # output back, through the binding.  Two sets of device inputs/outputs, an
    # upload stream and a read-back stream let step i+1's upload and step
    # i-1's read-back overlap step i's call, as a serving loop would; the L2
    # flush stays on the compute stream before each call, so the call still
    # starts cold.
    e2e = None
    if not args.no_e2e:
        if latent:
            keys = ("q", "input_row_offsets", "swa_cache_lengths", "swa_lookup_table", "comp_cache_lengths",
                    "comp_lookup_table", "comp_indices", "attn_sink")
        else:
            keys = ("q", "input_row_offsets", "cache_lengths", "kv_lookup_table") + (
                ("d_indices",) if blocks else ("token_indices", "counts"))
        host = {k: d[k].cpu().pin_memory() for k in keys}
        sets = [d, dict(d)]
        for k in keys + ("output",):
            sets[1][k] = torch.empty_like(d[k])
        out_host = [torch.empty(d["output"].shape, dtype=d["output"].dtype).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host[0].numel() * out_host[0].element_size()
        up_stream, down_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        uploaded = [torch.cuda.Event() for _ in range(2)]
        called = [torch.cuda.Event() for _ in range(2)]
        read_back = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]

        def e2e_step(i):
            j = i % 2
            s = sets[j]
            with torch.cuda.stream(up_stream):
                if used[j]:
                    up_stream.wait_event(called[j])  # the call two steps back has read this set's inputs
                for k, t in host.items():
                    s[k].copy_(t, non_blocking=True)
                uploaded[j].record(up_stream)
            stream.wait_event(uploaded[j])
            if used[j]:
                stream.wait_event(read_back[j])  # this set's output has been read back
            flush_buf.fill_(i & 0xFF)
            call(s)
            called[j].record(stream)
            with torch.cuda.stream(down_stream):
                down_stream.wait_event(called[j])
                out_host[j].copy_(s["output"], non_blocking=True)
                read_back[j].record(down_stream)
            used[j] = True

        for i in range(4):
            e2e_step(i)
        barrier()
        n_e2e = max(3, min(args.steps, 100))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(up_stream)
        for i in range(n_e2e):
            e2e_step(i)
        e1.record(down_stream)
        barrier()
        te = max_over_ranks(e0.elapsed_time(e1), world, dev)
        e2e = {"value": aggregate_rate(x.total_q, world, te / n_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "note": "each step: H2D of its inputs from pinned memory, an L2 flush, the call, D2H of its output; "
                       "two buffer sets, with step i+1's upload and step i-1's read-back on their own streams "
                       "overlapping step i's call"}

    kname = {1: "qsa simt_kernel", 2: "qsa mma_kernel", 3: "qsa stream_kernel", 4: "qsa rg_kernel"}[plan["kernel"]]
    if latent:
        alg_bytes = x.algorithmic_bytes()
        peak = measured_peaks()
        achieved = alg_bytes / (ms_per_step / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peak["hbm_gbs"], "traffic": recorded_traffic(x.name),
                "peak_source": f"{peak['source']} (MEASURED_PEAKS hbm_gbs copy)", "kernel": kname,
                "algorithmic_bytes_per_launch": alg_bytes}
    else:
        roof = roofline(x, ms_per_step, kname, recorded_traffic(x.name))
        alg_bytes = roof["algorithmic_bytes_per_launch"]
        achieved = roof["effective_gbs"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        cpu = cpu_baseline(x, args.cpu_seconds, args.cpu_threads or host_cores())

    if rank == 0:
        cfg = workload_config(x)
        cfg.update({"kernel": plan["kernel"], "splits": plan["splits"], "ctas": plan["ctas"],
                    "parallelism": f"replicas x{world}"})
        if args.heads_per_unit:
            cfg["heads_per_unit"] = args.heads_per_unit
        if args.tcgen05:
            cfg["tcgen05"] = args.tcgen05
        if plan["kernel"] == 2:
            roof["floor"] = latency_floor(x, ms_per_step, plan["splits"])
        if latent and plan["splits"] == 1 and (x.num_heads // min(x.num_heads, 16)) % 4 == 0:
            # the launch serves four 16-head groups of a row per CTA (qsa_plan counts one per group)
            cfg["ctas"] = plan["ctas"] // 4
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": x.dtype, "data": "synthetic (seeded numpy)", "config": cfg,
            "ms_per_step_median": sorted(per_step)[len(per_step) // 2], "ms_per_step_min": min(per_step),
            "effective_gbs": achieved, "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps,
            "clocks": clocks, "device_status": flags,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
