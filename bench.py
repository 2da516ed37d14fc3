#!/usr/bin/env python
"""Spec-verify step benchmark on GB300 (one JSON line on stdout, rank 0).

A step is the whole hot path over one batch: tq_store of the n_spec draft
tokens of every sequence, then tq_verify (split-KV partial attention and the
log-sum-exp merge in one launch, the last CTA of each (kv-head, sequence)
merging its splits), all through the C ABI.  The default
workload is the PoC shape with the k8v4 preset; the k3v4_nc PoC shape is
measured the same way and reported under "also".

Timing: W warm-up steps, then exactly K steps replayed from CUDA graphs of
`--graph-steps` steps each, bracketed by a barrier and a device synchronise,
timed with CUDA events on the launching stream, max over ranks.  Every step
of a graph uses a different copy of the cache (enough copies to exceed 4x L2),
so no step finds its cache in L2.

--impl reference times the CPU oracle (the plain C implementation the tests
pin the kernels to) on the host cores, on a bounded sample.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per spec-verify call and achieved HBM GB/s vs peak (k8v4, k3v4_nc)"
# seed offsets: the five configurations in order, then the PoC shape with the
# other key widths
CONFIG_INDEX = {"tiny_k8v4": 0, "poc_k8v4": 1, "poc_k3v4_nc": 2, "decode_k3v4_nc": 3, "longctx_k3v4_nc": 4,
                "poc_k4v4_nc": 5, "poc_k2v4_nc": 6, "cont_k8v4": 7}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50000)
    p.add_argument("--warmup", type=int, default=1000)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="poc_k8v4", choices=list(CONFIG_INDEX))
    p.add_argument("--also", default="poc_k3v4_nc,decode_k3v4_nc,longctx_k3v4_nc",
                   help="comma list of extra workloads ('' for none)")
    p.add_argument("--also-steps", type=int, default=400, help="timed steps of each extra workload (at most --steps)")
    p.add_argument("--splits", type=int, default=0, help="NUM_KV_SPLITS (0: the workload's)")
    p.add_argument("--graph-steps", type=int, default=500)
    p.add_argument("--e2e-steps", type=int, default=2000)
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


# --------------------------------------------------------------- plumbing

def dist_setup(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        mine = [s for s in self.samples if s[1][0] == self.uuid] or self.samples
        win = [p for (t, p) in mine if t0 - 0.06 <= t <= t1 + 0.06]
        if not win and mine:  # region shorter than a sample interval: nearest sample
            win = [min(mine, key=lambda s: abs(s[0] - 0.5 * (t0 + t1)))[1]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in win for n, v in zip(names, p[5:9]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback 6.8 TB/s"


def kernel_source_digest(path: str) -> str:
    """First 16 hex digits of the SHA-256 of a CUDA source with its // comments
    and blank lines removed (a comment edit leaves the kernel unchanged)."""
    import re

    lines = []
    for ln in open(path, encoding="utf-8").read().split("\n"):
        ln = re.sub(r"//.*$", "", ln).rstrip()
        if ln.strip():
            lines.append(ln)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def ncu_traffic(kernel_tag: str, workload: str):
    """Per-launch DRAM bytes of the stage-1 kernel from the committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    src = os.path.join(ROOT, "quantized_kv_cache_store_gb300", "csrc", "verify_tc.cu")
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}_ncu.txt")
    try:
        sha = kernel_source_digest(src)
        vals = {}
        for line in open(path):
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
        if vals.get("kernel_source_digest") != sha:
            return None
        return float(vals["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# --------------------------------------------------------------- our arm

def bench_workload(name, args, rank, world, pg, dev_props, steps=None):
    import torch

    from quantized_kv_cache_store_gb300 import tqkv
    from quantized_kv_cache_store_gb300.inputs import WORKLOADS, algorithmic_kv_bytes, make_inputs
    from quantized_kv_cache_store_gb300.step import SpecVerify

    wl = WORKLOADS[name]
    steps = steps or args.steps
    S = args.splits or wl.num_kv_splits
    seed = 1000 + CONFIG_INDEX[name] + 100 * rank  # each rank is its own replica batch
    inp = make_inputs(wl, seed)
    page = tqkv.tq_page_bytes(wl.preset_id)
    cache_bytes = inp.num_blocks * wl.Hk * page
    l2 = int(getattr(dev_props, "L2_cache_size", 128 << 20))
    n_caches = max(2, math.ceil(4 * l2 / cache_bytes))
    G = max(1, min(args.graph_steps, steps))
    sv = SpecVerify(inp, num_kv_splits=S, n_caches=n_caches)
    sv.prefill()
    torch.cuda.synchronize()

    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def capture(nsteps, start, fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(nsteps):
                fn((start + i) % n_caches)
        return g

    # eager warm-up of each entry point (first-call set-up happens outside capture)
    with torch.cuda.stream(stream):
        sv.step_one(0)
    torch.cuda.synchronize()
    step_graph = capture(G, 0, lambda i: sv.step_one(i))
    # K steps = full replays of G plus one shorter graph for the remainder
    full, rem = divmod(steps, G)
    rem_graph = capture(rem, 0, lambda i: sv.step_one(i)) if rem else None
    wfull, wrem = divmod(max(args.warmup, 3), G)
    wrem_graph = capture(wrem, 0, lambda i: sv.step_one(i)) if wrem else None

    def run(nfull, tail):
        for _ in range(nfull):
            step_graph.replay()
        if tail is not None:
            tail.replay()

    uuid = str(getattr(dev_props, "uuid", ""))
    uuid = uuid if uuid.startswith("GPU-") else ("GPU-" + uuid if uuid else "")
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.2)
    with torch.cuda.stream(stream):
        run(wfull, wrem_graph)
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        run(full, rem_graph)
        e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(pg)
    elapsed_ms = e0.elapsed_time(e1)
    time.sleep(0.1)
    clocks.stop()
    clk = clocks.summary(t0, t1)
    elapsed_ms = max_over_ranks(pg, elapsed_ms)
    us_per_step = elapsed_ms * 1e3 / steps
    # the same K-step region replayed a few more times: the spread of the value
    spread = []
    for _ in range(4):
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            run(full, rem_graph)
            e1.record(stream)
        torch.cuda.synchronize()
        spread.append(round(e0.elapsed_time(e1) * 1e3 / steps, 3))

    # per-kernel durations: each launch bracketed by external events in a graph
    kern_us = per_kernel_durations(sv, stream, G, n_caches)
    # the roofline kernel: the launch that reads the cache (the step's single
    # launch, tq_store_verify, when it applies, else stage 1)
    fused = kern_us.get("tq_store_verify") if kern_us else None
    stage1_us = fused if fused else (kern_us["tq_verify_stage1"] if kern_us else None)
    roof_kernel = "tq_store_verify (single launch)" if fused else "tq_verify_stage1"

    # verify-only (stage 1 + 2) throughput, same graph method
    vgraph = capture(G, 0, lambda i: sv.verify_call(i))
    with torch.cuda.stream(stream):
        vgraph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, min(20, steps // G))
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            vgraph.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    verify_us = ev0.elapsed_time(ev1) * 1e3 / (reps * G)

    alg_bytes = algorithmic_kv_bytes(wl, inp.seq_lens, page)
    peak, peak_src = measured_peaks()
    roof = None
    if stage1_us:
        achieved = alg_bytes / (stage1_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "kernel": roof_kernel, "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": ncu_traffic("stage1", name), "algorithmic_bytes": alg_bytes,
                "stage1_us": round(stage1_us, 3), "peak_source": peak_src}
    return dict(wl=wl, S=S, seed=seed, inp=inp, sv=sv, n_caches=n_caches, cache_bytes=cache_bytes,
                us_per_step=us_per_step, replays_us=spread, steps=steps, verify_us=verify_us, kernels_us=kern_us, roofline=roof,
                clocks=clk, alg_bytes=alg_bytes, G=G, stream=stream)


def single_launch(sv) -> bool:
    """Whether tq_verify / tq_store_verify run as one cooperative launch: up
    to 32 splits and every CTA (split x kv-head x sequence x row tile of 64
    rows) resident at once, one per SM."""
    import torch

    wl = sv.wl
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    rtiles = (wl.n_spec * wl.Hq // wl.Hk + 63) // 64
    return sv.S <= 32 and sv.S * wl.Hk * wl.B * rtiles <= sms


def per_kernel_durations(sv, stream, G, n_caches):
    """Average duration of each kernel: a CUDA graph of G launches of that
    kernel alone (the cache copy rotating as in the step), timed with events
    on the launching stream after a warm-up replay."""
    import torch

    from quantized_kv_cache_store_gb300 import tqkv

    calls = {
        "tq_store": lambda c: sv.store(c, stream),
        "tq_verify_stage1": lambda c: tqkv.tq_verify_stage1(sv.caches[c], sv.preset, sv.q, sv.block_table,
                                                            sv.seq_lens, sv.S, sv.wl.causal, sv.part_o,
                                                            sv.part_lse, stream),
        "tq_verify_stage2": lambda c: tqkv.tq_verify_stage2(sv.part_o, sv.part_lse, sv.out, stream),
    }
    if single_launch(sv):  # tq_verify and tq_store_verify are one launch each
        calls["tq_verify_fused"] = lambda c: sv.verify_call(c, stream)
        calls["tq_store_verify"] = lambda c: sv.step_one(c, stream)
    out = {}
    for name, fn in calls.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                fn(i % n_caches)
        with torch.cuda.stream(stream):
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(4):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        out[name] = e0.elapsed_time(e1) * 1e3 / (4 * G)
    return out


def e2e_measure(res, args):
    """Same step through the public API with HOST buffers: pinned host -> device
    copies of the step's inputs, the tq_store_verify call, device -> host copy of the
    result, every step, eager (no graph)."""
    import torch

    sv, inp = res["sv"], res["inp"]
    stream = res["stream"]
    drafts = inp.draft_rows()
    h_q = inp.q.contiguous().pin_memory()
    h_k = inp.k[drafts].contiguous().pin_memory()
    h_v = inp.v[drafts].contiguous().pin_memory()
    h_out = torch.empty(sv.out.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v))
    d2h = h_out.numel() * h_out.element_size()
    n = max(1, min(args.e2e_steps, args.steps))

    def one(i):
        sv.q.copy_(h_q, non_blocking=True)
        sv.k_new.copy_(h_k, non_blocking=True)
        sv.v_new.copy_(h_v, non_blocking=True)
        sv.step_one(i % res["n_caches"], stream)
        h_out.copy_(sv.out, non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(20):
            one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(n):
            one(i)
        e1.record(stream)
    torch.cuda.synchronize()
    return {"value": round(e0.elapsed_time(e1) * 1e3 / n, 3), "unit": "us", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n, "mode": "eager C-ABI calls, pinned host buffers"}


def isolated_latency(res, reps=20):
    """One step at a time after an L2 flush (a 256 MB write): median of reps
    event-timed single calls, each on a cold L2 and an idle GPU."""
    import torch

    sv, stream = res["sv"], res["stream"]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=sv.device)
    times = []
    for i in range(reps):
        with torch.cuda.stream(stream):
            flush.fill_(i & 255)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            sv.step_one(i % res["n_caches"], stream)
            e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    return round(statistics.median(times), 3)


def store_throughput(res, reps=5):
    """tq_store of every cached prefix token (the untimed cache fill of a
    step, HBM-write bound): device-resident fp16 K/V, event-timed, best of reps.
    Bytes = fp16 K and V read + cache slots written."""
    import torch

    from quantized_kv_cache_store_gb300 import tqkv

    sv, inp, stream = res["sv"], res["inp"], res["stream"]
    rows = inp.prefix_rows()[: 1 << 18]
    k = inp.k[rows].to(sv.device)
    v = inp.v[rows].to(sv.device)
    sl = torch.from_numpy(inp.slots[rows]).to(sv.device)
    cache = sv.caches[-1]
    best = None
    for _ in range(reps):
        with torch.cuda.stream(stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            tqkv.tq_store(cache, sv.preset, k, v, sl, stream)
            e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) * 1e3
        best = t if best is None else min(best, t)
    th = len(rows) * sv.wl.Hk
    nbytes = th * (2 * 128 * 2 + tqkv.tq_page_bytes(sv.preset) // 16)
    # the cache copy written here is restored, so later steps see the same bytes
    cache.copy_(sv.caches[0])
    torch.cuda.synchronize()
    return {"token_heads": th, "us": round(best, 3), "GB/s": round(nbytes / (best * 1e-6) / 1e9, 1),
            "bytes": nbytes}


def cpu_baseline(res, budget_s=12.0, max_calls=5):
    """The oracle as it stands (C, OpenMP over (sequence, kv-head)) on the
    host cores: store of the step's draft tokens + fp64 verify of every row,
    repeated while the budget lasts."""
    import numpy as np

    import oracle

    inp, wl = res["inp"], res["wl"]
    page = oracle.page_bytes(wl.preset_id)
    cache = np.zeros((inp.num_blocks, wl.Hk, page), np.uint8)
    pre = inp.prefix_rows()
    oracle.store(wl.preset_id, cache, inp.k.numpy()[pre], inp.v.numpy()[pre], inp.slots[pre])
    drafts = inp.draft_rows()
    kd, vd, sd = inp.k.numpy()[drafts], inp.v.numpy()[drafts], inp.slots[drafts]
    q = inp.q.numpy()
    times = []
    t_start = time.time()
    while not times or (time.time() - t_start < budget_s and len(times) < max_calls):
        t0 = time.perf_counter()
        oracle.store(wl.preset_id, cache, kd, vd, sd)
        oracle.verify(wl.preset_id, cache, q, inp.block_table, inp.seq_lens, wl.causal)
        times.append(time.perf_counter() - t0)
    cores = os.cpu_count()
    return {"value": round(statistics.median(times) * 1e6, 1), "unit": "us", "cores": cores,
            "kind": "oracle",
            "sample": f"{len(times)} full calls of {wl.name} (store of {len(drafts)} draft tokens + fp64 "
                      f"verify of all {wl.n_spec * wl.B * wl.Hq} rows), median, OpenMP {cores} threads"}


def run_ours(args):
    import torch

    from quantized_kv_cache_store_gb300 import _build, tqkv

    rank, world, local, pg = dist_setup(args)
    _build.build()
    tqkv.load()
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    main = bench_workload(args.workload, args, rank, world, pg, props)
    e2e = e2e_measure(main, args)
    iso_us = isolated_latency(main)
    store_tp = store_throughput(main)
    also = {}
    for name in [x for x in args.also.split(",") if x and x != args.workload]:
        r = bench_workload(name, args, rank, world, pg, props, steps=min(args.steps, args.also_steps))
        also[name] = {"us_per_step": round(r["us_per_step"] / world, 3), "steps": r["steps"],
                      "replays_us": r["replays_us"], "verify_us": round(r["verify_us"], 3),
                      "kernels_us": _round(r["kernels_us"]), "roofline": r["roofline"],
                      "num_kv_splits": r["S"], "clocks": r["clocks"],
                      "single_launch": single_launch(r["sv"])}
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            also[name]["cpu_baseline"] = cpu_baseline(r, budget_s=8.0, max_calls=2)
        del r
        torch.cuda.empty_cache()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(main)
    if rank != 0:
        return
    wl = main["wl"]
    out = {
        "metric": METRIC, "value": round(main["us_per_step"] / world, 3), "unit": "us", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(main["us_per_step"] / 1e3, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "fp16-mma/fp32-acc",
        "data": "synthetic (seeded N(0,1) fp16 Q/K/V, quantised into the paged cache by tq_store)",
        "config": {"workload": wl.name, "preset": wl.preset, "n_spec": wl.n_spec, "B": wl.B, "Hq": wl.Hq,
                   "Hk": wl.Hk, "D": 128, "seq_len": wl.seq_len, "cached_len": wl.seq_len - wl.n_spec,
                   "causal": wl.causal, "num_kv_splits": main["S"], "seed": main["seed"],
                   "step": "tq_store_verify: store of the n_spec*B draft tokens + split-KV attention + counter-synchronised merge, one cooperative launch",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2: {main['n_caches']} rotating cache copies of "
                         f"{main['cache_bytes'] / 1e6:.1f} MB",
                   "graph": f"CUDA graphs of {main['G']} steps"},
        "replays_us": main["replays_us"],
        "verify_us": round(main["verify_us"], 3),
        "kernels_us": _round(main["kernels_us"]),
        "roofline": main["roofline"],
        "cpu_baseline": cpu,
        "e2e": e2e,
        "isolated_us": iso_us,
        "store_prefill": store_tp,
        "gpu_launches": (1 if single_launch(main["sv"]) else 3) * args.steps,
        "clocks": main["clocks"],
        "also": also,
    }
    print(json.dumps(out), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def _round(d):
    return {k: round(v, 3) for k, v in d.items()} if d else d


# --------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle on the host cores, same workload / metric / unit."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    import oracle
    from quantized_kv_cache_store_gb300.inputs import WORKLOADS, make_inputs

    oracle.build()
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl, 1000 + CONFIG_INDEX[args.workload])
    page = oracle.page_bytes(wl.preset_id)
    cache = np.zeros((inp.num_blocks, wl.Hk, page), np.uint8)
    pre = inp.prefix_rows()
    oracle.store(wl.preset_id, cache, inp.k.numpy()[pre], inp.v.numpy()[pre], inp.slots[pre])
    drafts = inp.draft_rows()
    kd, vd, sd = inp.k.numpy()[drafts], inp.v.numpy()[drafts], inp.slots[drafts]
    q = inp.q.numpy()

    def step():
        oracle.store(wl.preset_id, cache, kd, vd, sd)
        oracle.verify(wl.preset_id, cache, q, inp.block_table, inp.seq_lens, wl.causal)

    t0 = time.perf_counter()
    step()
    t_one = time.perf_counter() - t0
    budget = 150.0
    k = max(1, min(args.steps, int(budget / max(t_one, 1e-6))))
    w = min(max(args.warmup, 0), 1)
    for _ in range(w):
        step()
    times = []
    for _ in range(k):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    v = statistics.mean(times) * 1e6
    cores = os.cpu_count()
    out = {"impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "us", "n_gpus": 1,
           "steps": k, "warmup": w, "ms_per_step": round(v / 1e3, 3), "higher_is_better": False,
           "scaling": "weak", "vs_baseline": None, "dtype": "fp32 encoder / fp64 attention",
           "data": "synthetic (same seeded workload as the GPU arm)",
           "config": {"workload": wl.name, "preset": wl.preset, "n_spec": wl.n_spec, "B": wl.B, "Hq": wl.Hq,
                      "Hk": wl.Hk, "D": 128, "seq_len": wl.seq_len, "cached_len": wl.seq_len - wl.n_spec,
                      "causal": wl.causal, "num_kv_splits": wl.num_kv_splits,
                      "seed": 1000 + CONFIG_INDEX[args.workload],
                      "step": "oracle store of the drafts + fp64 verify of all rows (split-free)"},
           "cpu_baseline": {"value": round(v, 1), "unit": "us", "cores": cores, "kind": "oracle",
                            "sample": f"{k} full oracle calls (steps capped from {args.steps} to fit "
                                      f"{budget:.0f} s), OpenMP {cores} threads"},
           "e2e": {"value": round(v, 1), "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
