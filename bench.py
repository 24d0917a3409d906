"""Benchmark of the DSA hot path on GB300 (one JSON line on stdout).

A step is one pass of the whole path -- indexer scores, top-k selection,
sparse absorbed-MLA attention -- over one batch of the workload, through the
library's C ABI.  The default workload is GLM-5.2 decode at 131072 cached
tokens with top-k 2048 (batch 1, bf16), the configuration the metric is quoted
on.  Every input is seeded and synthetic.

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and a device synchronise, timed with CUDA events on the launching stream.
The large streamed inputs (indexer keys and the latent cache) rotate over
several independently drawn copies whose total exceeds the L2 cache, so a step
never finds its keys in L2.

Under torchrun each rank runs an independent replica on its own GPU ("weak"
scaling, no data-path collective); the reported time is the maximum over
ranks and ``value`` counts the queries of all ranks.

``--impl reference`` times the host oracle (plain C, double precision) on this
machine's CPU cores on a bounded sample of the same workload, as the
comparison arm.
"""
from __future__ import annotations

import argparse
import gc
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

METRIC = "DSA decode queries/s at 128K ctx, top-2048, and % of GB300 HBM roofline"
UNIT = "queries/s"
DEFAULT_WORKLOAD = "glm52_decode_128k"
L2_BYTES = 135528448


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-graph", action="store_true",
                   help="launch each step on the stream instead of replaying CUDA graphs")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU work of the oracle baseline sample (all threads; a third "
                        "of it on one thread)")
    p.add_argument("--no-configs", action="store_true",
                   help="time only --workload, not the other workloads of the suite")
    return p.parse_args(argv)


# ------------------------------------------------------------------ plumbing

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def agree_steps(pg, steps: int, device) -> int:
    """Every rank times rank 0's step count (each calibrates its own)."""
    if pg is None:
        return steps
    import torch
    t = torch.tensor([steps], dtype=torch.int64, device=device)
    pg.broadcast(t, src=0)
    return int(t[0])


def max_over_ranks(pg, values, device):
    """Element-wise maximum of a list of floats over all ranks."""
    if pg is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(world: int, queries_per_rank: int, ms_per_step: float) -> float:
    """Whole-job queries/s: every rank decodes its own replica of the batch in
    each step, and the step takes the slowest rank's time."""
    return world * queries_per_rank / (ms_per_step / 1e3)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.25)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        mhz, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz),
                "power_w_max": max(power) if power else None}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


def kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    ent = table.get(f"{kernel}@{workload}")
    if not ent:
        return None
    h = hashlib.sha256()
    try:
        for name in ent["sources"]:
            with open(os.path.join(ROOT, "deepseek_sparse_attention_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
    except (OSError, KeyError):
        return None
    digest = h.hexdigest()[:16]
    return ent["bytes_per_launch"] if digest == ent["source_sha"] else None


# ------------------------------------------------------------------ work model

def algorithmic(wl):
    """Algorithmic bytes and flops of one step, and of one indexer launch.

    Indexer: every visible key (256 B; a pool key per 4 tokens in k-pool mode)
    once, the query heads and weights, and one float score written per key.
    Selection: the scores read once.  Attention: every selected row (R * 2 B)
    once, the absorbed query, and the float output + lse written.
    """
    esz = 4 if wl.dtype == "f32" else 2
    nv = wl.q_nvis()
    seq_of_q = [s for s, nq in enumerate(wl.q_lens) for _ in range(nq)]
    keys_per_seq = {}
    for s, L in zip(seq_of_q, nv):
        keys_per_seq[s] = max(keys_per_seq.get(s, 0), L // wl.kpool)
    key_bytes = sum(keys_per_seq.values()) * wl.idx_dim * esz          # keys read once per seq
    scored = sum(L // wl.kpool for L in nv)                            # (query, key) pairs
    n_sel = []
    for L in nv:
        if wl.kpool == 1:
            n_sel.append(min(L, wl.top_k))
        else:
            n_sel.append(L if L // wl.kpool <= wl.top_k // wl.kpool else wl.top_k + L % wl.kpool)
    q_bytes = wl.n_q * (wl.idx_heads * wl.idx_dim * esz + wl.idx_heads * 4)
    idx_bytes = key_bytes + q_bytes + scored * 4
    sel_bytes = scored * 4 + sum(n_sel) * 4
    row_bytes = sum(n_sel) * wl.width * esz
    att_bytes = row_bytes + wl.n_q * wl.heads * wl.width * esz + wl.n_q * wl.heads * (wl.kv_lora + 1) * 4
    flops_idx = scored * wl.idx_heads * wl.idx_dim * 2
    flops_att = sum(n_sel) * wl.heads * (wl.width + wl.kv_lora) * 2
    return {"step_bytes": idx_bytes + sel_bytes + att_bytes,
            "compulsory_bytes": key_bytes + q_bytes + row_bytes + wl.n_q * wl.heads * wl.width * esz
            + wl.n_q * wl.heads * (wl.kv_lora + 1) * 4,
            "index_launch_bytes": idx_bytes, "select_bytes": sel_bytes, "scored_keys": scored,
            "selected_rows": sum(n_sel),
            "flops": flops_idx + flops_att, "flops_index": flops_idx}


# ------------------------------------------------------------------ CPU arm

def oracle_baseline(wl, d, seconds: float, single_seconds: float):
    """The oracle on this machine's cores, as the CPU baseline.

    Host float copies of (at most two of) the workload's queries are made
    before any clock starts; the timed loops run only the oracle over them:
    every thread for about `seconds`, then one thread for about
    `single_seconds` (at least one query each)."""
    import oracle

    oracle.build()
    fn = host_query_args(wl, d)
    qs = list(dict.fromkeys((i * 7919) % wl.n_q for i in range(min(wl.n_q, 2))))
    args = [fn(q) for q in qs]

    def run(sec):
        done, t0 = 0, time.perf_counter()
        while True:
            oracle.decode_step(*args[done % len(args)])
            done += 1
            el = time.perf_counter() - t0
            if el >= sec:
                return done, el

    full = oracle.threads()
    n, el = run(seconds)
    oracle.set_threads(1)
    try:
        n1, el1 = run(single_seconds)
    finally:
        oracle.set_threads(full)
    what = f"the {wl.name} workload (quer{'y' if len(qs) == 1 else 'ies'} {qs}) through the oracle"
    return {"value": n / el, "unit": UNIT, "cores": full, "kind": "oracle",
            "sample": f"{n} queries of {what}, double precision, {full} OpenMP threads, "
                      f"{el:.1f} s; inputs copied to host memory before timing",
            "single_thread": {"value": n1 / el1, "unit": UNIT, "cores": 1,
                              "sample": f"{n1} queries of {what} on one thread, {el1:.1f} s"}}


def host_query_args(wl, d):
    """Closure giving the oracle's arguments for query q from (device or host)
    tensors of the workload."""
    def f(q):
        seq = [s for s, nq in enumerate(wl.q_lens) for _ in range(nq)][q]
        L = wl.q_nvis()[q]
        r0 = sum(wl.kv_lens[:seq])
        k0 = sum(wl.key_counts()[:seq])
        nk = L // wl.kpool
        g = lambda t: t.detach().float().cpu().numpy()
        return (g(d["q_idx"][q]), g(d["w"][q]), g(d["k_idx"][k0:k0 + nk]), g(d["q_abs"][q]),
                g(d["cache"][r0:r0 + L]), L, wl.top_k, wl.kpool, wl.scale, wl.kv_lora)
    return f


def oracle_fraction(wl, args_q, f: float):
    """A fraction f of one query's oracle work: the indexer over the first f*n
    keys, the selection of the top f*k of those, and attention over that many
    rows.  Every stage is linear in its size except the sort inside the
    selection (n log n), so the scaled time slightly favours the oracle."""
    import numpy as np
    import oracle

    q_idx, w, keys, q_abs, rows, L, k, kpool, scale, dv = args_q
    nk = max(1, int(round(keys.shape[0] * f)))
    s = oracle.index_scores(q_idx, w, keys[:nk])
    kk = max(1, int(round(min(k, L) * f)))
    sel = oracle.topk(s, kk // kpool if kpool > 1 else kk)
    sel = np.asarray(sel, dtype=np.int32) % rows.shape[0]
    oracle.sparse_mla(q_abs, rows, sel, scale, dv)


def run_reference(args):
    """The host oracle as the comparison arm (rank 0 only).

    Each of the K steps is a bounded sample of the workload: whole queries
    when one fits the per-step budget, else the same fraction of every stage of
    one query.  The budget keeps the whole run within about two minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    import workloads

    oracle.build()
    wl = workloads.named(args.workload)
    d = workloads.make(wl, "cpu")
    steps = args.steps if args.steps is not None else 10
    warm = args.warmup if args.warmup is not None else 1
    fn = host_query_args(wl, d)
    a0 = fn(0)
    t0 = time.perf_counter()
    oracle.decode_step(*a0)                      # calibration, untimed
    t_query = time.perf_counter() - t0
    budget = 90.0 / max(1, steps + warm)
    if budget >= t_query:
        per_step, frac = int(min(budget // t_query, max(1, wl.n_q))), 1.0
    else:
        per_step, frac = 1, max(budget / t_query, 1.0 / 4096)
    cache = {}

    def one_step(i):
        done = 0.0
        for j in range(per_step):
            q = ((i * per_step + j) * 7919) % wl.n_q
            if q not in cache:
                cache.clear()
                cache[q] = fn(q)
            if frac >= 1.0:
                oracle.decode_step(*cache[q])
            else:
                oracle_fraction(wl, cache[q], frac)
            done += frac
        return done

    for i in range(warm):
        one_step(i)
    t0 = time.perf_counter()
    total_q = 0.0
    for i in range(steps):
        total_q += one_step(warm + i)
    el = time.perf_counter() - t0
    value = total_q / el
    threads = oracle.threads()
    if frac >= 1.0:
        sample = (f"{per_step} whole quer{'y' if per_step == 1 else 'ies'} of the {wl.name} "
                  f"workload per step")
    else:
        sample = (f"{frac:.4g} of one {wl.name} query per step (every stage scaled by that "
                  f"fraction), counted as {frac:.4g} queries")
    sample += f"; oracle in double precision on {threads} threads"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": el / steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def workload_config(wl, world):
    return {"workload": wl.name, "description": wl.description, "batch": wl.n_q,
            "n_seq": wl.n_seq, "max_context": max(wl.kv_lens), "top_k": wl.top_k,
            "kpool": wl.kpool, "heads": wl.heads, "row_width": wl.width,
            "indexer": f"{wl.idx_heads}x{wl.idx_dim}", "parallelism": f"replicas x{world}",
            "l2": "inputs rotate over copies larger than L2"}


# ------------------------------------------------------------------ GPU arm

def graph_time_ms(call, n: int, stream) -> float:
    """Mean device time of call(i) over n launches: three untimed calls, then
    the n launches captured in one CUDA graph and replayed (once untimed), so
    that the per-call host cost of the Python binding -- tens of
    microseconds, longer than some of these kernels -- does not set the pace."""
    import torch

    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    gc.collect()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            call(i)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    del g
    gc.collect()
    return ms


def dominant_launch(dsa, wl, sh, b, d, keys, copies, stream, n_rep):
    """The launch that carries the step's dominant work, timed alone with CUDA
    events on the stream it runs on, over the same input rotation: the fused
    indexer + selection for small decode batches, else the indexer.  Also the
    indexer alone.  Returns (fused?, fused ms, indexer ms)."""
    import torch

    sb = torch.empty((wl.n_q, max(max(wl.kv_lens) // wl.kpool, 4)), device=keys[0].device)
    ld = sb.shape[1]
    ws_i = dsa.alloc_workspace(sh, b, dsa.OP_INDEX_SCORES, keys[0].device)
    idx_ms = graph_time_ms(lambda i: dsa.dsa_index_scores(sh, b, d["q_idx"], d["w"],
                                                          keys[i % copies], sb, ld, ws_i),
                           n_rep, stream)
    if dsa.dsa_check_device_error(ws_i, stream) != 0:
        raise RuntimeError("device error in the indexer loop")
    del sb
    fused = dsa.dsa_plan(sh, b, dsa.OP_INDEX_SELECT)["kernel_launches"] == 1
    sel_ms = 0.0
    if fused:
        ws_s = dsa.alloc_workspace(sh, b, dsa.OP_INDEX_SELECT, keys[0].device)
        width = dsa.dsa_index_row_width(sh)
        idx_s = torch.empty((wl.n_q, width), dtype=torch.int32, device=keys[0].device)
        nsel_s = torch.empty(wl.n_q, dtype=torch.int32, device=keys[0].device)
        sel_ms = graph_time_ms(lambda i: dsa.dsa_index_select(sh, b, d["q_idx"], d["w"],
                                                              keys[i % copies], idx_s, nsel_s,
                                                              ws_s),
                               n_rep, stream)
        if dsa.dsa_check_device_error(ws_s, stream) != 0:
            raise RuntimeError("device error in the fused selection loop")
    return fused, sel_ms, idx_ms


def roofline_of(wl, fused, sel_ms, idx_ms, peaks, peak_src):
    """The roofline object of the dominant launch (see dominant_launch)."""
    work = algorithmic(wl)
    if fused:
        dom = {"kernel": "index_select_fused", "ms": sel_ms,
               "bytes": work["index_launch_bytes"] + work["select_bytes"]}
    else:
        dom = {"kernel": "index_scores_tc" if wl.dtype == "bf16" else "index_scores (CUDA cores)",
               "ms": idx_ms, "bytes": work["index_launch_bytes"]}
    # A prefill chunk re-reads each key tile for many queries: its indexer does
    # far more flops per byte than the GPU's flop/byte balance and is bound by
    # the tensor pipe, so its roofline is in TFLOP/s against the bf16 peak.
    tensor_bound = (work["flops_index"] / max(work["index_launch_bytes"], 1) >
                    peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9))
    if tensor_bound and not fused:
        roof = {"bound": "tensor", "kernel": dom["kernel"],
                "achieved": work["flops_index"] / (dom["ms"] / 1e3) / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "flops_per_launch": work["flops_index"], "peak_source": f"{peak_src} bf16_tflops"}
    else:
        roof = {"bound": "hbm", "kernel": dom["kernel"],
                "achieved": dom["bytes"] / (dom["ms"] / 1e3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "bytes_per_launch": dom["bytes"],
                "peak_source": f"{peak_src} hbm_gbs"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = kernel_traffic(dom["kernel"], wl.name)
    roof["launch_us"] = dom["ms"] * 1e3
    return roof


def time_projections(dsa, wl, dev, stream, peaks, peak_src, n_rep=50):
    """The query absorption and the output up-projection of the workload's
    queries, each timed alone with CUDA events, the weights rotating over
    copies larger than L2 (each layer of a model has its own).  Algorithmic
    bytes: the weights, the inputs and the outputs once; flops 2 per
    multiply-add."""
    import torch
    import workloads

    nope, v_dim = 192, 256
    esz = 2 if wl.dtype == "bf16" else 4
    w_bytes = wl.heads * (nope + v_dim) * wl.kv_lora * esz
    copies = min(16, max(2, math.ceil(2 * L2_BYTES / w_bytes)))
    p = workloads.projections(wl, dev, nope=nope, v_dim=v_dim, copies=copies)
    sh = dsa.make_shape(wl.idx_heads, wl.idx_dim, wl.heads, wl.kv_lora, wl.rope, wl.top_k,
                        wl.kpool, wl.scale, wl.dtype)
    zero = torch.zeros(2, dtype=torch.int64, device=dev)
    ws = dsa.alloc_workspace(sh, dsa.make_batch(zero, zero, zero, 0, 0, 0, 1, 1),
                             dsa.OP_PROJECT, dev)
    q_abs = torch.empty((wl.n_q, wl.heads, wl.kv_lora + wl.rope), dtype=p["q_full"].dtype,
                        device=dev)
    out = torch.empty((wl.n_q, wl.heads, v_dim), device=dev)
    res = {}
    for name in ("absorb_q", "up_project"):
        def call(i):
            if name == "absorb_q":
                dsa.dsa_absorb_q(sh, p["q_full"], p["w_uk_copies"][i % copies], q_abs, ws)
            else:
                dsa.dsa_up_project(sh, p["o"], p["w_uv_copies"][i % copies], out, ws)
        ms = graph_time_ms(call, n_rep, stream)
        if dsa.dsa_check_device_error(ws, stream) != 0:
            raise RuntimeError(f"device error in the {name} loop")
        if name == "absorb_q":
            byts = (wl.heads * nope * wl.kv_lora * esz + p["q_full"].numel() * esz
                    + q_abs.numel() * esz)
            flops = 2 * wl.n_q * wl.heads * nope * wl.kv_lora
        else:
            byts = wl.heads * v_dim * wl.kv_lora * esz + p["o"].numel() * 4 + out.numel() * 4
            flops = 2 * wl.n_q * wl.heads * v_dim * wl.kv_lora
        t_mem = byts / (peaks["hbm_gbs"] * 1e9)
        t_flop = flops / (peaks["bf16_tflops"] * 1e12)
        ent = {"launch_us": ms * 1e3, "bytes_per_launch": byts, "flops_per_launch": flops,
               "weight_copies": copies}
        if t_mem >= t_flop:
            ach = byts / (ms / 1e3) / 1e9
            ent.update(bound="hbm", achieved=ach, unit="GB/s", peak=peaks["hbm_gbs"],
                       frac=ach / peaks["hbm_gbs"], peak_source=f"{peak_src} hbm_gbs")
        else:
            ach = flops / (ms / 1e3) / 1e12
            ent.update(bound="tensor", achieved=ach, unit="TFLOP/s", peak=peaks["bf16_tflops"],
                       frac=ach / peaks["bf16_tflops"], peak_source=f"{peak_src} bf16_tflops")
        res[name] = ent
    del p
    torch.cuda.empty_cache()
    return res


class StepBench:
    """One workload's inputs on the device and its timed step loop."""

    def __init__(self, dsa, wl, dev, stream, no_graph: bool):
        import torch
        import workloads

        self.dsa, self.wl, self.dev, self.stream = dsa, wl, dev, stream
        per_copy = algorithmic(wl)["step_bytes"]
        self.copies = min(8, max(2, math.ceil(2 * L2_BYTES / max(per_copy, 1))))
        d = self.d = workloads.make(wl, dev, copies=self.copies)
        self.sh = dsa.make_shape(wl.idx_heads, wl.idx_dim, wl.heads, wl.kv_lora, wl.rope,
                                 wl.top_k, wl.kpool, wl.scale, wl.dtype)
        self.b = dsa.make_batch(d["row_off"], d["key_off"], d["q_off"], wl.n_q, max(wl.q_lens),
                                max(wl.kv_lens), sum(wl.kv_lens), sum(wl.key_counts()))
        self.ws = dsa.alloc_workspace(self.sh, self.b, dsa.OP_DECODE_STEP, dev)
        width = dsa.dsa_index_row_width(self.sh)
        self.plan = dsa.dsa_plan(self.sh, self.b, dsa.OP_DECODE_STEP)
        self.out = torch.empty((wl.n_q, wl.heads, wl.kv_lora), device=dev)
        self.lse = torch.empty((wl.n_q, wl.heads), device=dev)
        self.idx = torch.empty((wl.n_q, width), dtype=torch.int32, device=dev)
        self.n_sel = torch.empty(wl.n_q, dtype=torch.int32, device=dev)
        self.keys, self.caches = d["k_idx_copies"], d["cache_copies"]
        self.no_graph = no_graph
        self.launch_mode = "stream launches"

    def launch(self, i, st):
        c = i % self.copies
        self.dsa.dsa_decode_step(self.sh, self.b, self.d["q_idx"], self.d["w"], self.keys[c],
                                 self.d["q_abs"], self.caches[c], self.out, self.lse, self.idx,
                                 self.n_sel, self.ws, st)

    def prepare(self, warm: int, steps: int = None):
        """Warm-up steps, then the CUDA graphs the timed steps replay: a decode
        loop replays its step from graphs (the launches of a step and of
        consecutive steps then overlap through programmatic dependent launch
        without host round trips): one graph of G steps over the input copies
        in turn -- all K timed steps when K is known and at most 256 -- and one
        single-step graph per copy for the remainder, so that exactly K steps
        run."""
        import torch

        dsa, dev = self.dsa, self.dev
        # Graphs of an earlier workload must not be destroyed while this one is
        # being captured (destroying a graph is not allowed during a capture):
        # collect any that are unreachable now.
        gc.collect()
        for i in range(max(warm, 3)):
            self.launch(i, self.stream)
        torch.cuda.synchronize(dev)
        if dsa.dsa_check_device_error(self.ws, self.stream) != 0:
            raise RuntimeError(f"device error during warm-up ({self.wl.name})")
        if self.no_graph:
            self.run_steps = lambda n: [self.launch(i, self.stream) for i in range(n)]
            return
        G = steps if steps is not None and 0 < steps <= 256 else self.copies * max(1, 48 // self.copies)
        g_all = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_all):
            for i in range(G):
                self.launch(i, torch.cuda.current_stream(dev))
        g_one = []
        for c in range(self.copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.launch(c, torch.cuda.current_stream(dev))
            g_one.append(g)
        copies = self.copies

        def run_steps(n):                            # holds the graphs, not self
            for _ in range(n // G):
                g_all.replay()
            for i in range(n % G):
                g_one[i % copies].replay()

        self.run_steps = run_steps
        run_steps(G)                                 # untimed: the graphs' first replays
        torch.cuda.synchronize(dev)
        if dsa.dsa_check_device_error(self.ws, self.stream) != 0:
            raise RuntimeError(f"device error in the graph warm-up ({self.wl.name})")
        self.launch_mode = f"CUDA graphs of {G} steps (+ single-step graphs for the remainder)"

    def release(self):
        """Destroys the graphs now (outside any capture) and frees the inputs."""
        import torch

        torch.cuda.synchronize(self.dev)
        self.run_steps = None
        self.d = self.keys = self.caches = None
        gc.collect()
        torch.cuda.empty_cache()

    def calibrate(self, seconds: float, lo: int = 20, hi: int = 200000) -> int:
        import torch

        t0 = time.perf_counter()
        self.run_steps(10)
        torch.cuda.synchronize(self.dev)
        per = (time.perf_counter() - t0) / 10
        return int(min(hi, max(lo, seconds / max(per, 1e-7))))

    def timed(self, steps: int, pg, local: int):
        """(ms for `steps` steps, clock record) between barriers and syncs."""
        import torch

        clocks = ClockSampler(local)
        clocks.start()
        if pg:
            pg.barrier()
        torch.cuda.synchronize(self.dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        self.run_steps(steps)
        e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        if pg:
            pg.barrier()
        clk = clocks.stop()
        if self.dsa.dsa_check_device_error(self.ws, self.stream) != 0:
            raise RuntimeError(f"device error during the timed region ({self.wl.name})")
        return e0.elapsed_time(e1), clk


def step_metrics(wl, per_step_ms, world, peaks):
    """Throughput and whole-step roofline figures of one step time."""
    work = algorithmic(wl)
    gbs = work["compulsory_bytes"] / (per_step_ms / 1e3) / 1e9
    tfs = work["flops"] / (per_step_ms / 1e3) / 1e12
    return {"value": job_throughput(world, wl.n_q, per_step_ms),
            "tokens_per_s": work["scored_keys"] / (per_step_ms / 1e3) * world,
            "step_hbm_gbs": gbs, "step_hbm_frac": gbs / peaks["hbm_gbs"],
            "step_tflops": tfs, "step_tensor_frac": tfs / peaks["bf16_tflops"]}


def time_e2e(dsa, sb, n_steps: int, no_graph: bool) -> dict:
    """The step end to end through the public call a host-fed caller makes,
    dsa_decode_step_host: every step's query inputs (q_idx, w, q_abs) are read
    from one page-locked host buffer and its output is written to page-locked
    host memory, inside the timed region.  Timed like the device-side value
    (the calls captured in CUDA graphs of G steps over the input copies,
    replayed), and also as plain stream calls, one per step."""
    import torch

    wl, d, dev, stream = sb.wl, sb.d, sb.dev, sb.stream
    names = ("q_idx", "w", "q_abs")
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += (d[k].numel() * d[k].element_size() + 255) // 256 * 256
    h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    hq = {}
    for k in names:
        n = d[k].numel() * d[k].element_size()
        h_in[offs[k]:offs[k] + n].copy_(d[k].reshape(-1).view(torch.uint8).cpu())
        hq[k] = h_in[offs[k]:offs[k] + n].view(d[k].dtype).view(d[k].shape)
    h_out = torch.empty(sb.out.shape, dtype=sb.out.dtype).pin_memory()
    ws = dsa.alloc_workspace(sb.sh, sb.b, dsa.OP_DECODE_STEP_HOST, dev)
    h2d = sum(d[k].numel() * d[k].element_size() for k in names)
    d2h = h_out.numel() * h_out.element_size()

    def call(i, st):
        c = i % sb.copies
        dsa.dsa_decode_step_host(sb.sh, sb.b, hq["q_idx"], hq["w"], sb.keys[c], hq["q_abs"],
                                 sb.caches[c], h_out, None, sb.idx, sb.n_sel, ws, st)

    def timed(fn, n):
        torch.cuda.synchronize(dev)
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        fn()
        x1.record(stream)
        torch.cuda.synchronize(dev)
        return x0.elapsed_time(x1) / n

    for i in range(3):
        call(i, stream)
    torch.cuda.synchronize(dev)
    n_stream = min(n_steps, 2000)
    stream_ms = timed(lambda: [call(i, stream) for i in range(n_stream)], n_stream)
    if no_graph:
        e2e_ms, launch = stream_ms, "stream launches"
    else:
        G = sb.copies * max(1, 48 // sb.copies)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(G):
                call(i, torch.cuda.current_stream(dev))
        g.replay()                                   # untimed: the graph's first replay
        reps = max(1, n_steps // G)
        e2e_ms = timed(lambda: [g.replay() for _ in range(reps)], reps * G)
        launch = f"CUDA graphs of {G} calls"
        torch.cuda.synchronize(dev)
        del g
    if dsa.dsa_check_device_error(ws, stream) != 0:
        raise RuntimeError(f"device error in the end-to-end loop ({wl.name})")
    return {"value": wl.n_q / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "api": "dsa_decode_step_host",
            "launch": launch, "stream_calls_ms_per_step": stream_ms}


def other_config(dsa, name, dev, stream, no_graph, pg, local, world, peaks, peak_src):
    """One more workload of the suite, timed like the headline (graph replay,
    rotated copies, clocks sampled): step time, throughput, the dominant
    launch's roofline."""
    import torch
    import workloads

    wl = workloads.named(name)
    sb = StepBench(dsa, wl, dev, stream, no_graph)
    sb.prepare(5)
    steps = agree_steps(pg, sb.calibrate(1.0), dev)
    ms, clk = sb.timed(steps, pg, local)
    fused, sel_ms, idx_ms = dominant_launch(dsa, wl, sb.sh, sb.b, sb.d, sb.keys, sb.copies, stream,
                                            max(10, min(steps, 200)))
    ms, sel_ms, idx_ms = max_over_ranks(pg, [ms, sel_ms, idx_ms], dev)
    per = ms / steps
    ent = {"unit": UNIT, "steps": steps, "ms_per_step": per, "dtype": wl.dtype,
           "config": workload_config(wl, world), "launch": sb.launch_mode,
           "gpu_launches": sb.plan["kernel_launches"] * steps, "plan": sb.plan, "clocks": clk}
    ent.update(step_metrics(wl, per, world, peaks))
    ent["roofline"] = roofline_of(wl, fused, sel_ms, idx_ms, peaks, peak_src)
    e2e = time_e2e(dsa, sb, max(20, steps // 2), no_graph)
    e2e["ms_per_step"] = max_over_ranks(pg, [e2e["ms_per_step"]], dev)[0]
    e2e["value"] = job_throughput(world, wl.n_q, e2e["ms_per_step"])
    ent["e2e"] = e2e
    sb.release()
    del sb
    ent["projections"] = time_projections(dsa, wl, dev, stream, peaks, peak_src)
    return ent


def run_ours(args):
    import torch

    import deepseek_sparse_attention_gb300 as dsa
    from deepseek_sparse_attention_gb300 import build as dsa_build
    import workloads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    if rank == 0:
        dsa_build.build()
    if pg:
        pg.barrier()
    dsa.load()

    wl = workloads.named(args.workload)
    stream = torch.cuda.current_stream(dev)
    sb = StepBench(dsa, wl, dev, stream, args.no_graph)
    sh, b, d, keys, caches, copies = sb.sh, sb.b, sb.d, sb.keys, sb.caches, sb.copies
    out, lse, idx, n_sel, ws = sb.out, sb.lse, sb.idx, sb.n_sel, sb.ws
    warm = args.warmup if args.warmup is not None else 20
    sb.prepare(warm, args.steps)
    launch_mode, plan = sb.launch_mode, sb.plan
    # default step count: about two seconds of timed work
    steps = args.steps if args.steps is not None else sb.calibrate(2.0)
    steps = agree_steps(pg, steps, dev)
    ms, clk = sb.timed(steps, pg, local)

    fused, sel_ms, idx_ms = dominant_launch(dsa, wl, sh, b, d, keys, copies, stream,
                                            max(10, min(steps, 2000)))
    # k-pool workloads: the pool-key compression of every pool of the
    # workload's sequences (q_len = kv_len: a prefill's worth of cells, seeded
    # synthetic [key | gate] cells and slot embedding), timed alone
    pool = None
    if wl.kpool > 1:
        gen = torch.Generator(device=dev).manual_seed(wl.seed + 4242)
        n_rows = sum(wl.kv_lens)
        cells = torch.randn((n_rows, 2 * wl.idx_dim), generator=gen, device=dev).to(keys[0].dtype)
        pos = 0.5 * torch.randn((wl.kpool, wl.idx_dim), generator=gen, device=dev)
        pkeys = torch.empty_like(keys[0])
        bp = dsa.make_batch(d["row_off"], d["key_off"], d["row_off"], n_rows, max(wl.kv_lens),
                            max(wl.kv_lens), n_rows, sum(wl.key_counts()))
        ws_p = dsa.alloc_workspace(sh, bp, dsa.OP_POOL_COMPRESS, dev)
        pc_ms = graph_time_ms(lambda i: dsa.dsa_pool_compress(sh, bp, cells, pos, pkeys, ws_p),
                              10, stream)
        if dsa.dsa_check_device_error(ws_p, stream) != 0:
            raise RuntimeError("device error in the pool compression loop")
        n_pools = sum(L // wl.kpool for L in wl.kv_lens)
        esz = cells.element_size()
        pc_bytes = n_pools * (wl.kpool * 2 * wl.idx_dim + wl.idx_dim) * esz + pos.numel() * 4
        pool = {"kernel": "pool_compress", "launch_us": pc_ms * 1e3, "pools": n_pools,
                "work": "every pool of the workload's sequences: cells [key | gate] -> pool keys",
                "bytes_per_launch": pc_bytes, "achieved_gbs": pc_bytes / (pc_ms / 1e3) / 1e9}
        del cells, pkeys

    # token-mode workloads: the indexer key preparation (rope on the first 64
    # dims, base 8e6, then the Walsh-Hadamard rotation, rounded) of every key of
    # the workload from seeded synthetic float32 projections, timed alone
    prep = None
    if wl.kpool == 1:
        gen = torch.Generator(device=dev).manual_seed(wl.seed + 4343)
        n_keys = sum(wl.key_counts())
        # three copies of the projections (more than the L2 holds) in turn
        xks = [torch.randn((n_keys, wl.idx_dim), generator=gen, device=dev) for _ in range(3)]
        pk = torch.cat([torch.arange(L, device=dev, dtype=torch.int64) for L in wl.kv_lens])
        kout = torch.empty_like(keys[0])
        pr_ms = graph_time_ms(lambda i: dsa.dsa_index_prepare(sh, xks[i % 3], pk, 64, 8e6, kout),
                              21, stream)
        pr_bytes = n_keys * (wl.idx_dim * 4 + 8 + wl.idx_dim * kout.element_size())
        prep = {"kernel": "index_prepare", "launch_us": pr_ms * 1e3, "vectors": n_keys,
                "work": "every key of the workload: float32 projection -> rope, Hadamard, dtype",
                "bytes_per_launch": pr_bytes, "achieved_gbs": pr_bytes / (pr_ms / 1e3) / 1e9,
                "traffic": kernel_traffic("index_prepare", wl.name)}
        del xks, pk, kout

    # end to end through the public call fed from host memory
    e2e = None
    if not args.no_e2e:
        e2e = time_e2e(dsa, sb, max(200, min(steps, 20000)), args.no_graph)

    ms, idx_ms, sel_ms = max_over_ranks(pg, [ms, idx_ms, sel_ms], dev)
    if e2e is not None:
        e2e["ms_per_step"] = max_over_ranks(pg, [e2e["ms_per_step"]], dev)[0]
        e2e["value"] = job_throughput(world, wl.n_q, e2e["ms_per_step"])

    peaks, peak_src = measured_peaks()
    projections = time_projections(dsa, wl, dev, stream, peaks, peak_src)
    # the other workloads of the suite, each timed the same way
    configs = {}
    if not args.no_configs:
        names = [n for n in workloads.NAMES if n != wl.name]
        # the headline's inputs the CPU baseline reads stay; the rotated copies go
        host_d = {k: d[k] for k in ("q_idx", "w", "q_abs", "k_idx", "cache", "row_off",
                                    "key_off", "q_off")} if not args.no_cpu_baseline else None
        del keys, caches, d, out, lse, idx, n_sel, ws
        sb.release()
        del sb
        for name in names:
            try:
                configs[name] = other_config(dsa, name, dev, stream, args.no_graph, pg, local,
                                             world, peaks, peak_src)
            except (RuntimeError, dsa.DsaError) as exc:     # recorded, not hidden
                configs[name] = {"error": f"{type(exc).__name__}: {exc}"}
                torch.cuda.synchronize(dev)
        d = host_d

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return None

    per_step_ms = ms / steps
    work = algorithmic(wl)
    achieved_idx = work["index_launch_bytes"] / (idx_ms / 1e3) / 1e9
    sm = step_metrics(wl, per_step_ms, world, peaks)
    line = {
        "metric": METRIC, "value": sm["value"], "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": max(warm, 3), "ms_per_step": per_step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": workload_config(wl, world), "launch": launch_mode,
        "tokens_per_s": sm["tokens_per_s"],
        "step_hbm_gbs": sm["step_hbm_gbs"], "step_hbm_frac": sm["step_hbm_frac"],
        "step_tflops": sm["step_tflops"],
        "roofline": roofline_of(wl, fused, sel_ms, idx_ms, peaks, peak_src),
        "indexer_alone": {"kernel": "index_scores_tc", "launch_us": idx_ms * 1e3,
                          "bytes_per_launch": work["index_launch_bytes"],
                          "achieved_gbs": achieved_idx, "frac": achieved_idx / peaks["hbm_gbs"],
                          "traffic": kernel_traffic("index_scores_tc", wl.name)},
        "clocks": clk,
        "gpu_launches": plan["kernel_launches"] * steps,
        "plan": plan,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if prep is not None:
        prep["frac"] = prep["achieved_gbs"] / peaks["hbm_gbs"]
        prep["peak_source"] = f"{peak_src} hbm_gbs"
        line["index_prepare"] = prep
    if pool is not None:
        pool["frac"] = pool["achieved_gbs"] / peaks["hbm_gbs"]
        pool["peak_source"] = f"{peak_src} hbm_gbs"
        pool["traffic"] = kernel_traffic("pool_compress", wl.name)
        line["pool_compress"] = pool
    line["projections"] = projections
    if configs:
        line["configs"] = configs
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(wl, d, args.cpu_seconds, args.cpu_seconds / 3)
    if pg:
        pg.destroy_process_group()
    return line


def main(argv=None):
    args = parse_args(argv)
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
