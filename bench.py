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
                   help="target CPU work of the oracle baseline sample")
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

def oracle_sample(wl, d_host_fn, seconds: float, max_queries: int = 1 << 30):
    """Run the oracle over queries of the workload until `seconds` of wall time
    have passed (at least one query); returns (queries, elapsed, threads)."""
    import oracle

    oracle.build()
    done, t0 = 0, time.perf_counter()
    nq = wl.n_q
    while True:
        q = (done * 7919) % nq          # spread the sample over the batch
        args = d_host_fn(q)
        oracle.decode_step(*args)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds or done >= max_queries:
            return done, el, oracle.threads()


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
    per_copy = algorithmic(wl)["step_bytes"]
    copies = max(2, math.ceil(2 * L2_BYTES / max(per_copy, 1)))
    copies = min(copies, 8)
    d = workloads.make(wl, dev, copies=copies)
    sh = dsa.make_shape(wl.idx_heads, wl.idx_dim, wl.heads, wl.kv_lora, wl.rope, wl.top_k,
                        wl.kpool, wl.scale, wl.dtype)
    b = dsa.make_batch(d["row_off"], d["key_off"], d["q_off"], wl.n_q, max(wl.q_lens),
                       max(wl.kv_lens), sum(wl.kv_lens), sum(wl.key_counts()))
    ws = dsa.alloc_workspace(sh, b, dsa.OP_DECODE_STEP, dev)
    width = dsa.dsa_index_row_width(sh)
    plan = dsa.dsa_plan(sh, b, dsa.OP_DECODE_STEP)
    out = torch.empty((wl.n_q, wl.heads, wl.kv_lora), device=dev)
    lse = torch.empty((wl.n_q, wl.heads), device=dev)
    idx = torch.empty((wl.n_q, width), dtype=torch.int32, device=dev)
    n_sel = torch.empty(wl.n_q, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    keys, caches = d["k_idx_copies"], d["cache_copies"]

    def launch(i, st):
        c = i % copies
        dsa.dsa_decode_step(sh, b, d["q_idx"], d["w"], keys[c], d["q_abs"], caches[c], out, lse,
                            idx, n_sel, ws, st)

    def step(i):
        launch(i, stream)

    # default step count: about two seconds of timed work
    warm = args.warmup if args.warmup is not None else 20
    for i in range(max(warm, 3)):
        step(i)
    torch.cuda.synchronize(dev)
    if dsa.dsa_check_device_error(ws, stream) != 0:
        raise RuntimeError("device error during warm-up")
    # A decode loop replays its step from CUDA graphs (the launches of a step
    # and of consecutive steps then overlap through programmatic dependent
    # launch without host round trips): one graph of G steps over the input
    # copies in turn, and one single-step graph per copy for the remainder, so
    # that exactly K steps run.
    run_steps = None
    launch_mode = "stream launches"
    if not args.no_graph:
        G = copies * max(1, 12 // copies)
        g_all = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_all):
            for i in range(G):
                launch(i, torch.cuda.current_stream(dev))
        g_one = []
        for c in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                launch(c, torch.cuda.current_stream(dev))
            g_one.append(g)

        def run_steps(n):
            for _ in range(n // G):
                g_all.replay()
            for i in range(n % G):
                g_one[i % copies].replay()

        run_steps(G)                                 # untimed: the graphs' first replays
        torch.cuda.synchronize(dev)
        if dsa.dsa_check_device_error(ws, stream) != 0:
            raise RuntimeError("device error in the graph warm-up")
        launch_mode = f"CUDA graphs of {G} steps (+ single-step graphs for the remainder)"
    else:
        def run_steps(n):
            for i in range(n):
                step(i)

    if args.steps is None:
        t0 = time.perf_counter()
        run_steps(60)
        torch.cuda.synchronize(dev)
        per = (time.perf_counter() - t0) / 60
        steps = int(min(200000, max(20, 2.0 / max(per, 1e-7))))
    else:
        steps = args.steps
    steps = agree_steps(pg, steps, dev)

    clocks = ClockSampler(local)
    clocks.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run_steps(steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    if dsa.dsa_check_device_error(ws, stream) != 0:
        raise RuntimeError("device error during the timed region")

    # dominant kernel, timed alone on the same stream with the same rotation
    sb = torch.empty((wl.n_q, max(max(wl.kv_lens) // wl.kpool, 4)), device=dev)
    ld = sb.shape[1]
    ws_i = dsa.alloc_workspace(sh, b, dsa.OP_INDEX_SCORES, dev)
    n_idx = max(10, min(steps, 2000))
    for i in range(3):
        dsa.dsa_index_scores(sh, b, d["q_idx"], d["w"], keys[i % copies], sb, ld, ws_i, stream)
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0.record(stream)
    for i in range(n_idx):
        dsa.dsa_index_scores(sh, b, d["q_idx"], d["w"], keys[i % copies], sb, ld, ws_i, stream)
    k1.record(stream)
    torch.cuda.synchronize(dev)
    idx_ms = k0.elapsed_time(k1) / n_idx

    # steps 1 and 2 as the step runs them: one fused launch for small decode
    # batches, which is then the step's dominant kernel
    fused = dsa.dsa_plan(sh, b, dsa.OP_INDEX_SELECT)["kernel_launches"] == 1
    sel_ms = 0.0
    if fused:
        ws_s = dsa.alloc_workspace(sh, b, dsa.OP_INDEX_SELECT, dev)
        idx_s, nsel_s = torch.empty_like(idx), torch.empty_like(n_sel)
        for i in range(3):
            dsa.dsa_index_select(sh, b, d["q_idx"], d["w"], keys[i % copies], idx_s, nsel_s, ws_s,
                                 stream)
        k0.record(stream)
        for i in range(n_idx):
            dsa.dsa_index_select(sh, b, d["q_idx"], d["w"], keys[i % copies], idx_s, nsel_s, ws_s,
                                 stream)
        k1.record(stream)
        torch.cuda.synchronize(dev)
        sel_ms = k0.elapsed_time(k1) / n_idx
        if dsa.dsa_check_device_error(ws_s, stream) != 0:
            raise RuntimeError("device error in the fused selection loop")

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
        for i in range(3):
            dsa.dsa_pool_compress(sh, bp, cells, pos, pkeys, ws_p, stream)
        n_pc = 10
        k0.record(stream)
        for i in range(n_pc):
            dsa.dsa_pool_compress(sh, bp, cells, pos, pkeys, ws_p, stream)
        k1.record(stream)
        torch.cuda.synchronize(dev)
        if dsa.dsa_check_device_error(ws_p, stream) != 0:
            raise RuntimeError("device error in the pool compression loop")
        pc_ms = k0.elapsed_time(k1) / n_pc
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
        xk = torch.randn((n_keys, wl.idx_dim), generator=gen, device=dev)
        pk = torch.cat([torch.arange(L, device=dev, dtype=torch.int64) for L in wl.kv_lens])
        kout = torch.empty_like(keys[0])
        for i in range(3):
            dsa.dsa_index_prepare(sh, xk, pk, 64, 8e6, kout, stream)
        n_pr = 20
        k0.record(stream)
        for i in range(n_pr):
            dsa.dsa_index_prepare(sh, xk, pk, 64, 8e6, kout, stream)
        k1.record(stream)
        torch.cuda.synchronize(dev)
        pr_ms = k0.elapsed_time(k1) / n_pr
        pr_bytes = n_keys * (wl.idx_dim * 4 + 8 + wl.idx_dim * kout.element_size())
        prep = {"kernel": "index_prepare", "launch_us": pr_ms * 1e3, "vectors": n_keys,
                "work": "every key of the workload: float32 projection -> rope, Hadamard, dtype",
                "bytes_per_launch": pr_bytes, "achieved_gbs": pr_bytes / (pr_ms / 1e3) / 1e9}
        del xk, pk, kout

    # end to end through the public call: pinned host inputs in, result out
    e2e = None
    if not args.no_e2e:
        hq = {k: d[k].cpu().pin_memory() for k in ("q_idx", "w", "q_abs")}
        dq = {k: torch.empty_like(d[k]) for k in hq}
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_nsel = torch.empty(n_sel.shape, dtype=n_sel.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in hq.values())
        d2h = h_out.numel() * 4 + h_nsel.numel() * 4
        n_e2e = max(10, min(steps, 5000))
        torch.cuda.synchronize(dev)
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        for i in range(n_e2e):
            for k in hq:
                dq[k].copy_(hq[k], non_blocking=True)
            c = i % copies
            dsa.dsa_decode_step(sh, b, dq["q_idx"], dq["w"], keys[c], dq["q_abs"], caches[c], out,
                                lse, idx, n_sel, ws, stream)
            h_out.copy_(out, non_blocking=True)
            h_nsel.copy_(n_sel, non_blocking=True)
        x1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = x0.elapsed_time(x1) / n_e2e
        e2e = {"value": wl.n_q / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    ms, idx_ms, sel_ms = max_over_ranks(pg, [ms, idx_ms, sel_ms], dev)
    if e2e is not None:
        e2e["ms_per_step"] = max_over_ranks(pg, [e2e["ms_per_step"]], dev)[0]
        e2e["value"] = job_throughput(world, wl.n_q, e2e["ms_per_step"])

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return None

    per_step_ms = ms / steps
    work = algorithmic(wl)
    value = job_throughput(world, wl.n_q, per_step_ms)
    peaks, peak_src = measured_peaks()
    achieved_idx = work["index_launch_bytes"] / (idx_ms / 1e3) / 1e9
    if fused:
        dom = {"kernel": "index_select_fused", "ms": sel_ms,
               "bytes": work["index_launch_bytes"] + work["select_bytes"]}
    else:
        dom = {"kernel": "index_scores_tc", "ms": idx_ms, "bytes": work["index_launch_bytes"]}
    achieved = dom["bytes"] / (dom["ms"] / 1e3) / 1e9
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
        roof = {"bound": "hbm", "kernel": dom["kernel"], "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "bytes_per_launch": dom["bytes"],
                "peak_source": f"{peak_src} hbm_gbs"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = kernel_traffic(dom["kernel"], wl.name)
    roof["launch_us"] = dom["ms"] * 1e3
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": max(warm, 3), "ms_per_step": per_step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": dict(workload_config(wl, world), launch=launch_mode),
        "tokens_per_s": work["scored_keys"] / (per_step_ms / 1e3) * world,
        "step_hbm_gbs": work["compulsory_bytes"] / (per_step_ms / 1e3) / 1e9,
        "step_hbm_frac": work["compulsory_bytes"] / (per_step_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
        "step_tflops": work["flops"] / (per_step_ms / 1e3) / 1e12,
        "roofline": roof,
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
    if not args.no_cpu_baseline:
        n, el, threads = oracle_sample(wl, host_query_args(wl, d), args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": n / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} quer{'y' if n == 1 else 'ies'} of the {wl.name} workload through the "
                      f"oracle (double precision, {threads} OpenMP threads), {el:.1f} s"}
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
