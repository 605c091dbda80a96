#!/usr/bin/env python3
"""Benchmark of the load-balanced paged GQA decode-attention step on GB300.

One step = plan (task map from device lengths) + persistent attention +
combine over one synthetic decode batch resident in HBM. Default workload:
the mixed-length Hy3-shape batch (64 requests, lengths log-uniform in
[128, 65536], 64 query / 8 KV heads, head dim 128, BF16 KV, page size 64).

Prints one JSON line. `value` = effective KV GB/s = (live K+V bytes + Q bytes
+ split-partial bytes written and read) / device time per step. The KV stream
(2.4 GB) is larger than L2, so no flush is needed between steps. The line's
`configs` record repeats the measurement on each of the five scope workloads
(tiny, uniform, mixed, skew, e4m3): medians of 200 CUDA-graph replays of the
step and of 200 attention launches (L2 flushed before each call where the KV
fits in it), the attention kernel's fraction of the measured and nominal HBM
peaks, the static split-KV schedule (S = 16) of the same kernel, and the
oracle's time on the host cores (also single-threaded for tiny and uniform).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload mixed|uniform|skew|fp8|tiny]

--impl reference times the float64 CPU oracle on the host cores (a bounded
sample of the same workload, scaled to the whole batch).
Under torchrun (N > 1) each rank runs its own batch (weak scaling, no
collective on the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step and effective KV GB/s (fraction of GB300 HBM peak)"
UNIT = "GB/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixed")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="total oracle time of the --impl reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-static", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches only")
    ap.add_argument("--no-prologue", action="store_true", help="skip the fused-prologue timing")
    ap.add_argument("--no-multi-token", action="store_true", help="skip the q_len > 1 timings")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload record (tiny, uniform, mixed, skew, fp8)")
    ap.add_argument("--prologue-only", action="store_true",
                    help="time only the fused prologue for the workload's head shape and cache dtype "
                         "(a decode step and an 8192-token prefill; no attention batch is created)")
    ap.add_argument("--prologue-reps", type=int, default=200, help="graph replays per prologue timing")
    ap.add_argument("--no-chain", action="store_true",
                    help="skip the plan -> prologue -> attention -> combine layer timing")
    ap.add_argument("--num-ctas", type=int, default=0,
                    help="CTAs the task map is planned for (0: the workload's stated count, else the "
                         "library's suggestion for the batch, hpc_decode_suggest_num_ctas)")
    ap.add_argument("--engine", choices=["auto", "mma_sync", "tcgen05"], default="auto",
                    help="attention kernel for workloads with several new tokens per request "
                         "(<workload>:qlen<N>); auto = the library's own choice")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist if world > 1 else None


def max_over_ranks(x: float, dist, device) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_workload(w, rank):
    from dataclasses import replace
    return w if rank == 0 else replace(w, seed=w.seed + 1000 * rank)


def step_bytes(lens, w, n_splits):
    """Algorithmic bytes of one step: live K+V (+e4m3 scales), Q (+ its scales),
    and the split partials (8 x (128 + 1) float32 per split, written once and
    read once)."""
    from load_balanced_paged_02_gb300 import workloads as wl
    kv = wl.kv_bytes(lens, w.num_kv_heads, w.kv_dtype)
    rows = len(lens) * w.q_len * w.num_q_heads
    q = rows * ((128 + 4) if w.q_dtype == "fp8" else 256)
    part = n_splits * w.q_len * 8 * 129 * 4
    pages = int(wl.chunk_counts(lens).sum()) * 4
    return dict(kv=kv, q=q, partials_rw=2 * part, metric=kv + q + 2 * part,
                attn=kv + q + part + pages, out=rows * 128 * 2)


class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def __enter__(self):
        self.t_begin = self.t_end = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        """Median SM clock and active throttle reasons over the samples taken
        between mark('t_begin') and mark('t_end') (all samples if too few)."""
        import datetime
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        parsed = []
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                parsed.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        inside = [p for p in parsed if self.t_begin and self.t_end and self.t_begin <= p[0] <= self.t_end]
        use = inside if len(inside) >= 3 else parsed
        for _, cur, mxv, flags in use:
            sm.append(cur)
            mx = mxv
            for name, v in zip(names, flags):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "window": "timed region" if use is inside else "whole run"}


NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (~8 TB/s)
L2_BYTES = 129 * 1024 * 1024


def workload_config(w):
    """The line's `config`: what identifies the workload, the same in both arms."""
    from load_balanced_paged_02_gb300 import workloads as wl
    lens = wl.draw_lengths(w)
    kv = wl.kv_bytes(lens, w.num_kv_heads, w.kv_dtype)
    return {"workload": w.name, "detail": w.note, "batch": w.batch, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "kv_dtype": "e4m3" if w.kv_dtype == "fp8" else "bf16",
            "q_dtype": "e4m3" if w.q_dtype == "fp8" else "bf16", "q_len": w.q_len,
            "live_tokens": int(np.maximum(lens, 0).sum()), "kv_bytes": int(kv),
            "l2": ("inputs larger than L2 (no flush)" if kv > L2_BYTES else
                   "inputs smaller than L2: the main loop does not flush; the configs record flushes")}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = {
    "decode_attn_kernel": ("attn.cu", "attn_common.cuh", "hpc_internal.cuh"),
    "decode_attn_mt_kernel": ("attn_mt.cu", "attn_common.cuh", "hpc_internal.cuh"),
    "decode_attn_tc_kernel": ("attn_tc.cu", "attn_common.cuh", "hpc_internal.cuh"),
}


def attn_kernel_name(kv_dtype, q_len, engine=None):
    """The attention kernel launched for q_len new tokens: the pinned engine
    (several new tokens only), else the library's automatic choice."""
    from load_balanced_paged_02_gb300 import binding as hb
    if q_len > 1 and engine is not None:
        return "decode_attn_tc_kernel" if engine == hb.ENGINE_TCGEN05 else "decode_attn_mt_kernel"
    if hb.auto_engine(kv_dtype, q_len) == hb.ENGINE_TCGEN05:
        return "decode_attn_tc_kernel"
    return "decode_attn_kernel" if q_len == 1 else "decode_attn_mt_kernel"


def kernel_source_hash(kernel="decode_attn_kernel"):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "load_balanced_paged_02_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, dtype, kernel="decode_attn_kernel"):
    """DRAM bytes per attention launch from a committed ncu summary, if it was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "attn_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(f"{workload}:{dtype}")
    if not rec or rec.get("kernel_hash") != kernel_source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- CPU oracle leg

def oracle_sample(case, w, seconds, seed=99):
    """Time the float64 oracle on a bounded sample of the workload and scale its
    rate to the whole batch. Rows (request, query head) are taken request by
    request in a seeded order (cycling over the batch if time allows) until
    about `seconds` of oracle time is spent. Returns (seconds per full step,
    threads used, text describing the sample)."""
    import oracle
    from load_balanced_paged_02_gb300 import workloads as wl
    lens = np.maximum(case["seq_lens"].cpu().numpy().astype(np.int64), 0)
    Hq = w.num_q_heads * w.q_len  # rows per request: (new token, query head)
    total = float(lens.sum()) * Hq
    order = [int(b) for b in np.random.default_rng(seed).permutation(len(lens)) if lens[b] > 0]
    spent, done, rows_done, k = 0.0, 0.0, 0, 0
    hosts = {}
    if total <= 4e6:
        # a small batch: whole-batch oracle calls, repeated within the budget
        host = wl.to_numpy_case(case)
        while spent < seconds or done == 0:
            t0 = time.perf_counter()
            oracle.attn_rows(host)
            spent += time.perf_counter() - t0
            done += total
            rows_done += len(lens) * Hq
        order = []
    while spent < seconds and order:
        b = order[k % len(order)]
        k += 1
        if b not in hosts:
            hosts[b] = wl.to_numpy_case(case, requests=[b])
        # whole request if it fits the remaining budget, else a prefix of its heads
        per_row = spent / done if done else None
        nh = Hq
        if per_row is not None:
            nh = int(max(1, min(Hq, (seconds - spent) / max(per_row * lens[b], 1e-12))))
        rows = [(0, h) for h in range(nh)]
        t0 = time.perf_counter()
        oracle.attn_rows(hosts[b], rows)
        spent += time.perf_counter() - t0
        done += float(lens[b]) * nh
        rows_done += nh
    full = spent * total / max(done, 1.0)
    text = (f"{rows_done} (request, query head{', new token' if w.q_len > 1 else ''}) rows covering "
            f"{int(done)} token-row pairs "
            f"({done / total:.2f} x the batch's {int(total)}), {spent:.1f} s of oracle time, "
            f"rate scaled to one whole batch")
    return full, oracle.num_threads(), text


def prologue_timing(w, dev, n_rep=200):
    """The fused prologue (hpc_rope_norm) for this workload's head shape: one
    decode step (one token per request) and a prefill-sized pass of 8192
    tokens, each replayed from a CUDA graph. Output dtypes follow the
    workload: e4m3 cache -> e4m3 K/V and e4m3 Q."""
    import torch
    from load_balanced_paged_02_gb300 import binding as hb
    from load_balanced_paged_02_gb300 import workloads as wl
    fp8 = w.kv_dtype == "fp8"
    out = {}
    peak, _ = measured_peaks()
    for label, T in (("decode", w.batch), ("prefill_8192", 8192)):
        pos = np.arange(T, dtype=np.int32) % 4096
        pc = wl.make_prologue_case(pos, w.num_q_heads, w.num_kv_heads, seed=77, device=dev, max_pos=4096,
                                   slots=np.arange(T, dtype=np.int32))
        pages = (T + 63) // 64
        kv_dt = torch.float8_e4m3fn if fp8 else torch.bfloat16
        k = torch.zeros((pages, 64, w.num_kv_heads, 128), dtype=kv_dt, device=dev)
        v = torch.zeros_like(k)
        ks = torch.zeros((pages, w.num_kv_heads, 64), dtype=torch.float32, device=dev) if fp8 else None
        vs = torch.zeros_like(ks) if fp8 else None
        q = torch.empty((T, w.num_q_heads, 128), dtype=kv_dt, device=dev)
        qs = torch.empty((T, w.num_q_heads), dtype=torch.float32, device=dev) if fp8 else None

        def call():
            hb.hpc_rope_norm(pc["qkv"], pc["positions"], pc["cos_sin"], pc["q_weight"], pc["k_weight"],
                             pc["slots"], q, k, v, q_scale=qs, k_scale=ks, v_scale=vs, eps=pc["eps"],
                             num_kv_heads=w.num_kv_heads)
        call()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n_rep):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        us = 1e3 * a.elapsed_time(b) / n_rep
        e = 1 if fp8 else 2
        per_row_out = 128 * e + (4 if fp8 else 0)
        byt = (T * (w.num_q_heads + 2 * w.num_kv_heads) * 256 + T * (512 + 8)
               + T * (w.num_q_heads + 2 * w.num_kv_heads) * per_row_out)
        gbs = byt / (us * 1e-6) / 1e9
        out[label] = {"tokens": T, "us": us, "bytes": byt, "GB/s": gbs, "frac": gbs / peak}
    return out


def chained_layer_timing(w, case, C, dev, n_rep=200, rounds=5):
    """One decode layer as a caller chains it: plan, the fused prologue writing
    each request's new token (position L - 1) into the cache and emitting Q
    (e4m3 with scales for an e4m3 cache), attention, combine; replayed from a
    CUDA graph, with the attention kernel waiting for the prologue before any
    load, and with HPC_ATTN_EARLY_KV (KV of chunks without the new token
    gathered while the prologue runs). The two graphs alternate over
    ``rounds`` blocks of ``n_rep`` replays; the medians of the blocks are
    reported."""
    import torch
    from load_balanced_paged_02_gb300 import binding as hb
    from load_balanced_paged_02_gb300 import workloads as wl
    fp8 = w.kv_dtype == "fp8"
    B, Hq, Hkv = w.batch, w.num_q_heads, w.num_kv_heads
    lens = case["seq_lens"].cpu().numpy().astype(np.int64)
    pt = case["page_table"].cpu().numpy()
    pos = np.maximum(lens - 1, 0).astype(np.int32)
    slots = np.where(lens > 0, pt[np.arange(B), pos // 64] * 64 + pos % 64, -1).astype(np.int32)
    pc = wl.make_prologue_case(pos, Hq, Hkv, seed=91, device=dev, max_pos=int(pos.max()) + 1, slots=slots)
    q = torch.empty((B, Hq, 128), dtype=torch.float8_e4m3fn if fp8 else torch.bfloat16, device=dev)
    qs = torch.empty((B, Hq), dtype=torch.float32, device=dev) if fp8 else None
    plan = hb.Plan(B, Hkv, C, dev)
    so, sl = hb.split_buffers(plan)
    out = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)

    def layer(early):
        hb.hpc_decode_plan(case["seq_lens"], Hkv, C, w.min_chunks, plan=plan)
        hb.hpc_rope_norm(pc["qkv"], pc["positions"], pc["cos_sin"], pc["q_weight"], pc["k_weight"], pc["slots"],
                         q, case["k_cache"], case["v_cache"], q_scale=qs, k_scale=case["k_scale"],
                         v_scale=case["v_scale"], eps=pc["eps"], num_kv_heads=Hkv,
                         num_pages=case["num_pages"])
        hb.hpc_decode_attn(q, case["k_cache"], case["v_cache"], case["page_table"], case["seq_lens"], plan, so,
                           sl, case["k_scale"], case["v_scale"], num_pages=case["num_pages"], q_scale=qs,
                           early_kv=early)
        hb.hpc_decode_combine(plan, so, sl, out, lse, Hkv)
    graphs = {}
    for early in (False, True):
        for _ in range(3):
            layer(early)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer(early)
        g.replay()
        graphs[early] = g
    torch.cuda.synchronize()
    if hb.hpc_decode_read_error(plan) != 0:
        raise RuntimeError("chained layer: device error word set")
    st = torch.cuda.current_stream(dev)
    blocks = {False: [], True: []}
    for _ in range(rounds):
        for early in (False, True):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            for _ in range(n_rep):
                graphs[early].replay()
            b.record(st)
            torch.cuda.synchronize()
            blocks[early].append(1e3 * a.elapsed_time(b) / n_rep)
    wait_us, early_us = float(np.median(blocks[False])), float(np.median(blocks[True]))
    del graphs, so, sl
    return {"layer": "plan -> hpc_rope_norm -> attention -> combine (cuda graph)",
            "query": "e4m3 + scales" if fp8 else "bf16",
            "us_wait_first": wait_us, "us_early_kv": early_us, "saved_us": wait_us - early_us,
            "blocks_us": {"wait_first": blocks[False], "early_kv": blocks[True]}}


# ---------------------------------------------------------------- arms

def multi_token_timing(w, case, plan, C, dev, q_lens=(2, 6), n_rep=100):
    """Attention + combine for q_len new tokens per request (causal verify rows)
    on the workload's own batch, cache and task map, replayed from a CUDA
    graph. Bytes: live K/V, the q_len query rows, the partials written and the
    page ids (the attention kernel's algorithmic bytes)."""
    import torch
    from dataclasses import replace
    from load_balanced_paged_02_gb300 import binding as hb
    peak, _ = measured_peaks()
    lens = case["seq_lens"].cpu().numpy()
    n_splits = int(plan.buf[3].item())
    Hkv = w.num_kv_heads
    res = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)
    for Q in q_lens:
        wq = replace(w, q_len=Q)
        q = torch.randn((w.batch, Q, w.num_q_heads, 128), generator=gen, device=dev).to(torch.bfloat16)
        so, sl = hb.split_buffers(plan, q_len=Q)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)

        def layer():
            hb.hpc_decode_attn(q, case["k_cache"], case["v_cache"], case["page_table"], case["seq_lens"], plan,
                               so, sl, case["k_scale"], case["v_scale"], num_pages=case["num_pages"])
            hb.hpc_decode_combine(plan, so, sl, out, lse, Hkv)
        for _ in range(3):
            layer()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer()
        g.replay()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream(dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_rep)]
        for e in ev:  # eager, per-kernel events
            e[0].record(st)
            hb.hpc_decode_attn(q, case["k_cache"], case["v_cache"], case["page_table"], case["seq_lens"], plan,
                               so, sl, case["k_scale"], case["v_scale"], num_pages=case["num_pages"])
            e[1].record(st)
            hb.hpc_decode_combine(plan, so, sl, out, lse, Hkv)
            e[2].record(st)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(n_rep):
            g.replay()
        b.record(st)
        torch.cuda.synchronize()
        attn_us = 1e3 * float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
        comb_us = 1e3 * float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
        layer_us = 1e3 * a.elapsed_time(b) / n_rep
        byt = step_bytes(lens, wq, n_splits)
        gbs = byt["attn"] / (attn_us * 1e-6) / 1e9
        flops = 4.0 * float(np.maximum(lens, 0).sum()) * w.num_q_heads * Q * 128  # QK^T and PV
        kvd = hb.kv_dtype_of(case["k_cache"])
        kname = attn_kernel_name(kvd, Q)
        res[f"q_len_{Q}"] = {"attn_us": attn_us, "combine_us": comb_us, "layer_graph_us": layer_us,
                             "attn_gbs": gbs, "frac_of_peak": gbs / peak,
                             "mma_tflops": flops / (attn_us * 1e-6) / 1e12,
                             "algorithmic_bytes_per_launch": byt["attn"], "kernel": kname,
                             "traffic": recorded_traffic(f"{w.name}:qlen{Q}",
                                                         "bf16" if kvd == hb.KV_BF16 else "e4m3", kname)}
        del so, sl, out, lse, q, g
    return res


def _median_us(fn, n, stream, flush=None):
    """Median device time of n calls of fn, each bracketed by its own CUDA
    events on ``stream``; ``flush`` (a buffer larger than L2) is rewritten
    before every call, outside the events."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in ev:
        if flush is not None:
            flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return 1e3 * float(np.median([a.elapsed_time(b) for a, b in ev]))


CONFIG_WORKLOADS = ("tiny", "uniform", "mixed", "skew", "fp8", "short")


def config_record(name, dev, n_rep=200, cpu_seconds=2.0, single_thread=False):
    """One of the five scope workloads at N = 1: the step (plan + attention +
    combine) captured as a CUDA graph, its median over n_rep replays; the
    attention kernel alone (median of n_rep eager launches) against the HBM
    roofline; the static split-KV schedule of the same kernel (S = 16); and the
    float64 oracle on the host cores (a bounded sample, scaled to the batch).
    Workloads whose KV fits in L2 flush it before every timed call."""
    import torch
    from load_balanced_paged_02_gb300 import binding as hb
    from load_balanced_paged_02_gb300 import workloads as wl
    w = wl.by_name(name)
    case = wl.make_case(w, device=dev)
    kvd = hb.kv_dtype_of(case["k_cache"])
    C = w.num_ctas or hb.suggest_num_ctas(case["seq_lens"], w.num_kv_heads, kvd, w.min_chunks)
    Hkv = w.num_kv_heads
    lens = case["seq_lens"].cpu().numpy()
    stream = torch.cuda.current_stream(dev)
    plan = hb.Plan(w.batch, Hkv, C, dev)
    hb.hpc_decode_plan(case["seq_lens"], Hkv, C, w.min_chunks, plan=plan)
    splan = hb.hpc_decode_plan_static(case["seq_lens"], Hkv, w.static_splits)
    so, sl = hb.split_buffers(plan)
    sso, ssl = hb.split_buffers(splan)
    out = torch.empty(case["q"].shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(case["q"].shape[:-1], dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    n_splits, s_splits = int(plan.buf[3].item()), int(splan.buf[3].item())
    byt = step_bytes(lens, w, n_splits)
    flush = None
    if byt["kv"] <= L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def attn(pl, a, b):
        hb.hpc_decode_attn(case["q"], case["k_cache"], case["v_cache"], case["page_table"], case["seq_lens"], pl,
                           a, b, case["k_scale"], case["v_scale"], num_pages=case["num_pages"],
                           q_scale=case["q_scale"])

    def step():
        hb.hpc_decode_plan(case["seq_lens"], Hkv, C, w.min_chunks, plan=plan)
        attn(plan, so, sl)
        hb.hpc_decode_combine(plan, so, sl, out, lse, Hkv)

    def sstep():
        hb.hpc_decode_plan_static(case["seq_lens"], Hkv, w.static_splits, plan=splan)
        attn(splan, sso, ssl)
        hb.hpc_decode_combine(splan, sso, ssl, out, lse, Hkv)

    graphs = []
    for fn in (step, sstep):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        graphs.append(g)
    torch.cuda.synchronize()
    if hb.hpc_decode_read_error(plan) != 0 or hb.hpc_decode_read_error(splan) != 0:
        raise RuntimeError(f"{name}: device error word set")
    step_us = _median_us(graphs[0].replay, n_rep, stream, flush)
    static_us = _median_us(graphs[1].replay, n_rep, stream, flush)
    attn_us = _median_us(lambda: attn(plan, so, sl), n_rep, stream, flush)
    peak, peak_kind = measured_peaks()
    gbs = byt["attn"] / (attn_us * 1e-6) / 1e9
    rec = {"detail": w.note, "num_ctas": C, "min_chunks": w.min_chunks, "splits": n_splits,
           "replays": n_rep, "l2": "flushed before every call" if flush is not None else "inputs larger than L2",
           "step_us_median": step_us, "value_GBps": byt["metric"] / (step_us * 1e-6) / 1e9,
           "attn_us_median": attn_us, "attn_algorithmic_bytes": byt["attn"], "attn_GBps": gbs,
           "frac_of_measured": gbs / peak, "measured_peak": peak, "peak_kind": peak_kind,
           "frac_of_nominal": gbs / NOMINAL_HBM_GBS,
           "static_split_kv": {"num_splits": w.static_splits, "splits": s_splits, "step_us_median": static_us,
                               "balanced_speedup": static_us / step_us}}
    del graphs, so, sl, sso, ssl
    if cpu_seconds > 0:
        import oracle
        full_s, cores, text = oracle_sample(case, w, cpu_seconds)
        rec["oracle"] = {"ms_per_step": full_s * 1e3, "value_GBps": byt["metric"] / full_s / 1e9,
                         "threads": cores, "sample": text}
        if single_thread:
            prev = oracle.num_threads()
            oracle.set_num_threads(1)
            try:
                full_s, cores, text = oracle_sample(case, w, cpu_seconds)
            finally:
                oracle.set_num_threads(prev)
            rec["oracle_1_thread"] = {"ms_per_step": full_s * 1e3, "value_GBps": byt["metric"] / full_s / 1e9,
                                      "threads": cores, "sample": text}
    del case, flush
    torch.cuda.empty_cache()
    return rec


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    import torch
    import oracle
    from load_balanced_paged_02_gb300 import workloads as wl
    oracle.build()
    w = wl.by_name(args.workload)
    case = wl.make_case(w, device="cpu")
    lens = case["seq_lens"].numpy()
    byt = step_bytes(lens, w, 0)
    # every step is a bounded sample; the whole run stays within --ref-seconds
    per_step = max(0.02, args.ref_seconds / max(args.steps + args.warmup, 1))
    times = []
    sample = None
    for k in range(args.warmup + args.steps):
        full, cores, sample = oracle_sample(case, w, per_step, seed=99 + k)
        if k >= args.warmup:
            times.append(full)
    t = float(np.mean(times))
    value = byt["metric"] / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")

    from load_balanced_paged_02_gb300 import _build
    from load_balanced_paged_02_gb300 import binding as hb
    from load_balanced_paged_02_gb300 import workloads as wl
    _build.build()
    hb.lib()
    if args.prologue_only:
        w = wl.by_name(args.workload)
        if rank == 0:
            print(json.dumps({"workload": w.name, "prologue": prologue_timing(w, dev, n_rep=args.prologue_reps)}),
                  flush=True)
        return 0

    w = rank_workload(wl.by_name(args.workload), rank)
    case = wl.make_case(w, device=dev)
    kvd = hb.kv_dtype_of(case["k_cache"])
    # the CTA count a workload states (tiny: 16, uniform: 148), else the library's
    # suggestion for the batch (hpc_decode_suggest_num_ctas); --num-ctas overrides both
    C = args.num_ctas if args.num_ctas > 0 else (
        w.num_ctas or hb.suggest_num_ctas(wl.draw_lengths(w), w.num_kv_heads, kvd, w.min_chunks, w.q_len))
    eng = {"auto": None, "mma_sync": hb.ENGINE_MMA_SYNC, "tcgen05": hb.ENGINE_TCGEN05}[args.engine]
    if w.q_len == 1:
        eng = None  # one new token: hpc_decode_attn's kernel
    Hkv = w.num_kv_heads
    lens = case["seq_lens"].cpu().numpy()
    stream = torch.cuda.current_stream(dev)

    plan = hb.Plan(w.batch, Hkv, C, dev)
    hb.hpc_decode_plan(case["seq_lens"], Hkv, C, w.min_chunks, plan=plan)
    so, sl = hb.split_buffers(plan, q_len=w.q_len)
    out = torch.empty(case["q"].shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(case["q"].shape[:-1], dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    n_splits = int(plan.buf[3].item())
    byt = step_bytes(lens, w, n_splits)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        hb.hpc_decode_plan(case["seq_lens"], Hkv, C, w.min_chunks, plan=plan)
        if ev is not None:
            ev[1].record(stream)
        hb.hpc_decode_attn(case["q"], case["k_cache"], case["v_cache"], case["page_table"],
                           case["seq_lens"], plan, so, sl, case["k_scale"], case["v_scale"],
                           num_pages=case["num_pages"], q_scale=case["q_scale"], engine=eng)
        if ev is not None:
            ev[2].record(stream)
        hb.hpc_decode_combine(plan, so, sl, out, lse, Hkv)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if hb.hpc_decode_read_error(plan) != 0:
        raise RuntimeError("device error word set during warm-up")
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()

    # The whole step captured once as a CUDA graph (how a serving engine
    # replays decode steps); replays re-run plan, attention and combine.
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        # one layer of a step: attention + combine on the step's task map, which
        # the pages build once per step and reuse for every layer
        layer_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(layer_graph):
            hb.hpc_decode_attn(case["q"], case["k_cache"], case["v_cache"], case["page_table"],
                               case["seq_lens"], plan, so, sl, case["k_scale"], case["v_scale"],
                               num_pages=case["num_pages"], q_scale=case["q_scale"], engine=eng)
            hb.hpc_decode_combine(plan, so, sl, out, lse, Hkv)
        for _ in range(3):
            graph.replay()
            layer_graph.replay()
        torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_stop, g_start, g_stop = (torch.cuda.Event(enable_timing=True) for _ in range(4))
    with ClockSampler(local) as clk:
        clk.mark("t_begin")
        # eager launches, with events around every kernel (per-kernel times)
        t_start.record(stream)
        for k in range(args.steps):
            step(evs[k])
        t_stop.record(stream)
        # graph replays of the same step (the step time reported as the value)
        if graph is not None:
            g_start.record(stream)
            for k in range(args.steps):
                graph.replay()
            g_stop.record(stream)
        torch.cuda.synchronize()
        clk.mark("t_end")
    layer_us = None
    if graph is not None:
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_layer = max(10, args.steps // 3)
        l0.record(stream)
        for _ in range(n_layer):
            layer_graph.replay()
        l1.record(stream)
        torch.cuda.synchronize()
        layer_us = 1e3 * l0.elapsed_time(l1) / n_layer
    eager_ms = t_start.elapsed_time(t_stop) / args.steps
    graph_ms = g_start.elapsed_time(g_stop) / args.steps if graph is not None else None
    plan_us = 1e3 * float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    attn_us = 1e3 * float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    comb_us = 1e3 * float(np.mean([e[2].elapsed_time(e[3]) for e in evs]))
    ms_step = max_over_ranks(graph_ms if graph_ms is not None else eager_ms, dist, dev)
    if dist is not None:
        dist.barrier()

    peak, peak_kind = measured_peaks()
    units_all = world * byt["metric"]
    value = units_all / (ms_step * 1e-3) / 1e9
    attn_gbs = byt["attn"] / (attn_us * 1e-6) / 1e9

    kname = attn_kernel_name(kvd, w.q_len, eng)
    result = None
    if rank == 0:
        clocks = clk.summary()
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if kvd == hb.KV_BF16 else ("e4m3 (q and kv)" if w.q_dtype == "fp8" else "e4m3 kv, bf16 q"),
            "data": "synthetic",
            "config": workload_config(w),
            "breakdown": {"num_ctas": C, "min_chunks": w.min_chunks,
                          "engine": args.engine if w.q_len > 1 else "one-token kernel",
                          "splits": n_splits, "bytes_per_step": byt,
                          "step": "cuda graph replay" if graph is not None else "eager launches",
                          "us_per_step": {"plan": plan_us, "attn": attn_us, "combine": comb_us,
                                          "eager_total": eager_ms * 1e3,
                                          "graph_total": graph_ms * 1e3 if graph_ms is not None else None,
                                          "layer_attn_combine": layer_us}},
            "roofline": {"bound": "hbm", "achieved": attn_gbs, "peak": peak, "unit": "GB/s",
                         "frac": attn_gbs / peak, "peak_kind": peak_kind,
                         "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": attn_gbs / NOMINAL_HBM_GBS,
                         "traffic": recorded_traffic(w.name, "bf16" if kvd == hb.KV_BF16 else "e4m3", kname),
                         "kernel": kname, "algorithmic_bytes_per_launch": byt["attn"]},
            "gpu_launches": (6 if graph is not None else 3) * args.steps,
            "clocks": clocks,
        }

    # ---- static split-KV schedule of the same kernel (comparison)
    if not args.no_static and rank == 0:
        splan = hb.hpc_decode_plan_static(case["seq_lens"], Hkv, w.static_splits)
        sso, ssl = hb.split_buffers(splan, q_len=w.q_len)
        n_static = max(10, args.steps // 3)

        def sstep():
            hb.hpc_decode_plan_static(case["seq_lens"], Hkv, w.static_splits, plan=splan)
            hb.hpc_decode_attn(case["q"], case["k_cache"], case["v_cache"], case["page_table"],
                               case["seq_lens"], splan, sso, ssl, case["k_scale"], case["v_scale"],
                               num_pages=case["num_pages"], q_scale=case["q_scale"], engine=eng)
            hb.hpc_decode_combine(splan, sso, ssl, out, lse, Hkv)
        for _ in range(3):
            sstep()
        torch.cuda.synchronize()
        run = sstep
        if graph is not None:
            sgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(sgraph):
                sstep()
            sgraph.replay()
            run = sgraph.replay
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n_static):
            run()
        b.record(stream)
        torch.cuda.synchronize()
        sms = a.elapsed_time(b) / n_static
        sbytes = step_bytes(lens, w, int(splan.buf[3].item()))
        result["static_split_kv"] = {"num_splits": w.static_splits, "ms_per_step": sms,
                                     "value": sbytes["metric"] / (sms * 1e-3) / 1e9,
                                     "speedup_of_balanced": sms / ms_step}
        del sso, ssl, splan

    # ---- end to end through the C ABI with host buffers (bf16 query path)
    if not args.no_e2e and case["q_scale"] is not None and rank == 0:
        result["e2e"] = {"unavailable": "hpc_decode_step_host takes a bf16 query"}
    if not args.no_e2e and w.q_len > 1 and rank == 0:
        result["e2e"] = {"unavailable": "hpc_decode_step_host takes one new token per request"}
    if not args.no_e2e and case["q_scale"] is None and w.q_len == 1:
        B, Hq, D = case["q"].shape
        h_q = case["q"].cpu().pin_memory()
        h_sl = case["seq_lens"].cpu().pin_memory()
        h_pt = case["page_table"].cpu().pin_memory()
        h_out = torch.empty_like(h_q).pin_memory()
        h_lse = torch.empty((B, Hq), dtype=torch.float32).pin_memory()
        ws = torch.empty(hb.step_workspace_bytes(B, Hq, Hkv, h_pt.shape[1], C), dtype=torch.uint8,
                         device=dev)

        def estep():
            hb.hpc_decode_step_host(h_q, h_sl, h_pt, case["k_cache"], case["v_cache"], ws, h_out, h_lse,
                                    k_scale=case["k_scale"], v_scale=case["v_scale"], num_ctas=C,
                                    min_chunks_per_cta=w.min_chunks, num_pages=case["num_pages"])
            stream.synchronize()
        # the same step captured once (hpc_decode_step_graph_*): one launch per step,
        # the copies in and out still inside every replay
        sg = hb.StepGraph(h_q, h_sl, h_pt, case["k_cache"], case["v_cache"], ws, h_out, h_lse,
                          k_scale=case["k_scale"], v_scale=case["v_scale"], num_ctas=C,
                          min_chunks_per_cta=w.min_chunks, num_pages=case["num_pages"])

        def gstep():
            sg.launch(stream)
            stream.synchronize()
        n_e2e = max(10, args.steps // 3)

        def per_step_ms(fn):
            for _ in range(3):
                fn()
            t0 = time.perf_counter()
            for _ in range(n_e2e):
                fn()
            return (time.perf_counter() - t0) * 1e3 / n_e2e
        host_ms = max_over_ranks(per_step_ms(estep), dist, dev)
        e_ms = max_over_ranks(per_step_ms(gstep), dist, dev)
        sg.close()
        if rank == 0:
            h2d = h_q.numel() * 2 + h_sl.numel() * 4 + h_pt.numel() * 4
            d2h = h_out.numel() * 2 + h_lse.numel() * 4
            result["e2e"] = {"value": world * byt["metric"] / (e_ms * 1e-3) / 1e9, "unit": UNIT,
                             "ms_per_step": e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                             "api": "hpc_decode_step_graph_launch (captured hpc_decode_step_host on pinned, "
                                    "mapped host buffers: a staging kernel reads q/seq_lens/page_table over "
                                    "the host link, the combine writes out/lse into host memory; stream "
                                    "synchronised every step; KV cache resident in HBM)",
                             "step_host_ms_per_step": host_ms}

    # ---- the fused prologue that feeds this path (NEXT-1), for context
    if rank == 0 and not args.no_prologue:
        result["prologue"] = prologue_timing(w, dev)

    # ---- several new tokens per request on the same batch and cache (NEXT-4)
    if rank == 0 and not args.no_multi_token and w.q_len == 1 and w.q_dtype == "bf16":
        result["multi_token"] = multi_token_timing(w, case, plan, C, dev)

    # ---- the layer chained with the prologue, KV gathered before Q is ready (NEXT-3)
    if rank == 0 and not args.no_chain and w.q_len == 1 and w.q_dtype == "bf16":
        result["chained_layer"] = chained_layer_timing(w, case, C, dev)

    # ---- the five scope workloads, each with its static split-KV comparison (N = 1 only)
    if rank == 0 and world == 1 and not args.no_configs:
        result["configs"] = {n: config_record(n, dev, cpu_seconds=0.0 if args.no_cpu_baseline else 2.0,
                                              single_thread=n in ("tiny", "uniform"))
                             for n in CONFIG_WORKLOADS}

    # ---- CPU oracle baseline (rank 0 only, N = 1 only)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        full_s, cores, text = oracle_sample(case, w, args.cpu_seconds)
        result["cpu_baseline"] = {"value": byt["metric"] / full_s / 1e9, "unit": UNIT, "cores": cores,
                                  "kind": "oracle", "sample": text, "ms_per_step": full_s * 1e3}

    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
