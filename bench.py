#!/usr/bin/env python
"""Benchmark of batched paged-KV decode attention on GB300.

One step = the whole decode hot path over one batch: the host plan (split-KV
schedule) followed by run (the schedule upload and the TMA-pipelined decode
kernel, which also merges its split rows, replayed from one CUDA graph per
step) on inputs resident in HBM.  The end-to-end figure runs the same step eagerly
through the public API with host buffers.  The default workload
is the batch-64 GQA decode batch (64 requests, 32 qo / 8 kv heads, head_dim
128, bf16, lengths uniform in [512, 4096], page size 16, pages drawn from a
20000-page pool).  Its K/V bytes (0.58 GB) exceed the 129 MB L2, so no flush
is needed between steps.

Prints ONE JSON line.  ``--impl reference`` times the fp64 CPU oracle on the
host cores instead (the reference arm).  The path runs on one GPU: launched
with WORLD_SIZE > 1 (torchrun), the GPU arm refuses with an error, and the
reference arm runs on rank 0 only (the other ranks exit without work).
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
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak) and µs/call per batch"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")
KERNEL_SOURCES = ["paged_kv_decode_28_gb300/csrc/pkd_decode.cu", "paged_kv_decode_28_gb300/csrc/pkd_ptx.cuh",
                  "paged_kv_decode_28_gb300/csrc/pkd_internal.h"]
APPEND_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "append_traffic.json")
APPEND_SOURCES = ["paged_kv_decode_28_gb300/csrc/pkd_append.cu", "paged_kv_decode_28_gb300/csrc/pkd_internal.h"]
PREFILL_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "prefill_traffic.json")
PREFILL_SOURCES = ["paged_kv_decode_28_gb300/csrc/pkd_tile2.cu", "paged_kv_decode_28_gb300/csrc/pkd_ptx.cuh",
                   "paged_kv_decode_28_gb300/csrc/pkd_internal.h"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5,
                    help="standard workload index (1..5); 5, the long-context fp8 batch, is the largest")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--all-configs", action="store_true", help="also print one line per standard workload")
    ap.add_argument("--batch", type=int, default=None,
                    help="shrink the workload to its first N requests (small cases for profiling)")
    ap.add_argument("--op", choices=["decode", "append", "tree", "prefill", "mla", "merge", "single"], default="decode",
                    help="append: pkd_append_kv (new tokens written into the workload's pool); tree: "
                    "prefix-tree decode on the 3-level tree workload; prefill: append-prefill attention; mla: MLA "
                    "decode; merge: the standalone pkd_merge_state / pkd_merge_states on cascade-shaped states")
    ap.add_argument("--kv-layout", choices=["NHD", "HND"], default="NHD",
                    help="page layout of the K/V pools: NHD [P, Hk, D] pages or HND [Hk, P, D] pages")
    ap.add_argument("--append-tokens", type=int, default=0,
                    help="--op append: new tokens per request in the bulk case (0: enough that the "
                    "bytes moved exceed twice the 129 MB L2)")
    return ap.parse_args()


def kernel_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(b) -> int:
    """K/V bytes of the valid keys of every (request, kv head) row, plus q, out,
    lse and the fp8 scales.  Split-KV partials and the schedule are excluded."""
    e_kv = b.k_cache.element_size()
    e_q = b.q.element_size()
    kv = int(np.asarray(b.kv_lens, dtype=np.int64).sum()) * b.num_kv_heads * b.head_dim * 2 * e_kv
    if b.prefix_page_indices is not None:
        kv += b.prefix_len * b.num_kv_heads * b.head_dim * 2 * e_kv  # shared prefix counted once
    qo = b.batch * b.num_qo_heads * b.head_dim * 2 * e_q
    lse = 4 * b.batch * b.num_qo_heads
    scales = 8 * b.num_kv_heads if b.k_scale is not None else 0
    return kv + qo + lse + scales


def decode_kernel_bytes(b) -> int:
    """Algorithmic bytes of the kernels between the library's timing events:
    the decode kernel (all of algorithmic_bytes) or, for the cascade, the
    prefix kernel and the suffix decode that overlaps it (every K/V byte, q and
    the scales; the merge after them writes out and lse)."""
    n = algorithmic_bytes(b)
    if b.prefix_page_indices is not None:
        n -= b.batch * b.num_qo_heads * (b.head_dim * b.q.element_size() + 4)
    return n


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def launch_world() -> tuple:
    """(world_size, rank) from the torchrun environment ((1, 0) when absent)."""
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))


def cpu_sample_batch(b, n_req: int):
    """The first n_req requests of a batch, with their pages gathered into a
    compact host pool (input preparation for the CPU oracle)."""
    import torch

    pages, indptr, last = [], [0], []
    for r in range(n_req):
        own = b.kv_page_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]]
        pages.append(own)
        indptr.append(indptr[-1] + len(own))
        last.append(int(b.kv_last_page_len[r]))
    allp = np.concatenate(pages).astype(np.int64)
    sel = torch.as_tensor(allp, device=b.k_cache.device)
    k = b.k_cache[sel].cpu().contiguous()
    v = b.v_cache[sel].cpu().contiguous()
    q = b.q[:n_req].cpu().contiguous()
    idx = np.arange(len(allp), dtype=np.int32)
    lens = b.kv_lens[:n_req]
    return q, k, v, np.asarray(indptr, np.int32), idx, np.asarray(last, np.int32), lens


_ALL_THREADS = []  # the oracle's thread count before any run narrowed it


def time_cpu_oracle(b, target_s: float, max_req=None, threads=None):
    """Run the C fp64 oracle on a bounded sample of requests (all qo heads),
    on all host cores or on `threads` of them.
    Returns (GB/s of algorithmic bytes, seconds, requests, threads)."""
    from oracle import c_oracle

    if not _ALL_THREADS:  # OpenMP keeps a thread count set by a run for the next ones
        _ALL_THREADS.append(c_oracle.max_threads())
    threads = _ALL_THREADS[0] if threads is None else int(threads)
    e_kv = b.k_cache.element_size()
    ks = None if b.k_scale is None else b.k_scale.cpu()
    vs = None if b.v_scale is None else b.v_scale.cpu()

    def run(n):
        q, k, v, indptr, idx, last, lens = cpu_sample_batch(b, n)
        t0 = time.perf_counter()
        c_oracle.paged_decode(q, k, v, indptr, idx, last, sm_scale=b.sm_scale, k_scale=ks, v_scale=vs,
                              num_threads=threads)
        dt = time.perf_counter() - t0
        nbytes = (int(np.asarray(lens, np.int64).sum()) * b.num_kv_heads * b.head_dim * 2 * e_kv
                  + n * b.num_qo_heads * b.head_dim * 2 * b.q.element_size() + 4 * n * b.num_qo_heads)
        return nbytes, dt

    nb1, dt1 = run(1)
    n = int(max(1, min(max_req or b.batch, math.floor(target_s / max(dt1, 1e-6)))))
    nbytes, dt = run(n)
    reps = 1
    if target_s > 0 and dt < 0.5 * target_s:  # whole batch is quick: repeat it to time a few seconds
        reps = int(min(100, math.ceil(0.5 * target_s / max(dt, 1e-6))))
        tot = 0.0
        for _ in range(reps):
            tot += run(n)[1]
        dt = tot / reps
    return nbytes / dt / 1e9, dt * reps, n, threads


def l2_bytes(dev) -> int:
    """The device's L2 size in bytes (129 MB on GB300 when the query is missing)."""
    import torch

    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2**20)


def l2_note(nbytes: int, l2: int) -> str:
    if nbytes > l2:
        return f"inputs {nbytes / 1e9:.2f} GB > {l2 / 1e6:.0f} MB L2; no flush between steps"
    return f"inputs {nbytes / 1e9:.3f} GB < {l2 / 1e6:.0f} MB L2: L2-resident between steps (no flush)"


def run_ours(args):
    import torch

    import paged_kv_decode_28_gb300 as pkd
    from paged_kv_decode_28_gb300 import _build
    from paged_kv_decode_28_gb300 import workloads as wl

    _build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    b = wl.make_config(args.config, device=dev, batch=args.batch)
    if args.kv_layout == "HND":  # the same pages re-laid as [Hk, P, D] blocks
        for name in ("k_cache", "v_cache"):
            c = getattr(b, name)
            setattr(b, name, c.view(torch.uint8).permute(0, 2, 1, 3).contiguous().view(c.dtype))
            del c
    cascade = b.prefix_page_indices is not None
    idx = torch.from_numpy(b.kv_page_indices).to(dev)
    pre = torch.from_numpy(b.prefix_page_indices).to(dev) if cascade else None
    plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=16 if cascade else 0, device=dev,
                    kv_layout=args.kv_layout)
    stream = torch.cuda.current_stream(dev)
    out = torch.empty_like(b.q)
    lse = torch.empty(b.batch, b.num_qo_heads, dtype=torch.float32, device=dev)
    kw = dict(sm_scale=b.sm_scale, k_scale=b.k_scale, v_scale=b.v_scale, out=out, lse=lse)
    # a workload smaller than L2 would be read from L2 in every step after the
    # first: R independent copies of q, K and V (R * bytes >= 4 x L2) are used
    # in turn, so each step reads its inputs from HBM
    l2 = l2_bytes(dev)
    ws_bytes = algorithmic_bytes(b)
    R = 1 if ws_bytes > l2 else int(math.ceil(4 * l2 / ws_bytes))
    copies = [(b.q, b.k_cache, b.v_cache)] + [(b.q.clone(), b.k_cache.clone(), b.v_cache.clone())
                                              for _ in range(R - 1)]
    cur = [0]  # the copy the next run uses

    def do_plan():
        plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size, q_dtype=b.q.dtype, kv_dtype=b.k_cache.dtype)

    def do_run():
        q_r, k_r, v_r = copies[cur[0] % R]
        if cascade:
            plan.cascade_decode(pre, b.prefix_last_page_len, q_r, k_r, v_r, **kw)
        else:
            plan.run(q_r, k_r, v_r, **kw)

    for _ in range(max(args.warmup, 3)):
        do_plan()
        do_run()
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0

    # ---- run is captured in CUDA graphs (plan stays on the host before every
    # replay, as in serving); one graph per timed step so that each step's
    # decode launch is bracketed by its own events from the library's hook
    K = args.steps
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, z in kev:  # torch creates the CUDA event at its first record; the library re-records it
        a.record(stream)
        z.record(stream)
    torch.cuda.synchronize()
    graphs = []
    for i in range(K):
        plan.set_timing_events(*kev[i])
        cur[0] = i  # step i reads copy i % R
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            do_run()
        graphs.append(g)
    plan.set_timing_events(None, None)
    for i in range(max(args.warmup, 3, K)):  # every graph is uploaded before the timed steps
        do_plan()
        graphs[i % K].replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(K):
            do_plan()
            graphs[i].replay()
        e1.record(stream)
        torch.cuda.synchronize()
    clk = clocks.summary()
    ms_total = e0.elapsed_time(e1)
    ms_total_max = ms_total
    ms_step = ms_total_max / K
    kern_ms = [a.elapsed_time(z) for a, z in kev]
    kern_avg_ms = sum(kern_ms) / K
    # the same replays with a read of a 2 x L2 buffer between steps (outside the
    # decode kernel's events), so that none of a step's input can still be in
    # L2; a read leaves clean lines behind, where a write would leave dirty ones
    # whose write-back would then fall inside the timed kernel
    flush = torch.ones(l2, dtype=torch.float16, device=dev)
    for i in range(K):
        do_plan()
        flush.sum()
        graphs[i].replay()
    torch.cuda.synchronize()
    kern_ms_flushed = [a.elapsed_time(z) for a, z in kev]
    del flush
    nbytes = algorithmic_bytes(b)
    value = nbytes / (ms_step * 1e-3) / 1e9
    assert plan.check_device_errors() == 0
    # host time of one plan (the schedule for this batch into pinned memory),
    # timed on its own after the timed steps
    plan_s = []
    for _ in range(min(K, 50)):
        t0 = time.perf_counter()
        do_plan()
        plan_s.append(time.perf_counter() - t0)
    torch.cuda.synchronize()

    # ---- end to end through the C ABI with host buffers: q and the page table in, out and lse back
    q_h = b.q.cpu().pin_memory()
    idx_h = torch.from_numpy(b.kv_page_indices.copy()).pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    q_d = torch.empty_like(b.q)
    idx_d = torch.empty_like(idx)
    e2e_i = [0]

    def e2e_step():  # eager, through the public API
        _, k_r, v_r = copies[e2e_i[0] % R]
        e2e_i[0] += 1
        q_d.copy_(q_h, non_blocking=True)
        idx_d.copy_(idx_h, non_blocking=True)
        plan.plan(b.kv_indptr, idx_d, b.kv_last_page_len, b.page_size, q_dtype=b.q.dtype, kv_dtype=b.k_cache.dtype)
        if cascade:
            plan.cascade_decode(pre, b.prefix_last_page_len, q_d, k_r, v_r, **kw)
        else:
            plan.run(q_d, k_r, v_r, **kw)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(K):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_value = nbytes / (e2e_s / K) / 1e9
    h2d = q_h.numel() * q_h.element_size() + idx_h.numel() * 4 + (b.batch + 1) * 4 + b.batch * 4
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * 4

    peak, peak_kind = measured_hbm_peak()
    achieved = decode_kernel_bytes(b) / (kern_avg_ms * 1e-3) / 1e9
    traffic = None
    try:
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
        ent = tr.get("configs", {}).get(str(args.config))
        # the record holds only for the kernel sources it was captured on, the full batch and NHD pages
        if ent and tr.get("kernel_hash") == kernel_hash() and args.batch is None and args.kv_layout == "NHD":
            traffic = ent.get("dram_bytes_per_launch")
    except Exception:
        pass

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": 1,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "us_per_call": round(ms_step * 1e3, 2),
        "tokens_per_s": round(b.batch / (ms_step * 1e-3), 1),
        "host_plan_us": round(statistics.median(plan_s) * 1e6, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {torch.bfloat16: "bf16", torch.float16: "f16"}[b.q.dtype] + (
            "+e4m3kv" if b.k_cache.dtype == torch.float8_e4m3fn else ""),
        "data": "synthetic (seeded N(0,1) values, seeded lengths and page placement)",
        "config": {
            "workload": b.name,
            "batch": b.batch,
            "num_qo_heads": b.num_qo_heads,
            "num_kv_heads": b.num_kv_heads,
            "head_dim": b.head_dim,
            "page_size": b.page_size,
            "kv_layout": args.kv_layout,
            "kv_tokens": int(np.asarray(b.kv_lens, np.int64).sum()),
            "algorithmic_bytes_per_step": nbytes,
            "l2": (l2_note(nbytes, l2) if R == 1 else
                   (f"inputs {nbytes / 1e9:.3f} GB < {l2 / 1e6:.0f} MB L2: {R} copies of q, K and V used in "
                    f"turn ({R * nbytes / 1e9:.2f} GB), so every step reads from HBM"))
                  + "; a second pass reads 2 x L2 bytes before every step (roofline.kernel_us_l2_flushed)",
            "parallelism": "one GPU",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": ("pkd prefix_pair_kernel + decode_kernel (the suffix decode starts on the SMs the prefix "
                       "kernel leaves free; events from before the prefix kernel to the end of the decode grid)"
                       if cascade else "pkd decode_kernel"),
            "bytes_per_launch": decode_kernel_bytes(b),
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "kernel_us": round(kern_avg_ms * 1e3, 2),
            # spread of the per-step decode launch (events around each launch)
            "kernel_us_p10_p50_p90": [round(float(x) * 1e3, 2) for x in np.percentile(kern_ms, [10, 50, 90])],
            # the decode kernel when a read of 2 x L2 bytes precedes every step (same graphs)
            "kernel_us_l2_flushed": round(sum(kern_ms_flushed) / K * 1e3, 2),
            "frac_l2_flushed": round(decode_kernel_bytes(b) / (sum(kern_ms_flushed) / K * 1e-3) / 1e9 / peak, 4),
            # every kernel of the step (host plan included) against the same peak
            "whole_step": {"achieved": round(value, 1), "frac": round(value / peak, 4)},
        },
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "us_per_step": round(e2e_s / K * 1e6, 2)},
        # upload copy + decode (+ prefix kernel + merge for the cascade)
        "gpu_launches": K * (4 if cascade else 2),
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        gbs, secs, n_req, threads = time_cpu_oracle(b, target_s=10.0)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": f"{n_req} of {b.batch} requests, all {b.num_qo_heads} qo heads "
                                          f"(C fp64 oracle, {secs:.1f} s)"}
        # the same oracle on one core, over a shorter sample
        gbs1, secs1, n1, _ = time_cpu_oracle(b, target_s=3.0, threads=1)
        line["cpu_baseline"]["single_thread"] = {"value": round(gbs1, 4), "unit": UNIT, "cores": 1,
                                                 "sample": f"{n1} of {b.batch} requests ({secs1:.1f} s)"}
    return line


def run_reference(args):
    """The reference arm: the fp64 CPU oracle on the host cores, on a bounded
    sample of the same workload each step."""
    import torch

    from paged_kv_decode_28_gb300 import workloads as wl
    from oracle import c_oracle

    c_oracle.build()
    # the same seeded inputs as the GPU arm (generated by the device RNG when a GPU is present)
    b = wl.make_config(args.config, device="cuda" if torch.cuda.is_available() else "cpu")
    threads = c_oracle.max_threads()
    K, W = args.steps, max(args.warmup, 0)
    budget = 150.0  # seconds for the whole run
    _, dt1, _, _ = time_cpu_oracle(b, target_s=0.0, max_req=1)
    per_step = budget / max(K + W, 1)
    n_req = int(max(1, min(b.batch, math.floor(per_step / max(dt1, 1e-6)))))
    q, k, v, indptr, idx, last, lens = cpu_sample_batch(b, n_req)
    ks = None if b.k_scale is None else b.k_scale.cpu()
    vs = None if b.v_scale is None else b.v_scale.cpu()

    def step():
        c_oracle.paged_decode(q, k, v, indptr, idx, last, sm_scale=b.sm_scale, k_scale=ks, v_scale=vs,
                              num_threads=threads)

    for _ in range(W):
        step()
    t0 = time.perf_counter()
    for _ in range(K):
        step()
    secs = (time.perf_counter() - t0) / K
    e_kv = b.k_cache.element_size()
    nbytes = (int(np.asarray(lens, np.int64).sum()) * b.num_kv_heads * b.head_dim * 2 * e_kv
              + n_req * b.num_qo_heads * b.head_dim * 2 * b.q.element_size() + 4 * n_req * b.num_qo_heads)
    value = nbytes / secs / 1e9
    sample = f"{n_req} of {b.batch} requests per step, all {b.num_qo_heads} qo heads (C fp64 oracle)"
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": UNIT,
        "n_gpus": 1,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(secs * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) values, seeded lengths and page placement)",
        "config": {"workload": b.name, "batch": b.batch, "num_qo_heads": b.num_qo_heads,
                   "num_kv_heads": b.num_kv_heads, "head_dim": b.head_dim, "page_size": b.page_size,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_append(args):
    """pkd_append_kv on a workload's pool geometry: a bulk append
    (args.append_tokens new tokens per request; bandwidth-bound, reported
    against the HBM peak) and the one-token-per-request append of a decode step
    (latency)."""
    import torch

    import paged_kv_decode_28_gb300 as pkd
    from paged_kv_decode_28_gb300 import _build
    from paged_kv_decode_28_gb300 import workloads as wl

    _build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    lens = np.asarray(wl.config_lengths(args.config, args.batch), dtype=np.int64)
    P, _, Hk, _, kvd = wl.config_geometry(args.config)
    row_bytes = Hk * 128 * 2 * (2 + (1 if kvd == "e4m3" else 2))  # K and V of one token, read + written
    A = args.append_tokens or -(-int(2 * 129e6) // (len(lens) * row_bytes))
    new_dtype = torch.float16 if kvd == "f16" else torch.bfloat16
    # page table sized for A more tokens per request (the pages the new tokens
    # land in), pages in a seeded random order; pool values are never read
    rng = np.random.default_rng(900 + args.config)
    need = int(((lens + A + P - 1) // P).sum())
    indptr_h, idx_h, _ = wl.lengths_to_page_table(lens + A, P, rng.permutation(need))
    pool_dtype = {"bf16": torch.bfloat16, "f16": torch.float16, "e4m3": torch.float8_e4m3fn}[kvd]
    shape = (need, Hk, P, 128) if args.kv_layout == "HND" else (need, P, Hk, 128)
    k_cache = torch.empty(shape, dtype=pool_dtype, device=dev)
    v_cache = torch.empty_like(k_cache)
    k_scale = v_scale = None
    if kvd == "e4m3":
        k_scale = torch.full((Hk,), 0.02, device=dev)
        v_scale = torch.full((Hk,), 0.02, device=dev)
    B = len(lens)
    gen = torch.Generator(device=dev).manual_seed(1)
    k_new = torch.randn(B * A, Hk, 128, device=dev, generator=gen).to(new_dtype)
    v_new = torch.randn(B * A, Hk, 128, device=dev, generator=gen).to(new_dtype)
    bi = torch.arange(B, device=dev, dtype=torch.int32).repeat_interleave(A)
    pos = (torch.as_tensor(lens.astype(np.int32), device=dev).repeat_interleave(A) +
           torch.arange(A, device=dev, dtype=torch.int32).repeat(B))
    indptr = torch.as_tensor(np.asarray(indptr_h, dtype=np.int32), device=dev)
    idx = torch.as_tensor(np.asarray(idx_h, dtype=np.int32), device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(n_tok, steps):
        for _ in range(max(args.warmup, 3)):
            pkd.append_kv(k_new[:n_tok], v_new[:n_tok], bi[:n_tok], pos[:n_tok], indptr, idx, k_cache, v_cache,
                          k_scale=k_scale, v_scale=v_scale, err=err, kv_layout=args.kv_layout)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            pkd.append_kv(k_new[:n_tok], v_new[:n_tok], bi[:n_tok], pos[:n_tok], indptr, idx, k_cache, v_cache,
                          k_scale=k_scale, v_scale=v_scale, err=err, kv_layout=args.kv_layout)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    K = args.steps
    with ClockSampler(0) as clocks:
        ms_bulk = timed(B * A, K)
    clk = clocks.summary()
    # one token per request (the first new token of every request), as in a
    # decode step: device time per append from a captured graph of 16 appends
    # replayed K times, and the time per append issued one call at a time
    # from Python (host marshalling included)
    sel = torch.arange(B, device=dev) * A
    k1, v1, b1, p1 = k_new[sel].contiguous(), v_new[sel].contiguous(), bi[sel].contiguous(), pos[sel].contiguous()

    def one():
        pkd.append_kv(k1, v1, b1, p1, indptr, idx, k_cache, v_cache, k_scale=k_scale, v_scale=v_scale, err=err,
                      kv_layout=args.kv_layout)

    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            one()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(16):
            one()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    us_step = e0.elapsed_time(e1) / (16 * K) * 1e3
    e0.record(stream)
    for _ in range(K):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    us_call = e0.elapsed_time(e1) / K * 1e3
    assert int(err.item()) == 0
    e_new, e_kv = 2, k_cache.element_size()
    nbytes = B * A * Hk * 128 * 2 * (e_new + e_kv) + B * A * 8  # rows read + written, plus indices
    achieved = nbytes / (ms_bulk * 1e-3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    # DRAM bytes of one launch from an ncu capture of the same kernel source on
    # this workload's geometry, scaled by the tokens appended (traffic grows in
    # proportion to the tokens)
    traffic = None
    try:
        with open(APPEND_TRAFFIC_FILE) as f:
            tr = json.load(f)
        ent = tr.get("configs", {}).get(str(args.config))
        if tr.get("kernel_hash") == kernel_hash(APPEND_SOURCES) and ent and args.kv_layout == "NHD":
            traffic = int(ent["dram_bytes"] * (B * A) / ent["tokens"])
    except Exception:
        pass
    # the oracle on a bounded sample: 256 of the new tokens into a 512-page pool of the same geometry
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import kv_append as ka

        n_s = min(256, B * A)
        pool = torch.zeros(512, P, Hk, 128, dtype=pool_dtype)
        ip = torch.tensor([0, 512], dtype=torch.int32)
        pi = torch.arange(512, dtype=torch.int32)
        ps = torch.arange(n_s, dtype=torch.int32) % (512 * P)
        ks = k_scale.cpu() if k_scale is not None else None
        t0 = time.perf_counter()
        ka.append_kv(pool, pool, k_new[:n_s].cpu(), v_new[:n_s].cpu(), torch.zeros(n_s, dtype=torch.int32), ps, ip,
                     pi, P, ks, ks)
        dt = time.perf_counter() - t0
        cpu = {"value": round(n_s * Hk * 128 * 2 * (e_new + e_kv) / dt / 1e9, 5), "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": f"{n_s} new tokens into a 512-page pool of the same geometry "
               f"(python oracle, {dt:.2f} s)"}
    return {
        "metric": "kv append (pkd_append_kv): achieved HBM GB/s",
        "value": round(achieved, 1), "unit": "GB/s", "n_gpus": 1, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_bulk, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": kvd, "data": "synthetic (seeded N(0,1) rows)",
        "config": {"workload": f"append {A} tokens to each request of {wl.CONFIG_NAMES[args.config]}",
                   "batch": B, "num_kv_heads": Hk, "head_dim": 128, "page_size": P, "kv_layout": args.kv_layout,
                   "new_dtype": str(new_dtype),
                   "bytes_per_step": int(nbytes), "parallelism": "one GPU",
                   "l2": f"{nbytes / 1e9:.2f} GB moved per step "
                   f"{'>' if nbytes > 129e6 else '<'} 129 MB L2; no flush between steps"},
        "roofline": {"bound": "hbm", "kernel": "pkd append_kv_kernel", "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback", "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic},
        "decode_step_append_us": {"graph_replay": round(us_step, 2), "python_call": round(us_call, 2),
                                  "bytes": int(B * row_bytes)},
        "cpu_baseline": cpu, "gpu_launches": K, "clocks": clk,
    }


def tree_bytes(b) -> int:
    """K/V bytes of every shared node (once) and of every request's own keys,
    plus q, out and lse."""
    e = b.k_cache.element_size()
    row = b.num_kv_heads * b.head_dim * 2 * e  # K and V of one key, all kv heads
    kv = int(np.asarray(b.kv_lens, dtype=np.int64).sum()) * row
    for _, ip, _, last in b.levels:
        for n in range(len(ip) - 1):
            pages = int(ip[n + 1] - ip[n])
            kv += ((pages - 1) * b.page_size + int(last[n])) * row if pages else 0
    return kv + b.batch * b.num_qo_heads * (b.head_dim * 2 * b.q.element_size() + 4)


def prefill_flops(b) -> int:
    """Multiply-adds of S = q K^T and O = P V, two flops each, over the keys
    each query token sees (causal: up to its own position)."""
    n = 0
    for r in range(len(b.qo_indptr) - 1):
        q_len = int(b.qo_indptr[r + 1] - b.qo_indptr[r])
        kv = int(b.kv_lens[r])
        # token i sees kv - q_len + i + 1 keys
        n += q_len * (kv - q_len) + q_len * (q_len + 1) // 2
    return 4 * n * b.num_qo_heads * b.head_dim


def measured_tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def run_tree(args):
    """Prefix-tree decode (pkd_plan_tree / pkd_tree_decode) on the 3-level
    tree workload: run captured in CUDA graphs, both plans on the host before
    every replay."""
    import torch

    import paged_kv_decode_28_gb300 as pkd
    from paged_kv_decode_28_gb300 import _build
    from paged_kv_decode_28_gb300 import workloads as wl

    _build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    b = wl.make_config_tree(device=dev, batch=args.batch)
    idx = torch.from_numpy(b.kv_page_indices).to(dev)
    lv = [(ri, ki, torch.from_numpy(np.asarray(ix)).to(dev), last) for ri, ki, ix, last in b.levels]
    plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=16, device=dev)
    out = torch.empty_like(b.q)
    lse = torch.empty(b.batch, b.num_qo_heads, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def do_plan():
        plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size)
        plan.plan_tree(lv)

    def do_run():
        plan.tree_decode(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale, out=out, lse=lse)

    for _ in range(max(args.warmup, 3)):
        do_plan()
        do_run()
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    K = args.steps
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        do_run()
    for _ in range(3):
        do_plan()
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        e0.record(stream)
        for _ in range(K):
            do_plan()
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    clk = clocks.summary()
    ms_step = e0.elapsed_time(e1) / K
    assert plan.check_device_errors() == 0
    nbytes = tree_bytes(b)
    achieved = nbytes / (ms_step * 1e-3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import attention as orc

        rows = [(r, h) for r in range(0, b.batch, max(1, b.batch // 8)) for h in (0, b.num_qo_heads - 1)]
        bc = b.to("cpu")
        t0 = time.perf_counter()
        orc.multilevel_cascade_decode(bc.q, bc.k_cache, bc.v_cache, bc.levels, bc.kv_indptr, bc.kv_page_indices,
                                      bc.kv_last_page_len, sm_scale=b.sm_scale, rows=rows)
        dt = time.perf_counter() - t0
        frac = len(rows) / (b.batch * b.num_qo_heads)
        cpu = {"value": round(nbytes * frac / dt / 1e9, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{len(rows)} of {b.batch * b.num_qo_heads} (request, qo head) rows, bytes scaled by "
               f"that fraction (python fp64 oracle, {dt:.2f} s)"}
    return {
        "metric": "prefix-tree decode (pkd_tree_decode): achieved HBM GB/s per step", "value": round(achieved, 1),
        "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 5),
        "us_per_call": round(ms_step * 1e3, 2), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) values, seeded lengths and page placement)",
        "config": {"workload": b.name, "batch": b.batch, "num_qo_heads": b.num_qo_heads,
                   "num_kv_heads": b.num_kv_heads, "page_size": b.page_size, "bytes_per_step": nbytes,
                   "l2": l2_note(nbytes, l2_bytes(dev)),
                   "parallelism": "one GPU"},
        "roofline": {"bound": "hbm", "kernel": "whole step (schedule upload, own-page decode, tree kernel, merge)",
                     "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback", "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None},
        "cpu_baseline": cpu, "gpu_launches": 4 * K, "clocks": clk,
    }


def run_prefill(args):
    """Paged append-prefill (pkd_plan_prefill / pkd_prefill_run) on the
    prefill workload: K back-to-back launches timed with CUDA events."""
    import torch

    import paged_kv_decode_28_gb300 as pkd
    from paged_kv_decode_28_gb300 import _build
    from paged_kv_decode_28_gb300 import workloads as wl

    _build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    b = wl.make_config_prefill(device=dev, batch=args.batch)
    idx = torch.from_numpy(b.kv_page_indices).to(dev)
    plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, device=dev)
    plan.plan_prefill(b.qo_indptr, b.kv_indptr, idx, b.kv_last_page_len, b.page_size, causal=True)
    out = torch.empty_like(b.q)
    lse = torch.empty(b.q.shape[0], b.num_qo_heads, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        plan.prefill(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        e0.record(stream)
        for _ in range(K):
            plan.prefill(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale, out=out, lse=lse)
        e1.record(stream)
        torch.cuda.synchronize()
    clk = clocks.summary()
    ms_step = e0.elapsed_time(e1) / K
    assert plan.check_device_errors() == 0
    flops = prefill_flops(b)
    achieved = flops / (ms_step * 1e-3) / 1e12
    # DRAM bytes of one launch from an ncu capture of the same kernel source on
    # the same workload (null for another source or another batch)
    traffic = None
    try:
        with open(PREFILL_TRAFFIC_FILE) as f:
            tr = json.load(f)
        if tr.get("kernel_hash") == kernel_hash(PREFILL_SOURCES) and tr.get("workload") == b.name and \
                int(tr.get("query_tokens", -1)) == int(b.q.shape[0]):
            traffic = int(tr["dram_bytes_per_launch"])
    except Exception:
        pass
    peak, peak_kind = measured_tensor_peak()
    e = b.k_cache.element_size()
    nbytes = (int(np.asarray(b.kv_lens, np.int64).sum()) * b.num_kv_heads * b.head_dim * 2 * e
              + 2 * b.q.numel() * b.q.element_size() + lse.numel() * 4)
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import attention as orc

        T = b.q.shape[0]
        rows = [(t, h) for t in range(0, T, max(1, T // 16)) for h in (0, b.num_qo_heads - 1)]
        bc = b.to("cpu")
        t0 = time.perf_counter()
        orc.paged_prefill(bc.q, bc.qo_indptr, bc.k_cache, bc.v_cache, bc.kv_indptr, bc.kv_page_indices,
                          bc.kv_last_page_len, causal=True, sm_scale=b.sm_scale, rows=rows)
        dt = time.perf_counter() - t0
        frac = len(rows) / (T * b.num_qo_heads)
        cpu = {"value": round(flops * frac / dt / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"{len(rows)} of {T * b.num_qo_heads} (token, qo head) rows, flops scaled by that "
               f"fraction (python fp64 oracle, {dt:.2f} s)"}
    return {
        "metric": "paged append-prefill attention (pkd_prefill_run): achieved TFLOP/s",
        "value": round(achieved, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) values, seeded lengths and page placement)",
        "config": {"workload": b.name, "batch": b.batch, "query_tokens": int(b.q.shape[0]),
                   "num_qo_heads": b.num_qo_heads, "num_kv_heads": b.num_kv_heads, "page_size": b.page_size,
                   "causal": True, "flops_per_step": flops, "bytes_per_step": nbytes,
                   "l2": l2_note(nbytes, l2_bytes(dev)),
                   "parallelism": "one GPU"},
        "roofline": {"bound": "tensor", "kernel": "pkd tile2_kernel (paired query tiles)", "achieved": round(achieved, 2),
                     "peak": peak, "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops, burst)"
                     if peak_kind == "measured" else "fallback", "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "hbm_gbs": round(nbytes / (ms_step * 1e-3) / 1e9, 1)},
        "cpu_baseline": cpu, "gpu_launches": K, "clocks": clk,
    }


def mla_bytes(b) -> int:
    """Each request's latent and rotary rows once (1152 bytes per key), plus q,
    out and lse."""
    kv = int(np.asarray(b.kv_lens, np.int64).sum()) * (512 + 64) * 2
    B, H = b.batch, b.num_heads
    return kv + B * H * (576 * 2 + 512 * 2 + 4)


def run_mla(args):
    """MLA decode (pkd_mla_decode) on the 64-request DeepSeek-V3 workload: K
    back-to-back calls (host planning and the unit upload included) timed with
    CUDA events."""
    import torch

    import paged_kv_decode_28_gb300 as pkd
    from paged_kv_decode_28_gb300 import _build
    from paged_kv_decode_28_gb300 import workloads as wl

    _build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    b = wl.make_config_mla(device=dev, batch=args.batch)
    idx = torch.from_numpy(np.asarray(b.kv_page_indices, np.int32)).to(dev)
    out = torch.empty((b.batch, b.num_heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((b.batch, b.num_heads), dtype=torch.float32, device=dev)
    ws = None
    stream = torch.cuda.current_stream(dev)

    def step():
        nonlocal ws
        _, _, ws = pkd.mla_decode(b.q_nope, b.q_pe, b.ckv_cache, b.kpe_cache, b.kv_indptr, idx, b.kv_last_page_len,
                                  sm_scale=b.sm_scale, out=out, lse=lse, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        e0.record(stream)
        for _ in range(K):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    clk = clocks.summary()
    ms_step = e0.elapsed_time(e1) / K
    nbytes = mla_bytes(b)
    achieved = nbytes / (ms_step * 1e-3) / 1e9
    flops = int(np.asarray(b.kv_lens, np.int64).sum()) * b.num_heads * (576 + 512) * 2
    peak, peak_kind = measured_hbm_peak()
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import mla as orc

        rows = [(r, h) for r in range(0, b.batch, max(1, b.batch // 8)) for h in (0, b.num_heads - 1)]
        t0 = time.perf_counter()
        orc.mla_decode(b.q_nope.cpu(), b.q_pe.cpu(), b.ckv_cache.cpu(), b.kpe_cache.cpu(), b.kv_indptr,
                       b.kv_page_indices, b.kv_last_page_len, sm_scale=b.sm_scale, rows=rows)
        dt = time.perf_counter() - t0
        frac = len(rows) / (b.batch * b.num_heads)
        cpu = {"value": round(nbytes * frac / dt / 1e9, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{len(rows)} of {b.batch * b.num_heads} (request, head) rows, bytes scaled by that "
               f"fraction (python fp64 oracle, {dt:.2f} s, pool copied to the host first)"}
    return {
        "metric": "MLA decode (pkd_mla_decode): achieved HBM GB/s per call", "value": round(achieved, 1),
        "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 5),
        "us_per_call": round(ms_step * 1e3, 2), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) values, seeded lengths and page placement)",
        "config": {"workload": b.name, "batch": b.batch, "num_heads": b.num_heads, "page_size": b.page_size,
                   "kv_tokens": int(np.asarray(b.kv_lens, np.int64).sum()), "bytes_per_step": nbytes,
                   "flops_per_step": flops, "tflops": round(flops / (ms_step * 1e-3) / 1e12, 1),
                   "l2": l2_note(nbytes, l2_bytes(dev)),
                   "parallelism": "one GPU"},
        "roofline": {"bound": "hbm", "kernel": "pkd mla_kernel + mla_merge_kernel (whole call)",
                     "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback", "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None},
        "cpu_baseline": cpu, "gpu_launches": 2 * K, "clocks": clk,
    }


def run_merge(args):
    """The standalone merge_state (two states) and merge_states (k = 4 states)
    calls: n = 16384 rows x 32 qo heads x 128 dims of bf16 values with fp32
    log-sum-exps (each input well above L2), K back-to-back calls each, timed
    with CUDA events.  Bytes: every input and output once."""
    import torch

    import paged_kv_decode_28_gb300 as pkd
    from paged_kv_decode_28_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    n, H, D, k = (args.batch or 16384), 32, 128, 4
    va = torch.randn((n, H, D), generator=gen, device=dev).to(torch.bfloat16)
    vb = torch.randn((n, H, D), generator=gen, device=dev).to(torch.bfloat16)
    sa = torch.randn((n, H), generator=gen, device=dev) * 4
    sb = torch.randn((n, H), generator=gen, device=dev) * 4
    vk = torch.randn((n, k, H, D), generator=gen, device=dev).to(torch.bfloat16)
    sk = torch.randn((n, k, H), generator=gen, device=dev) * 4
    out = torch.empty_like(va)
    s_out = torch.empty_like(sa)
    K = args.steps
    peak, peak_kind = measured_hbm_peak()
    res = {}
    for name, fn, nbytes in (
            ("merge_state", lambda: pkd.merge_state(va, sa, vb, sb, out=out, s_out=s_out),
             3 * va.numel() * 2 + 3 * sa.numel() * 4),
            ("merge_states", lambda: pkd.merge_states(vk, sk),
             vk.numel() * 2 + sk.numel() * 4 + va.numel() * 2 + sa.numel() * 4)):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(0) as clocks:
            e0.record()
            for _ in range(K):
                fn()
            e1.record()
            torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / K * 1e3
        gbs = nbytes / (us * 1e-6) / 1e9
        res[name] = {"us_per_call": round(us, 2), "bytes_per_call": int(nbytes), "achieved": round(gbs, 1),
                     "frac": round(gbs / peak, 4), "clocks": clocks.summary()}
    return {"metric": "standalone merge_state / merge_states: achieved HBM GB/s per call",
            "value": res["merge_state"]["achieved"], "unit": "GB/s", "n_gpus": 1, "steps": K,
            "warmup": max(args.warmup, 3), "higher_is_better": True, "dtype": "bf16 values, f32 lse",
            "data": "synthetic (seeded N(0,1) values)",
            "config": {"workload": f"n={n} x {H} heads x {D} dims; merge_states over k={k} states",
                       "l2": l2_note(3 * va.numel() * 2, l2_bytes(dev)), "parallelism": "one GPU"},
            "roofline": {"bound": "hbm", "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", **res}}


def run_single(args):
    """One request through pkd_single_decode (q [32, 128], contiguous f16 K/V
    [2048, 32, 128]: the single-request workload's shape): host plan, the
    schedule in the upload kernel's parameters and the decode, K back-to-back
    calls timed with CUDA events.  The calls rotate over enough input copies
    (4 x L2 in all) that every call reads its K/V from HBM."""
    import torch

    import paged_kv_decode_28_gb300 as pkd
    from paged_kv_decode_28_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(21)
    L, Hq, Hk, D = 2048, 32, 32, 128
    nbytes = 2 * L * Hk * D * 2 + 2 * Hq * D * 2 + Hq * 4
    R = max(1, int(math.ceil(4 * l2_bytes(dev) / nbytes)))
    inputs = [(torch.randn((Hq, D), generator=gen, device=dev).half(),
               torch.randn((L, Hk, D), generator=gen, device=dev).half(),
               torch.randn((L, Hk, D), generator=gen, device=dev).half()) for _ in range(R)]
    ws = torch.empty(pkd.workspace_bytes(1, Hq, Hk, D, pkd.num_ctas(0), 0), dtype=torch.uint8, device=dev)
    out = torch.empty((Hq, D), dtype=torch.float16, device=dev)
    lse = torch.empty(Hq, dtype=torch.float32, device=dev)
    for i in range(max(args.warmup, 3)):
        pkd.single_decode(*inputs[i % R], workspace=ws, out=out, lse=lse)
    torch.cuda.synchronize()
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        e0.record()
        for i in range(K):
            pkd.single_decode(*inputs[i % R], workspace=ws, out=out, lse=lse)
        e1.record()
        torch.cuda.synchronize()
    clk = clocks.summary()
    ms = e0.elapsed_time(e1) / K
    achieved = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    return {"metric": "single-request decode (pkd_single_decode): achieved HBM GB/s per call",
            "value": round(achieved, 1), "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": max(args.warmup, 3),
            "ms_per_step": round(ms, 5), "us_per_call": round(ms * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic (seeded N(0,1) values)",
            "config": {"workload": f"one request, {L} keys, {Hq}/{Hk} heads, f16, contiguous K/V",
                       "bytes_per_call": nbytes, "input_copies": R,
                       "l2": f"{R} input copies ({R * nbytes / 1e6:.0f} MB) used in turn", "parallelism": "one GPU"},
            "roofline": {"bound": "hbm", "kernel": "whole call (host plan, schedule upload kernel, decode)",
                         "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": None},
            "cpu_baseline": None, "gpu_launches": 2 * K, "clocks": clk}


def main():
    args = parse_args()
    world, rank = launch_world()
    if world > 1 or args.gpus != 1:
        if args.impl == "reference" and args.op == "decode":
            # the reference arm is the CPU oracle: rank 0 runs it, the others have no work
            if rank == 0:
                print(json.dumps(run_reference(args)), flush=True)
            return
        print(f"bench.py: this path runs on one GPU only (got --gpus {args.gpus}, WORLD_SIZE {world}); "
              "its cascade and MLA kernels use cluster-multicast loads that stay within one GPU's memory",
              file=sys.stderr, flush=True)
        sys.exit(2)
    if args.op in ("append", "tree", "prefill", "mla", "merge", "single"):
        line = {"append": run_append, "tree": run_tree, "prefill": run_prefill, "mla": run_mla,
                "merge": run_merge, "single": run_single}[args.op](args)
        print(json.dumps(line), flush=True)
        return
    if args.impl == "reference":
        line = run_reference(args)
    else:
        line = run_ours(args)
        if args.all_configs:
            for c in (1, 2, 3, 4, 5):
                if c == args.config:
                    continue
                a2 = argparse.Namespace(**{**vars(args), "config": c, "no_cpu_baseline": True})
                try:
                    print(json.dumps(run_ours(a2)), flush=True)
                except Exception as exc:  # keep the headline line even if one extra workload fails
                    print(json.dumps({"config": c, "error": str(exc)}), file=sys.stderr, flush=True)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
