#!/usr/bin/env python3
"""Benchmark of the CSA + HCA hybrid attention step on B300.

One step = one ``hybrid_attend`` over one batch: compression of the blocks the
step's tokens close, the lightning indexer and top-k, sparse shared-KV MQA
and HCA dense MQA.  Headline workload: 64K-context decode, batch 16 (H=64,
d=512, indexer 4x64, top-k 512), caches built before the timed region.  The
same JSON line also carries, under ``workloads``, the step time, throughput
and rooflines of the 128K prefill, the ragged decode and the 1M-token decode.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own batch
(independent sequences: weak scaling, no collective on the data path); the
reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA+HCA attention tokens/s at 64K–1M ctx; % of HBM / tensor-core roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
EXTRA_WORKLOADS = ("prefill_128k", "ragged_decode", "decode_1m", "swa_prefill_32k", "inverse_rope_32k")
# sliding-window attention over the raw tokens, measured as a call of its own
# (not part of the hybrid step): one 32768-token prefill, the 128K prefill's
# heads and width, and the 4096-token window of the SWA page's example
SWA_PREFILL = {"name": "swa_prefill_32k", "length": 32768, "H": 64, "d": 512, "window": 4096, "seed": 7}
# the inverse-RoPE correction of an attention output, as a call of its own:
# the output of that 32768-token prefill, the last 64 of each head's 512 dims
ROPE_CFG = {"name": "inverse_rope_32k", "length": 32768, "H": 64, "d": 512, "d_rope": 64, "base": 10000.0,
            "seed": 8}

# DRAM traffic per call of the dominant call from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum over the call's kernels),
# keyed by (workload, call, indexer key format), with the sha256 of the sources at capture time;
# a changed source makes the figure stale and it is reported as null.
NCU_TRAFFIC = {
    # ncu capture of the decode_64k indexer call: index_chunk_scan_kernel 33,600,256 B read and
    # 0 B written + index_select_kernel 1,354,752 B read (means of two captured calls)
    ("decode_64k", "index_topk", "bf16"): {
        "bytes_per_launch": 34955008,
        "sources": {"indexer.cu": "f828009532c54521f3d1dd94c713f2f6257ef836e3719296be83a8f0835cb362",
                    "common.cuh": "b93a7dad1acde03c5b427f390c736715adf747f244ae8d972599ce95b5ac6ab8"},
    },
}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="decode_64k")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--copies", type=int, default=8, help="rotating state copies (decode)")
    ap.add_argument("--min-seconds", type=float, default=2.0, help="repeat the K-step region this long")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="measure only --workload (no 'workloads' object for the other configurations)")
    ap.add_argument("--extra", default=",".join(EXTRA_WORKLOADS),
                    help="comma-separated workloads measured after the headline one")
    ap.add_argument("--index-fp8", action="store_true",
                    help="the indexer reads FP8 E4M3 keys with per-row scales (quantised once with the caches)")
    ap.add_argument("--ctx", type=int, default=0,
                    help="every sequence this long instead of the workload's lengths (smaller cases of the same "
                         "shape, e.g. for a profiler capture); the JSON line then names the override")
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# ---------------------------------------------------------------------------
# algorithmic work (bytes and flops) of one step, per kernel
# ---------------------------------------------------------------------------
def index_key_bytes(p, fp8=False):
    """Bytes of one indexer key: dI bf16 values, or dI E4M3 codes and an fp32 scale."""
    return p["dI"] + 4 if fp8 else 2 * p["dI"]


def step_work(p, fp8=False):
    """Algorithmic bytes/flops of one hybrid step on problem p (dict from workloads)."""
    H, d, HI, dI, k, mC, mH = p["H"], p["d"], p["HI"], p["dI"], p["top_k"], p["mC"], p["mH"]
    kb = index_key_bytes(p, fp8)
    w = {"compress": 0, "index_topk": 0, "sparse_attend": 0, "dense_attend": 0}
    flops = {"index": 0, "sparse": 0, "dense": 0}
    for L, nq in zip(p["lengths"], p["n_q"]):
        lo = L - nq
        # compression: tokens of blocks closed by query positions are read once, entries written once
        n_blk_c = L // mC - lo // mC if nq else 0
        n_blk_h = L // mH - lo // mH if nq else 0
        tok = max(n_blk_c * mC, n_blk_h * mH)
        w["compress"] += 2 * d * tok + 4 * tok + 2 * d * (n_blk_c + n_blk_h)
        for t in range(lo, L):
            nC, rC = (t + 1) // mC, (t + 1) % mC
            nH, rH = (t + 1) // mH, (t + 1) % mH
            sel = min(k, nC)
            w["index_topk"] += 2 * HI * dI + nC * kb + 4 * k
            w["sparse_attend"] += 2 * ((sel + rC) * d + 2 * H * d) + 4 * k + 4 * H
            w["dense_attend"] += 2 * ((nH + rH) * d + 2 * H * d) + 4 * H
            flops["index"] += 2 * dI * nC
            flops["sparse"] += 4 * H * d * (sel + rC)
            flops["dense"] += 4 * H * d * (nH + rH)
    return w, flops


def step_work_fast(p, fp8=False):
    """Closed-form version of step_work for prefill-sized problems (same counts)."""
    if sum(p["n_q"]) <= 4096:
        return step_work(p, fp8)
    H, d, HI, dI, k, mC, mH = p["H"], p["d"], p["HI"], p["dI"], p["top_k"], p["mC"], p["mH"]
    kb = index_key_bytes(p, fp8)
    import numpy as np
    w = {"compress": 0, "index_topk": 0, "sparse_attend": 0, "dense_attend": 0}
    flops = {"index": 0, "sparse": 0, "dense": 0}
    for L, nq in zip(p["lengths"], p["n_q"]):
        lo = L - nq
        t = np.arange(lo, L, dtype=np.int64)
        nC, rC = (t + 1) // mC, (t + 1) % mC
        nH, rH = (t + 1) // mH, (t + 1) % mH
        sel = np.minimum(k, nC)
        n_blk_c, n_blk_h = L // mC - lo // mC, L // mH - lo // mH
        tok = max(n_blk_c * mC, n_blk_h * mH)
        w["compress"] += 2 * d * tok + 4 * tok + 2 * d * (n_blk_c + n_blk_h)
        w["index_topk"] += int((2 * HI * dI + nC * kb + 4 * k).sum())
        w["sparse_attend"] += int((2 * ((sel + rC) * d + 2 * H * d) + 4 * k + 4 * H).sum())
        w["dense_attend"] += int((2 * ((nH + rH) * d + 2 * H * d) + 4 * H).sum())
        flops["index"] += int((2 * dI * nC).sum())
        flops["sparse"] += int((4 * H * d * (sel + rC)).sum())
        flops["dense"] += int((4 * H * d * (nH + rH)).sum())
    return w, flops


def call_roofline(name, us, work, flops, decode, peaks, peak_src):
    """Roofline of one C-ABI call timed alone: HBM bytes for decode calls and the
    indexer, bf16 tensor flops for prefill attention.  A call timed alone is
    measured against the burst peak; the sustained peak's fraction is given
    beside it."""
    s = us * 1e-6
    if decode or name not in ("sparse_attend", "dense_attend"):
        alg = work[name]
        achieved = alg / s / 1e9
        peak = float(peaks["hbm_gbs"])
        return {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "frac_of_8TBps": achieved / 8000.0,
                "peak_source": f"hbm_gbs ({peak_src})", "alg_bytes_per_launch": alg, "avg_us": us}
    fl = flops["sparse" if name == "sparse_attend" else "dense"]
    achieved = fl / s / 1e12
    peak = float(peaks["bf16_tflops"])
    sus = float(peaks.get("bf16_tflops_sustained", peak))
    return {"bound": "tensor", "kernel": name, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "frac_of_sustained": achieved / sus, "peak_sustained": sus,
            "peak_source": f"bf16_tflops burst ({peak_src}); call timed alone",
            "alg_flops_per_launch": fl, "avg_us": us}


def step_roofline(work, flops, ms_step, peaks):
    step_bytes = sum(work.values())
    step_flops = sum(flops.values())
    s = ms_step * 1e-3
    sus = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    return {"alg_bytes": step_bytes, "alg_flops": step_flops,
            "GBps": step_bytes / s / 1e9,
            "frac_hbm_measured": step_bytes / s / 1e9 / float(peaks["hbm_gbs"]),
            "frac_hbm_8TBps": step_bytes / s / 8e12,
            "TFLOPs": step_flops / s / 1e12,
            "frac_bf16_burst": step_flops / s / 1e12 / float(peaks["bf16_tflops"]),
            "frac_bf16_sustained": step_flops / s / 1e12 / sus}


# ---------------------------------------------------------------------------
# ranks: each serves its own batch (weak scaling, no collective on the data path)
# ---------------------------------------------------------------------------
def max_over_ranks(ms, device=None):
    """The slowest rank's time (the job's time); the value itself on one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(tokens_per_rank_step, world, ms_per_step):
    """Whole-job tokens/s: every rank's tokens over the job's (max-over-ranks) step time."""
    return tokens_per_rank_step * world / (ms_per_step * 1e-3)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

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
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# oracle on the host cores
# ---------------------------------------------------------------------------
def oracle_sample(p, n_queries):
    """Inputs restricted to the first n_queries queries (a bounded sample of the workload)."""
    from compressed_sparse_attention_21_b300 import workloads as wl
    import numpy as np
    inp = wl.to_numpy(p)
    if n_queries >= int(inp["cu_q"][-1]):
        return inp, np.arange(int(inp["cu_q"][-1]))
    # keep the sequences that own the first n_queries queries
    b_last = int(np.searchsorted(inp["cu_q"], n_queries - 1, side="right") - 1)
    B = b_last + 1
    sub = dict(inp)
    for key in ("cu_kv", "cu_q", "cu_csa", "cu_hca"):
        sub[key] = inp[key][:B + 1]
    sub["kv"] = inp["kv"][:inp["cu_kv"][B]]
    sub["gate"] = inp["gate"][:inp["cu_kv"][B]]
    sub["qI"] = inp["qI"][:inp["cu_q"][B]]
    sub["q"] = inp["q"][:inp["cu_q"][B]]
    sub["kI"] = inp["kI"][:inp["cu_csa"][B]]
    return sub, np.arange(n_queries)


def oracle_queries_per_step(w, p):
    """Queries of one oracle step: every query of a decode batch, a 64-query sample of a prefill."""
    return sum(p["n_q"]) if w.decode else min(64, sum(p["n_q"]))


def time_oracle(p, target_s=10.0, max_reps=50, n_queries=None):
    import oracle
    oracle.build()
    total_q = sum(p["n_q"])
    nq = total_q if n_queries is None else min(n_queries, total_q)
    inp, eval_q = oracle_sample(p, nq)
    times = []
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        oracle.hybrid_queries(inp, eval_q=eval_q)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all >= target_s or len(times) >= max_reps:
            break
    per = statistics.mean(times)
    return {"value": nq / per, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{nq} of {total_q} queries of {p['workload']}, whole step from raw inputs "
                      f"(compression of every block the queries need, indexer, top-k, both attentions), "
                      f"{len(times)} repetitions, {sum(times):.1f} s"}


# ---------------------------------------------------------------------------
# reference arm: the oracle, timed on the host cores, on the same workload
# ---------------------------------------------------------------------------
def run_reference(args):
    from compressed_sparse_attention_21_b300 import workloads as wl
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = wl.WORKLOADS[args.workload]
    p = wl.make_problem(w, lengths=[args.ctx] * w.batch if args.ctx > 0 else None)
    nq = oracle_queries_per_step(w, p)
    inp, eval_q = oracle_sample(p, nq)
    for _ in range(max(args.warmup, 0)):
        oracle.hybrid_queries(inp, eval_q=eval_q)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.hybrid_queries(inp, eval_q=eval_q)
    dt = time.perf_counter() - t0
    value = nq * args.steps / dt
    total_q = sum(p["n_q"])
    sample = (f"every query of {w.name} per step ({nq} decode queries, whole step from raw inputs)"
              if nq == total_q else
              f"{nq} of {total_q} queries of {w.name} per step (whole step from raw inputs)")
    cfg = workload_config(w, p)
    if args.ctx > 0:
        cfg["ctx_override"] = args.ctx
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, p):
    return {"workload": w.name, "batch": w.batch, "ctx": (max(p["lengths"]) if w.lengths is None else w.lengths[0]),
            "lengths": "uniform [32768,131072], not multiples of 128" if w.lengths is None else "fixed",
            "queries_per_seq": "1 (decode)" if w.decode else "all positions (prefill)", "H": w.H, "d": w.d,
            "indexer": f"{w.HI}x{w.dI}", "top_k": w.top_k, "ratio_csa": w.mC, "ratio_hca": w.mH,
            "gate_std": w.gate_std, "seed": w.seed}


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------
def ncu_traffic(wname, dom, fp8):
    t_rec = NCU_TRAFFIC.get((wname, dom, "fp8" if fp8 else "bf16"))
    if not t_rec:
        return None
    csrc = os.path.join(ROOT, "compressed_sparse_attention_21_b300", "csrc")
    for f, sha in t_rec["sources"].items():
        path = os.path.join(csrc, f)
        if not os.path.exists(path) or hashlib.sha256(open(path, "rb").read()).hexdigest() != sha:
            return None
    return t_rec["bytes_per_launch"]


def measure(w, args, dev, peaks, peak_src, world, rank, local, headline):
    """Time one workload: the hybrid step (CUDA graph over rotating state copies),
    each C-ABI call alone, and, for the headline, e2e and the CPU baseline."""
    import torch
    import torch.distributed as dist
    from compressed_sparse_attention_21_b300 import _lib as csa
    from compressed_sparse_attention_21_b300 import workloads as wl

    p = wl.make_problem(w, lengths=[args.ctx] * w.batch if args.ctx > 0 else None)   # each rank: its own batch
    work, flops = step_work_fast(p, args.index_fp8)
    step_bytes = sum(work.values())

    cpu_base = None
    if headline and rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_base = time_oracle(p, target_s=10.0, n_queries=oracle_queries_per_step(w, p))

    layout = csa.Layout(p["lengths"], p["n_q"], w.mC, w.mH, device=dev)
    full = csa.Layout(p["lengths"], p["lengths"], w.mC, w.mH, device=dev)
    base = {k: p[k].to(dev) for k in ("kv", "gate", "qI", "kI", "q")}
    if not headline:   # host copies of the large tensors are not needed again
        del p["kv"], p["q"]
    if w.decode:
        # rotate enough copies that one rotation's bytes exceed the 126 MB L2 several times
        ncopies = max(1, args.copies if headline else min(args.copies, max(2, -(-(4 * 126 << 20) // step_bytes))))
    else:
        ncopies = 1
    copies = []
    out_bufs = []   # per copy: one device buffer holding both outputs and LSEs (one host copy per step)
    q_bytes = base["q"].numel() * 2
    for c in range(ncopies):
        t = {k: (v if c == 0 else v.clone()) for k, v in base.items() if k not in ("q", "qI")}
        # the step's inputs q and q_idx in one device buffer (one host copy per step)
        qbuf = torch.empty(q_bytes + base["qI"].numel() * 2, dtype=torch.uint8, device=dev)
        t["q"] = qbuf[:q_bytes].view(torch.bfloat16).view(base["q"].shape)
        t["qI"] = qbuf[q_bytes:].view(torch.bfloat16).view(base["qI"].shape)
        t["q"].copy_(base["q"])
        t["qI"].copy_(base["qI"])
        nq_, H_, d_ = base["q"].shape
        obuf = torch.empty(2 * q_bytes + 2 * nq_ * H_ * 4, dtype=torch.uint8, device=dev)
        outs = (obuf[:q_bytes].view(torch.bfloat16).view(nq_, H_, d_),
                obuf[q_bytes:2 * q_bytes].view(torch.bfloat16).view(nq_, H_, d_),
                obuf[2 * q_bytes:2 * q_bytes + nq_ * H_ * 4].view(torch.float32).view(nq_, H_),
                obuf[2 * q_bytes + nq_ * H_ * 4:].view(torch.float32).view(nq_, H_))
        out_bufs.append((qbuf, obuf))
        csa_cache = torch.empty((full.total_csa, w.d), dtype=torch.bfloat16, device=dev)
        hca_cache = torch.empty((full.total_hca, w.d), dtype=torch.bfloat16, device=dev)
        if w.decode:   # caches hold every entry before the step (built by a prefill-shaped call)
            csa.csa_compress(full, t["kv"], t["gate"], csa_cache)
            csa.hca_compress(full, t["kv"], t["gate"], hca_cache)
        # FP8 indexer keys live beside the caches, quantised when the entries are made
        fp8 = csa.quantize_index_keys(full, t["kI"]) if args.index_fp8 else None
        h = csa.Hybrid(layout, t["kv"], t["gate"], t["qI"], t["kI"], t["q"], w.top_k, w.scale,
                       csa_cache=csa_cache, hca_cache=hca_cache, k_idx_fp8=fp8, outputs=outs)
        h.io = out_bufs[-1]
        copies.append(h)
    del base
    torch.cuda.synchronize()

    # cache build time (prefill-shaped compression of the whole context), reported apart
    cache_build_ms = None
    if w.decode:
        h0 = copies[0]
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(3):
            csa.csa_compress(full, h0.kv, h0.gate, h0.csa_cache)
            csa.hca_compress(full, h0.kv, h0.gate, h0.hca_cache)
        ev0.record()
        for _ in range(10):
            csa.csa_compress(full, h0.kv, h0.gate, h0.csa_cache)
            csa.hca_compress(full, h0.kv, h0.gate, h0.hca_cache)
        ev1.record()
        torch.cuda.synchronize()
        cache_build_ms = ev0.elapsed_time(ev1) / 10

    # warm-up (eager; also creates the library's per-stream helper)
    for i in range(max(args.warmup, 3)):
        copies[i % ncopies]()
    torch.cuda.synchronize()

    # one CUDA graph replays one step on each copy in turn
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for h in copies:
            h()
    torch.cuda.synchronize()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()

    # K steps per timed region: the headline times exactly --steps; a prefill
    # step of the other workloads takes ~0.1 s, so it times two steps a region
    K = args.steps if (headline or w.decode) else min(args.steps, 2)

    def timed_region(K):
        """Exactly K steps (graph replays of ncopies steps plus eager remainder)."""
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        full_reps, rem = divmod(K, ncopies)
        for _ in range(full_reps):
            graph.replay()
        for i in range(rem):
            copies[i]()
        e1.record()
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), dev)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    reps = []
    min_s = args.min_seconds if headline else min(args.min_seconds, 1.0)
    t_start = time.perf_counter()
    while True:
        reps.append(timed_region(K))
        if time.perf_counter() - t_start >= min_s and len(reps) >= 3:
            break
    clocks = sampler.stop()
    ms_region = statistics.median(reps)
    ms_step = ms_region / K
    tokens_per_step = sum(p["n_q"])
    value = job_value(tokens_per_step, world, ms_step)

    # launches inside the step: an instrumented eager pass counts them per kernel
    csa.timing_reset()
    csa.timing_enable(True)
    for i in range(K):
        copies[i % ncopies]()
    torch.cuda.synchronize()
    kt = csa.timing_read()
    csa.timing_enable(False)
    csa.timing_reset()
    launches_per_step = sum(n for n, _ in kt.values()) / K

    # per-call durations: each C-ABI call of the step alone, back to back over
    # the rotating copies in one CUDA graph (no host gaps), CUDA events around
    # the replays on the capturing stream
    ws_idx, ws_sp, ws_de = {}, {}, {}
    calls = {
        "compress": lambda h: (csa.csa_compress(layout, h.kv, h.gate, h.csa_cache),
                               csa.hca_compress(layout, h.kv, h.gate, h.hca_cache)),
        "index_topk": (lambda h: csa.lightning_index_topk_fp8(layout, h.q_idx, h.k_idx_fp8[0], h.k_idx_fp8[1],
                                                              w.top_k, idx_out=h.idx, with_scores=False,
                                                              ws=ws_idx[id(h)]))
        if args.index_fp8 else
        (lambda h: csa.lightning_index_topk(layout, h.q_idx, h.k_idx, w.top_k, idx_out=h.idx,
                                            with_scores=False, ws=ws_idx[id(h)])),
        "sparse_attend": lambda h: csa.sparse_mqa_attend(layout, h.q, h.csa_cache, h.kv, h.idx, w.top_k, w.scale,
                                                         out=h.o_csa, lse=h.lse_csa, ws=ws_sp[id(h)]),
        "dense_attend": lambda h: csa.hca_dense_attend(layout, h.q, h.hca_cache, h.kv, w.scale, out=h.o_hca,
                                                       lse=h.lse_hca, ws=ws_de[id(h)]),
    }
    for h in copies:
        ws_n = (csa.index_fp8_workspace_size if args.index_fp8 else csa.index_workspace_size)(layout, w.HI, w.dI,
                                                                                               w.top_k)
        ws_idx[id(h)] = torch.zeros(max(1, ws_n), dtype=torch.uint8, device=dev)
        ws_sp[id(h)] = torch.zeros(max(1, csa.attend_workspace_size(layout, w.H, w.d, w.mC, w.top_k)),
                                   dtype=torch.uint8, device=dev)
        ws_de[id(h)] = torch.zeros(max(1, csa.attend_workspace_size(layout, w.H, w.d, w.mH, 0)), dtype=torch.uint8,
                                   device=dev)
    call_us = {}
    for name, fn in calls.items():
        for h in copies:   # warm
            fn(h)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for h in copies:
                fn(h)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps_c = 1
        while True:
            e0.record()
            for _ in range(reps_c):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            if ms >= 20.0 or reps_c >= 4096:
                break
            reps_c *= 4
        call_us[name] = ms * 1e3 / (reps_c * ncopies)
        del g
    if csa.check_device_error() != 0:
        raise RuntimeError(f"device error word set during the {w.name} measurement")

    kernels = {}
    for name, us in call_us.items():
        entry = {"avg_us": us, "kernels": sorted(k for k in kt if k.split("_")[0] in name.split("_")[0] or
                                                  (name == "index_topk" and k.startswith("index")))}
        entry["alg_bytes"] = work[name]
        entry["alg_GBps"] = work[name] / (us * 1e-6) / 1e9
        fl = {"sparse_attend": flops["sparse"], "dense_attend": flops["dense"], "index_topk": flops["index"]}.get(name)
        if fl:
            entry["alg_TFLOPs"] = fl / (us * 1e-6) / 1e12
        kernels[name] = entry
    kernels["launches_per_step"] = {k: n / K for k, (n, _) in kt.items()}

    # dominant call and its roofline: HBM-bound for decode (bytes), tensor-bound
    # for prefill attention (flops)
    dom = max(call_us, key=lambda k: call_us[k])
    roof = call_roofline(dom, call_us[dom], work, flops, w.decode, peaks, peak_src)
    roof["traffic"] = ncu_traffic(w.name, dom, args.index_fp8) if args.ctx == 0 else None
    step_roof = step_roofline(work, flops, ms_step, peaks)

    # end to end through the public API with host buffers (pinned)
    e2e = None
    if headline and not args.no_e2e:
        e2e = measure_e2e(copies, p, args, world, dev, tokens_per_step, ncopies)

    cfg = workload_config(w, p)
    if args.ctx > 0:
        cfg["ctx_override"] = args.ctx
    cfg["index_keys"] = "fp8_e4m3 + fp32 row scale" if args.index_fp8 else "bf16"
    cfg["l2"] = (f"{ncopies} rotating copies of the step state; {step_bytes / 2**20:.1f} MiB algorithmic per step, "
                 f"{ncopies * step_bytes / 2**20:.0f} MiB per rotation vs 126 MB L2") if ncopies > 1 else \
        "inputs larger than L2"
    out = {"value": value, "ms_per_step": ms_step, "steps": K, "config": cfg, "roofline": roof,
           "step_roofline": step_roof, "cpu_baseline": cpu_base, "e2e": e2e,
           "gpu_launches": int(round(launches_per_step * K)), "launches_per_step": launches_per_step,
           "kernels": kernels, "clocks": clocks, "cache_build_ms": cache_build_ms, "timed_region_reps": len(reps)}
    del copies, graph, layout, full
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def swa_flops(lengths, n_q, H, d, window):
    """Algorithmic flops of sliding-window attention: per query and head, the
    scores and the weighted sum over min(t + 1, window) keys of width d."""
    tot = 0
    for L, nq in zip(lengths, n_q):
        for t0, t1 in ((L - nq, min(L, window)), (max(L - nq, window), L)):
            if t1 <= t0:
                continue
            if t1 <= window:   # t + 1 keys for t in [t0, t1)
                tot += (t0 + 1 + t1) * (t1 - t0) // 2
            else:              # window keys each
                tot += window * (t1 - t0)
    return 4 * H * d * tot


def measure_swa(args, dev, peaks, peak_src, world, cfg=SWA_PREFILL):
    """swa_attend alone on a prefill: CUDA graph of back-to-back calls, CUDA
    events on the capturing stream, clocks sampled over the timed region."""
    import torch
    from compressed_sparse_attention_21_b300 import _lib as csa
    from compressed_sparse_attention_21_b300 import workloads as wl

    L, H, d, win = cfg["length"], cfg["H"], cfg["d"], cfg["window"]
    q = wl.randn(cfg["seed"], 4, (L, H, d), std=1.0).to(dev)
    kv = wl.randn(cfg["seed"], 0, (L, d), std=1.0).to(dev)
    layout = csa.Layout([L], [L], 4, 128, device=dev)
    scale = 1.0 / float(d) ** 0.5
    out = torch.empty_like(q)
    lse = torch.empty((L, H), dtype=torch.float32, device=dev)
    ws = torch.zeros(max(1, csa.swa_workspace_size(layout, H, d, win)), dtype=torch.uint8, device=dev)
    call = lambda: csa.swa_attend(layout, q, kv, win, scale, out=out, lse=lse, ws=ws)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(int(dev.index or 0))
    sampler.start()
    time.sleep(0.3)
    reps = []
    t_start = time.perf_counter()
    while True:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(2):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        reps.append(max_over_ranks(e0.elapsed_time(e1), dev) / 2)
        if time.perf_counter() - t_start >= min(args.min_seconds, 1.0) and len(reps) >= 3:
            break
    clocks = sampler.stop()
    if csa.check_device_error() != 0:
        raise RuntimeError("device error word set during the sliding-window measurement")
    ms = statistics.median(reps)
    fl = swa_flops([L], [L], H, d, win)
    achieved = fl / (ms * 1e-3) / 1e12
    roof = {"bound": "tensor", "kernel": "swa_attend", "achieved": achieved, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
            "peak_source": f"bf16_tflops burst ({peak_src}); call timed alone",
            "alg_flops_per_launch": fl, "avg_us": ms * 1e3, "traffic": None}
    conf = {"workload": cfg["name"], "batch": 1, "ctx": L, "lengths": "fixed", "queries_per_seq": "all positions",
            "H": H, "d": d, "window": win, "seed": cfg["seed"], "l2": "inputs larger than L2"}
    del q, kv, out, lse, ws, g
    torch.cuda.empty_cache()
    return {"value": job_value(L, world, ms), "ms_per_step": ms, "steps": 2 * len(reps), "roofline": roof,
            "clocks": clocks, "unit": "tokens/s", "config": conf, "calls_us": {"swa_attend": ms * 1e3}}


def rope_bytes(total_q, H, d_rope):
    """Algorithmic bytes of the in-place inverse-RoPE correction: each query's
    rope slice of every head read and written once (bf16)."""
    return 2 * total_q * H * d_rope * 2


def measure_rope(args, dev, peaks, peak_src, world, cfg=ROPE_CFG):
    """csa_inverse_rope alone on a prefill-sized output: CUDA graph of
    back-to-back calls over rotating copies of the output (their slices exceed
    L2), CUDA events on the capturing stream."""
    import torch
    from compressed_sparse_attention_21_b300 import _lib as csa
    from compressed_sparse_attention_21_b300 import workloads as wl

    L, H, d, dr = cfg["length"], cfg["H"], cfg["d"], cfg["d_rope"]
    x = wl.randn(cfg["seed"], 0, (L, H, d), std=1.0).to(dev)
    outs = [x] + [x.clone() for _ in range(2)]   # 3 x 268 MB of rope slices per rotation
    layout = csa.Layout([L], [L], 4, 128, device=dev)
    call = lambda o: csa.inverse_rope(layout, o, dr, cfg["base"])
    for _ in range(max(args.warmup, 3)):
        for o in outs:
            call(o)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for o in outs:
            call(o)
    g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(int(dev.index or 0))
    sampler.start()
    time.sleep(0.3)
    reps = []
    t_start = time.perf_counter()
    while True:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(10):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        reps.append(max_over_ranks(e0.elapsed_time(e1), dev) / (10 * len(outs)))
        if time.perf_counter() - t_start >= min(args.min_seconds, 1.0) and len(reps) >= 3:
            break
    clocks = sampler.stop()
    if csa.check_device_error() != 0:
        raise RuntimeError("device error word set during the inverse-RoPE measurement")
    ms = statistics.median(reps)
    nb = rope_bytes(L, H, dr)
    achieved = nb / (ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "kernel": "inverse_rope", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "peak_source": f"hbm_gbs ({peak_src})", "alg_bytes_per_launch": nb,
            "avg_us": ms * 1e3, "traffic": None}
    conf = {"workload": cfg["name"], "batch": 1, "ctx": L, "queries_per_seq": "all positions", "H": H, "d": d,
            "d_rope": dr, "base": cfg["base"], "seed": cfg["seed"],
            "l2": f"{len(outs)} rotating outputs, {len(outs) * nb / 2 / 2**20:.0f} MiB of rope slices vs 126 MB L2"}
    n_outs = len(outs)
    del x, outs, g
    torch.cuda.empty_cache()
    return {"value": job_value(L, world, ms), "ms_per_step": ms, "steps": 10 * n_outs * len(reps),
            "roofline": roof, "clocks": clocks, "unit": "tokens/s", "config": conf,
            "calls_us": {"inverse_rope": ms * 1e3}}


def measure_e2e(copies, p, args, world, dev, tokens_per_step, ncopies):
    """The same metric through the C ABI with host buffers: every step copies its
    queries in from pinned host memory and both outputs and LSEs out.

    Pipelined: a copy-in stream, the compute stream and a copy-out stream, one
    state copy per step in flight, so one step's copies overlap the
    neighbouring steps' compute; the whole rotation of steps is captured once in
    a CUDA graph and replayed, as a serving loop runs it.  The serial form (copy
    in, step, copy out, one after the other on one stream) is given beside it."""
    import torch
    # host side: the step's inputs (q, q_idx) packed as the device buffer holds them, and one output area per copy
    h0 = copies[0]
    in_host = h0.io[0].cpu().pin_memory()
    outs = [torch.empty(c.io[1].shape, dtype=torch.uint8).pin_memory() for c in copies]
    bi = in_host.numel()
    bo = outs[0].numel()

    def copy_out(hh, o):
        o.copy_(hh.io[1], non_blocking=True)

    def serial_step(i):
        hh = copies[i % ncopies]
        hh.io[0].copy_(in_host, non_blocking=True)
        hh()
        copy_out(hh, outs[i % ncopies])

    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def pipelined_rotation():
        """Every copy once: copy-in on s_in, the step on the current stream, copy-out on s_out."""
        cur = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(cur)
        s_in.wait_event(start)
        s_out.wait_event(start)
        ev_out = []
        for i, hh in enumerate(copies):
            ev_in, ev_done, ev_o = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(s_in):
                hh.io[0].copy_(in_host, non_blocking=True)
                ev_in.record(s_in)
            cur.wait_event(ev_in)
            hh()
            ev_done.record(cur)
            s_out.wait_event(ev_done)
            with torch.cuda.stream(s_out):
                copy_out(hh, outs[i])
                ev_o.record(s_out)
            ev_out.append(ev_o)
        for ev in ev_out:
            cur.wait_event(ev)

    def timed(run):
        import torch.distributed as dist
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), dev)

    # serial, captured: copy in, step, copy out on one stream
    for i in range(3):
        serial_step(i)
    g_ser = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_ser):
        for i in range(ncopies):
            serial_step(i)
    g_ser.replay()
    torch.cuda.synchronize()
    reps = max(1, args.steps // ncopies)
    ms_ser = timed(lambda: [g_ser.replay() for _ in range(reps)]) / (reps * ncopies)

    # pipelined, captured
    pipelined_rotation()
    torch.cuda.synchronize()
    g_pipe = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_pipe):
        pipelined_rotation()
    g_pipe.replay()
    torch.cuda.synchronize()
    ms_pipe = timed(lambda: [g_pipe.replay() for _ in range(reps)]) / (reps * ncopies)
    return {"value": job_value(tokens_per_step, world, ms_pipe), "unit": "tokens/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": ms_pipe,
            "steps": reps * ncopies,
            "path": "per step: pinned host q/q_idx copied in (one copy), hybrid_attend through the C ABI, both "
                    "outputs and LSEs copied out to pinned host memory (one copy); copy-in, compute and copy-out on "
                    "three streams with "
                    f"one of {ncopies} state copies per step, so copies overlap the neighbouring steps; the "
                    "rotation captured once in a CUDA graph and replayed",
            "serial": {"value": job_value(tokens_per_step, world, ms_ser), "ms_per_step": ms_ser,
                       "path": "copy in, step, copy out one after the other on one stream (CUDA graph)"}}


def main(argv=None):
    args = parse(argv)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist
    from compressed_sparse_attention_21_b300 import _lib as csa
    from compressed_sparse_attention_21_b300 import build as csa_build
    from compressed_sparse_attention_21_b300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        csa_build.build()
    if world > 1:
        dist.barrier()
    csa.load()
    peaks, peak_src = load_peaks()

    w = wl.WORKLOADS[args.workload]
    head = measure(w, args, dev, peaks, peak_src, world, rank, local, headline=True)

    extra = {}
    if not args.no_extra and args.ctx == 0:
        for name in [x for x in args.extra.split(",") if x and x != w.name]:
            if name == SWA_PREFILL["name"]:
                extra[name] = measure_swa(args, dev, peaks, peak_src, world)
                continue
            if name == ROPE_CFG["name"]:
                extra[name] = measure_rope(args, dev, peaks, peak_src, world)
                continue
            r = measure(wl.WORKLOADS[name], args, dev, peaks, peak_src, world, rank, local, headline=False)
            extra[name] = {k: r[k] for k in ("value", "ms_per_step", "steps", "roofline", "step_roofline", "clocks",
                                             "launches_per_step", "cache_build_ms")}
            extra[name]["unit"] = "tokens/s"
            extra[name]["config"] = r["config"]
            extra[name]["calls_us"] = {k: v["avg_us"] for k, v in r["kernels"].items() if isinstance(v, dict)
                                       and "avg_us" in v}

    cfg = head["config"]
    cfg["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
    line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 (indexer keys fp8 e4m3)" if args.index_fp8 else "bf16",
            "data": "synthetic", "config": cfg, "roofline": head["roofline"],
            "step_roofline": head["step_roofline"], "cpu_baseline": head["cpu_baseline"], "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"], "launches_per_step": head["launches_per_step"],
            "kernels": head["kernels"], "clocks": head["clocks"], "cache_build_ms": head["cache_build_ms"],
            "timed_region_reps": head["timed_region_reps"],
            "peaks": {"source": peak_src, "hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"],
                      "bf16_tflops_sustained": peaks.get("bf16_tflops_sustained")}}
    if extra:
        line["workloads"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
