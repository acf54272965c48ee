#!/usr/bin/env python3
"""Benchmark of the grouped-query attention forward on B300.

One step = one pass of the whole hot path over one batch of synthetic input:
a prefill call (gqa_fwd) on the BERT-base-shaped encoder workload (B=32,
Hq=12, Hkv=3, S=1024, D=64, key lengths U[512,1024]) followed by a decode
call (gqa_decode, split-KV + combine) on the Llama-style decode workload
(B=64, Hq=64, Hkv=8, D=128, cache lengths U[1024,8192]).  The headline
``value`` is prefill TFLOP/s (algorithmic flops / prefill kernel time); the
``decode`` object carries KV-cache GB/s.  Inputs are resident in HBM; between
timed steps a 256 MB buffer is written to flush L2, and the decode step
streams 1.2 GB of cache anyway.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--prefill WORKLOAD] [--no-cpu-baseline]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(no collective on the data path; weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from grouped_query_attention_08_b300 import inputs, roofline  # noqa: E402

METRIC = "GQA prefill TFLOP/s & decode KV-cache GB/s on 1 B300, % of roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

# DRAM traffic per launch from one ncu capture, valid only while the kernel
# source is unchanged (sha256 of the file below); None = not captured for the
# current source.
NCU_TRAFFIC = {
    # one launch on bert_base
    "prefill": {"source": "grouped_query_attention_08_b300/csrc/prefill_sm103.cuh",
                "sha256": "66cde4ea4676e13ce3cc2f3449d42839bb4c0aee1f7be5fe558b7cf635d72e8c",
                "workload": "bert_base", "bytes": 88589824},
    # a B=16 capture scaled to B=64 by valid KV bytes
    "decode": {"source": "grouped_query_attention_08_b300/csrc/decode_sm103.cuh",
               "sha256": "3da23f2311d8b3f1dad3c2a6686fd96218f2aa4cc6d53874bd51a4448f128b40",
               "workload": "llama_decode", "bytes": 1271529128},
}


def _sha(path):
    with open(os.path.join(ROOT, path), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def _traffic(kind):
    t = NCU_TRAFFIC[kind]
    if t["bytes"] is None or t["sha256"] is None:
        return None
    return t["bytes"] if _sha(t["source"]) == t["sha256"] else None


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        # raw samples (the JSON line carries their summary)
        self.path = os.path.join(tempfile.gettempdir(), "gqa_bench_clocks_%d.csv" % os.getpid())

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _whole_job_rate(work_per_step, steps, ws, seconds):
    """Work all ranks did per second: every rank (replica) does `work_per_step`
    per step, and `seconds` is the slowest rank's time for `steps` steps."""
    return work_per_step * steps * ws / seconds


def _max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class OracleSampler:
    """Times the fp64 oracle (as it stands) on row samples of a prefill workload."""

    def __init__(self, workload):
        import numpy as np
        import oracle
        self.oracle = oracle
        self.w = w = inputs.WORKLOADS[workload]
        inp = inputs.make_workload(w)
        self.q = inp["q"].float().numpy()
        self.k = inp["k"].float().numpy()
        self.v = inp["v"].float().numpy()
        self.lens = None if inp["seqlens_k"] is None else inp["seqlens_k"].numpy()
        self.total = w.B * w.Hq * w.Sq
        oracle.build()
        # admissible keys of every (b, h, i) row, for the flop count of a sample
        i = np.arange(w.Sq)
        Lb = np.full(w.B, w.Sk) if self.lens is None else self.lens.astype(np.int64)
        lim = Lb[:, None] + 0 * i[None, :]
        if w.causal:
            lim = np.minimum(lim, i[None, :] + w.Sk - w.Sq + 1)
        lim = np.maximum(lim, 0)                                    # [B, Sq]
        self.row_keys = np.broadcast_to(lim[:, None, :], (w.B, w.Hq, w.Sq)).reshape(-1)

    def rows(self, n, seed=12345):
        return inputs.sample_rows(self.total, n, seed).numpy()

    def run(self, rows):
        """Returns (seconds, algorithmic flops) of one oracle call on these rows."""
        w = self.w
        t0 = time.perf_counter()
        self.oracle.attention(self.q, self.k, self.v, scale=w.scale, causal=w.causal, seqlens_k=self.lens,
                              rows=rows)
        dt = time.perf_counter() - t0
        return dt, 4 * w.D * int(self.row_keys[rows].sum())

    def calibrate(self, seconds):
        """Row count whose oracle call takes about `seconds` (capped at the whole workload)."""
        n = 256
        while True:
            dt, _ = self.run(self.rows(n))
            if dt >= 0.5 * seconds or n >= self.total:
                return n, dt
            n = int(min(self.total, max(2 * n, n * 0.8 * seconds / max(dt, 1e-4))))


def cpu_baseline(workload, seconds=10.0):
    """The oracle timed on the host cores on a bounded sample (about `seconds` of work)."""
    o = OracleSampler(workload)
    n, dt = o.calibrate(seconds)
    rows = o.rows(n)
    reps = 1 if dt >= 0.5 * seconds else int(max(1, round(seconds / max(dt, 1e-4))))
    tot_t, tot_f = 0.0, 0
    for _ in range(reps):
        t, f = o.run(rows)
        tot_t += t
        tot_f += f
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": tot_f / tot_t / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": "%d of %d query rows of %s x %d repeat(s) (fp64 oracle, OpenMP), %.1f s" % (
                n, o.total, workload, reps, tot_t)}


def run_reference(args):
    """The oracle as the reference arm: every step is one oracle call on a row
    sample sized so that the whole warm-up + timed run takes about two minutes."""
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    w = inputs.WORKLOADS[args.prefill]
    o = OracleSampler(args.prefill)
    per_step = max(0.02, 120.0 / (args.steps + args.warmup))
    n, _ = o.calibrate(per_step)
    rows = o.rows(n)
    for _ in range(args.warmup):
        o.run(rows)
    tot_t, tot_f = 0.0, 0
    for _ in range(args.steps):
        t, f = o.run(rows)
        tot_t += t
        tot_f += f
    val = tot_f / tot_t / 1e12
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    cb = {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
          "sample": "%d of %d query rows of %s per step (fp64 oracle, OpenMP)" % (n, o.total, args.prefill)}
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t * 1e3 / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": _workload_name(w), "sampled_rows_per_step": n},
            "cpu_baseline": cb,
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def time_prefill_workload(gqa, name, device, flush, reps=10, warmup=3):
    """Per-call time of gqa_fwd on a named prefill workload (CUDA events, L2
    flushed before every call); returns TFLOP/s of algorithmic work."""
    w = inputs.WORKLOADS[name]
    inp = inputs.make_workload(w)
    d = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.empty_like(d["q"])
    if isinstance(w, inputs.SparseWorkload):
        base = inputs.WORKLOADS[w.base]
        lens = None if inp["seqlens_k"] is None else inp["seqlens_k"].tolist()
        flops = 4 * base.D * roofline.blockmask_pairs(base.B, base.Hq, base.Sq, base.Sk, base.causal,
                                                      inp["block_mask"], w.block_size, lens)
        lse = torch.empty((base.B, base.Hq, base.Sq), dtype=torch.float32, device=device)

        def call():
            gqa.gqa_fwd_sparse(d["q"], d["k"], d["v"], d["block_mask"], w.block_size, causal=base.causal,
                               seqlens_k=d["seqlens_k"], scale=base.scale, out=out, lse=lse)
    elif isinstance(w, inputs.VarlenWorkload):
        # packed sequences: only real (query, key) pairs are work
        lq = (inp["cu_seqlens_q"][1:] - inp["cu_seqlens_q"][:-1]).tolist()
        lk = (inp["cu_seqlens_k"][1:] - inp["cu_seqlens_k"][:-1]).tolist()
        flops = roofline.varlen_flops(w.Hq, w.D, lq, lk, w.causal)
        lse = torch.empty((w.Hq, d["q"].shape[0]), dtype=torch.float32, device=device)

        def call():
            gqa.gqa_fwd_varlen(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"],
                               max_seqlen_q=d["max_seqlen_q"], max_seqlen_k=d["max_seqlen_k"], causal=w.causal,
                               scale=w.scale, out=out, lse=lse)
    else:
        lens = None if inp["seqlens_k"] is None else inp["seqlens_k"].tolist()
        flops = roofline.prefill_flops(w.B, w.Hq, w.Sq, w.Sk, w.D, w.causal, lens)
        lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=device)

        def call():
            gqa.gqa_fwd(d["q"], d["k"], d["v"], causal=w.causal, seqlens_k=d["seqlens_k"], scale=w.scale,
                        out=out, lse=lse)

    for _ in range(warmup):
        flush.fill_(1)
        call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for i in range(reps):
        flush.fill_(i & 0xFF)
        evs[i][0].record()
        call()
        evs[i][1].record()
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / reps
    return {"tflops": flops / (ms * 1e-3) / 1e12, "ms": ms, "workload": _workload_name(w),
            "algorithmic_flops_per_launch": flops}


def time_decode_fp8(gqa, name, device, flush, reps=20, warmup=3):
    """Per-call time of gqa_decode_fp8 (split + combine) on a named FP8-cache
    decode workload, L2 flushed before every call; returns GB/s of e4m3 KV bytes."""
    w = inputs.WORKLOADS[name]
    inp = inputs.make_workload(w)
    d = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lens = inp["cache_seqlens"].tolist()
    kv_bytes = roofline.decode_kv_bytes(w.Hkv, w.D, lens, elem_bytes=1)
    out = torch.empty_like(d["q"])
    wsb = gqa.gqa_decode_fp8_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, 0, w.Smax)
    work = torch.empty((max(wsb, 16),), dtype=torch.uint8, device=device)

    def call():
        gqa.gqa_decode_fp8(d["q"], d["kcache"], d["vcache"], d["cache_seqlens"], d["k_scale"], d["v_scale"],
                           scale=w.scale, out=out, workspace=work)

    for _ in range(warmup):
        flush.fill_(1)
        call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for i in range(reps):
        flush.fill_(i & 0xFF)
        evs[i][0].record()
        call()
        evs[i][1].record()
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / reps
    return {"value": kv_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s (e4m3 KV-cache bytes read / decode time)",
            "ms": ms, "kv_bytes_per_step": kv_bytes,
            "tokens_per_s": sum(lens) / (ms * 1e-3),
            "workload": "%s decode B%d Hq%d Hkv%d D%d Smax%d cache lengths U[%d,%d], FP8 e4m3 cache" % (
                w.name, w.B, w.Hq, w.Hkv, w.D, w.Smax, w.lens[0], w.lens[1])}


def time_backward(gqa, name, device, flush, reps=10, warmup=3):
    """Per-call time of gqa_bwd (Dsum, dQ, dK/dV kernels) on a named dense
    prefill workload, with the forward's out and lse as inputs and a seeded
    N(0,1) upstream gradient; L2 flushed before every call.  Returns TFLOP/s
    of algorithmic work (10 * D flops per admissible pair)."""
    w = inputs.WORKLOADS[name]
    inp = inputs.make_workload(w)
    d = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    g = torch.Generator("cpu").manual_seed(w.seed + 101)
    dout = torch.randn(tuple(d["q"].shape), generator=g, dtype=torch.float32).to(torch.bfloat16).to(device)
    out, lse = gqa.gqa_fwd(d["q"], d["k"], d["v"], causal=w.causal, seqlens_k=d["seqlens_k"], scale=w.scale)
    lens = None if inp["seqlens_k"] is None else inp["seqlens_k"].tolist()
    flops = roofline.backward_flops(w.B, w.Hq, w.Sq, w.Sk, w.D, w.causal, lens)
    dq, dk, dv = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
    dsum = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=device)

    def call():
        gqa.gqa_bwd(d["q"], d["k"], d["v"], out, dout, lse, causal=w.causal, seqlens_k=d["seqlens_k"],
                    scale=w.scale, dq=dq, dk=dk, dv=dv, dsum=dsum)

    for _ in range(warmup):
        flush.fill_(1)
        call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for i in range(reps):
        flush.fill_(i & 0xFF)
        evs[i][0].record()
        call()
        evs[i][1].record()
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / reps
    tf = flops / (ms * 1e-3) / 1e12
    peaks, psrc = _peaks()
    peak = peaks["bf16_tflops"]
    return {"tflops": tf, "ms": ms, "frac": tf / peak, "peak_tflops": peak, "peak_source": psrc + " bf16 burst",
            "workload": "backward of " + _workload_name(w), "algorithmic_flops_per_launch": flops,
            "launches_per_call": 3}


def _workload_name(w):
    if isinstance(w, inputs.SparseWorkload):
        return "%s: %s under a block mask, %d-token blocks, band of +-%d blocks plus key block 0" % (
            w.name, _workload_name(inputs.WORKLOADS[w.base]), w.block_size, w.window)
    if isinstance(w, inputs.VarlenWorkload):
        return "%s packed prefill B%d Hq%d Hkv%d D%d %s lengths U[%d,%d] (queries = keys), no padding" % (
            w.name, w.B, w.Hq, w.Hkv, w.D, "causal" if w.causal else "non-causal", w.lens[0], w.lens[1])
    lens = "full" if w.lens is None else "U[%d,%d]" % w.lens
    return "%s prefill B%d Hq%d Hkv%d Sq%d Sk%d D%d %s keys %s" % (
        w.name, w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, "causal" if w.causal else "non-causal", lens)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--warmup-seconds", type=float, default=1.5,
                    help="minimum wall time of back-to-back warm-up steps right before the timed steps")
    ap.add_argument("--min-timed-ms", type=float, default=250.0,
                    help="each timed step repeats the pass (flush, prefill, decode) R times, R chosen from "
                         "the warm-up so that the K steps take at least this long")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--prefill", default="bert_base",
                    choices=["bert_base", "bert_large_long", "causal_long"])
    ap.add_argument("--decode", default="llama_decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip timing the other prefill workloads after the main run")
    ap.add_argument("--other-reps", type=int, default=10)
    ap.add_argument("--backward-workloads", default="bert_base,causal_long",
                    help="comma-separated dense prefill workloads whose backward (gqa_bwd) is timed after "
                         "the main run; empty for none")
    ap.add_argument("--other-workloads",
                    default="bert_base,bert_large_long,causal_long,bert_base_varlen,bert_large_long_sparse,"
                            "llama_decode_fp8",
                    help="comma-separated workloads timed after the main run (FP8-cache decode workloads "
                         "report under decode_fp8)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import grouped_query_attention_08_b300 as gqa
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    gqa.load_library()

    wp = inputs.WORKLOADS[args.prefill]
    wd = inputs.WORKLOADS[args.decode]
    pin = inputs.make_workload(wp)
    din = inputs.make_workload(wd)
    P = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in pin.items()}
    Dd = {k: v.to(device) for k, v in din.items()}
    lens_p = None if pin["seqlens_k"] is None else pin["seqlens_k"].tolist()
    flops_p = roofline.prefill_flops(wp.B, wp.Hq, wp.Sq, wp.Sk, wp.D, wp.causal, lens_p)
    bytes_p = roofline.prefill_bytes(wp.B, wp.Hq, wp.Hkv, wp.Sq, wp.Sk, wp.D, lens_p)
    lens_d = din["cache_seqlens"].tolist()
    kv_bytes_d = roofline.decode_kv_bytes(wd.Hkv, wd.D, lens_d)
    bytes_d = roofline.decode_bytes(wd.B, wd.Hq, wd.Hkv, wd.D, lens_d)

    out_p = torch.empty_like(P["q"])
    lse_p = torch.empty((wp.B, wp.Hq, wp.Sq), dtype=torch.float32, device=device)
    out_d = torch.empty_like(Dd["q"])
    nsplit = gqa.gqa_decode_num_splits(wd.B, wd.Hkv, wd.Smax, 0)
    wsb = gqa.gqa_decode_workspace_bytes(wd.B, wd.Hq, wd.Hkv, wd.D, 0, wd.Smax)
    work = torch.empty((max(wsb, 16),), dtype=torch.uint8, device=device)
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=device)

    def prefill():
        gqa.gqa_fwd(P["q"], P["k"], P["v"], causal=wp.causal, seqlens_k=P["seqlens_k"], scale=wp.scale,
                    out=out_p, lse=lse_p)

    def decode():
        gqa.gqa_decode(Dd["q"], Dd["kcache"], Dd["vcache"], Dd["cache_seqlens"], scale=wd.scale,
                       num_splits=0, out=out_d, workspace=work)

    def step(i):
        flush.fill_(i & 0xFF)
        prefill()
        decode()

    # one untimed step checks that the path runs cleanly before anything else
    step(1)
    torch.cuda.synchronize()
    if gqa.gqa_device_status() != 0:
        raise RuntimeError("device error in the first step")

    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        # Warm-up inside the clock sampler and right before the timed steps:
        # at least W steps and at least --warmup-seconds of back-to-back work,
        # so that a short timed region starts on a GPU already in its
        # steady state (no idle gap, clocks up, caches and TLBs warm).
        t0 = time.perf_counter()
        n_warm = 0
        while n_warm < args.warmup or time.perf_counter() - t0 < args.warmup_seconds:
            for _ in range(8):
                step(n_warm)
                n_warm += 1
            torch.cuda.synchronize()
        if gqa.gqa_device_status() != 0:
            raise RuntimeError("device error during warm-up")
        # Inner repetitions: every timed step runs the pass R times, so that
        # the K steps (exactly K, as asked) take at least --min-timed-ms even
        # when K is small; R comes from the warm-up's wall time per pass and is
        # the same on every rank (the largest).
        pass_ms = (time.perf_counter() - t0) * 1e3 / max(1, n_warm)
        R = max(1, math.ceil(args.min_timed_ms / (K * pass_ms))) if args.min_timed_ms > 0 else 1
        R = int(_max_over_ranks(float(R), ws, device))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K * R)]
        _barrier(ws)
        torch.cuda.synchronize()
        t_start.record()
        for i in range(K):
            for rr in range(R):
                j = i * R + rr
                flush.fill_(j & 0xFF)
                ev[j][0].record()
                prefill()
                ev[j][1].record()
                decode()
                ev[j][2].record()
        t_end.record()
        torch.cuda.synchronize()
        _barrier(ws)
    clk = clocks.summary()
    if gqa.gqa_device_status() != 0:
        raise RuntimeError("device error in the timed region")
    t_pre = [e[0].elapsed_time(e[1]) for e in ev]     # every pass (K * R)
    t_dec = [e[1].elapsed_time(e[2]) for e in ev]
    total_ms = t_start.elapsed_time(t_end)
    pre_s = _max_over_ranks(sum(t_pre) / 1e3, ws, device)
    dec_s = _max_over_ranks(sum(t_dec) / 1e3, ws, device)
    total_s = _max_over_ranks(total_ms / 1e3, ws, device)

    # per-pass distribution (this rank): median and min beside the mean
    per_step = {"inner_reps": R, "passes": K * R, "prefill_ms": {"mean": statistics.fmean(t_pre), "median": statistics.median(t_pre),
                               "min": min(t_pre), "max": max(t_pre)},
                "decode_ms": {"mean": statistics.fmean(t_dec), "median": statistics.median(t_dec),
                              "min": min(t_dec), "max": max(t_dec)},
                "warmup_steps_run": n_warm, "timed_region_ms": total_ms}

    value = _whole_job_rate(flops_p, K * R, ws, pre_s) / 1e12
    dec_gbs = _whole_job_rate(kv_bytes_d, K * R, ws, dec_s) / 1e9
    peaks, psrc = _peaks()
    pre_avg = pre_s / (K * R)
    dec_avg = dec_s / (K * R)
    pre_ach = flops_p / pre_avg / 1e12
    dec_ach = bytes_d / dec_avg / 1e9
    tr_p, tr_d = _traffic("prefill"), _traffic("decode")
    roof_p = {"bound": "tensor", "achieved": pre_ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
              "frac": pre_ach / peaks["bf16_tflops"], "traffic": tr_p,
              "peak_source": "%s bf16 burst (MEASURED_PEAKS.json)" % psrc if psrc == "measured" else
              "fallback 1.8 PFLOP/s bf16",
              "frac_of_sustained": pre_ach / peaks.get("bf16_tflops_sustained", 1400.0),
              "algorithmic_flops_per_launch": flops_p, "kernel": "prefill_kernel<64>" if wp.D == 64 else
              "prefill_kernel<128>"}
    roof_d = {"bound": "hbm", "achieved": dec_ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
              "frac": dec_ach / peaks["hbm_gbs"], "traffic": tr_d,
              "algorithmic_bytes_per_launch": bytes_d, "kernels": "decode_split_kernel + combine_kernel"}

    # ---- end to end through the public API with host buffers (prefill)
    e2e = None
    if rank == 0 or ws > 1:
        hq = pin["q"].pin_memory()
        hk = pin["k"].pin_memory()
        hv = pin["v"].pin_memory()
        hl = None if pin["seqlens_k"] is None else pin["seqlens_k"].pin_memory()
        ho = torch.empty(out_p.shape, dtype=out_p.dtype).pin_memory()
        hlse = torch.empty(lse_p.shape, dtype=torch.float32).pin_memory()
        dq, dk, dv = torch.empty_like(P["q"]), torch.empty_like(P["k"]), torch.empty_like(P["v"])
        dl = None if hl is None else torch.empty_like(P["seqlens_k"])
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hl) if t is not None)
        d2h = ho.numel() * ho.element_size() + hlse.numel() * 4

        staging = {"q": dq, "k": dk, "v": dv, "out": out_p, "lse": lse_p}
        if dl is not None:
            staging["seqlens"] = dl

        def e2e_step():
            # the public host-buffer entry point: batch chunks whose copies in,
            # attention and copies out overlap on three streams
            gqa.gqa_fwd_host(hq, hk, hv, causal=wp.causal, seqlens_k=hl, scale=wp.scale, out=ho, lse=hlse,
                             staging=staging)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(ws)
        a.record()
        for _ in range(args.e2e_steps):
            e2e_step()
        b.record()
        torch.cuda.synchronize()
        e2e_s = _max_over_ranks(a.elapsed_time(b) / 1e3, ws, device)
        e2e = {"value": _whole_job_rate(flops_p, args.e2e_steps, ws, e2e_s) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "what": "prefill through gqa_fwd_host: pinned host inputs copied in and outputs copied out "
                       "every step, in batch chunks overlapped with the computation"}

    # ---- the other prefill workloads, timed the same way (not part of `value`)
    others = {}
    dec8 = None
    if not args.no_other_workloads:
        del P, pin, out_p, lse_p
        for name in [n for n in args.other_workloads.split(",") if n]:
            w = inputs.WORKLOADS[name]
            if isinstance(w, inputs.DecodeWorkload) and w.dtype == "fp8kv":
                dec8 = time_decode_fp8(gqa, name, device, flush, reps=max(args.other_reps, 1) * 2)
            elif name == args.prefill:
                others[name] = {"tflops": value / ws, "ms": pre_avg * 1e3}
            else:
                others[name] = time_prefill_workload(gqa, name, device, flush, reps=args.other_reps)
        torch.cuda.synchronize()
        if gqa.gqa_device_status() != 0:
            raise RuntimeError("device error while timing the other prefill workloads")
    bwd = {}
    if not args.no_other_workloads:
        for name in [n for n in args.backward_workloads.split(",") if n]:
            bwd[name] = time_backward(gqa, name, device, flush, reps=args.other_reps)
        torch.cuda.synchronize()
        if gqa.gqa_device_status() != 0:
            raise RuntimeError("device error while timing the backward")

    cb = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(args.prefill)

    launches_per_step = 1 + 1 + (1 if nsplit > 1 else 0)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": total_s * 1e3 / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": _workload_name(wp) + " + " + (
                "%s decode B%d Hq%d Hkv%d D%d Smax%d cache lengths U[%d,%d]" % (
                    wd.name, wd.B, wd.Hq, wd.Hkv, wd.D, wd.Smax, wd.lens[0], wd.lens[1])),
                "l2": "256 MB L2 flush before every step; decode inputs (2.1 GB caches) exceed L2",
                "parallelism": "replicas" if ws > 1 else "single GPU",
                "prefill_ms": pre_avg * 1e3, "decode_ms": dec_avg * 1e3, "decode_num_splits": nsplit,
                "warmup": "%d steps and >= %.1f s of back-to-back steps inside the clock sampler, "
                          "immediately before the timed steps" % (args.warmup, args.warmup_seconds),
                "step": "%d passes (L2 flush, prefill, decode) per timed step, so that the %d steps take "
                        ">= %.0f ms; prefill_ms / decode_ms are per pass" % (R, K, args.min_timed_ms)},
            "per_step": per_step,
            "roofline": roof_p,
            "decode": {"value": dec_gbs, "unit": "GB/s (KV-cache bytes read / decode time)",
                       "roofline": roof_d, "kv_bytes_per_step": kv_bytes_d},
            "clocks": clk,
            "e2e": e2e,
            "gpu_launches": launches_per_step * K * R,
            "cpu_baseline": cb,
            "prefill_workloads": others,
            "decode_fp8": dec8,
            "backward": bwd,
        }
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
