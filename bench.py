#!/usr/bin/env python
"""Benchmark of the attention training step (forward + backward) on GB300.

One step = attn_fwd + attn_bwd_preprocess + attn_bwd + attn_bwd_postprocess over
the largest dense workload, causal GQA B=4, Hq=32, Hkv=8, S=4096, D=128 (bf16,
synthetic N(0,1) inputs); the headline value is its fwd+bwd TFLOP/s.  The same
line carries, under extra keys, the causal MHA B=8 H=32 S=1024 D=64 and the THD
varlen H=16 D=128 workloads (each timed the same way, with its own roofline), the
top-k sparse workload, and the CPU oracle's rate.  Prints one JSON line.
`--impl reference` times the fp64 CPU oracle on the headline workload instead
(one query head per step, on the host cores).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
           [--workload NAME] [--no-extras] [--no-sparse] [--no-split]
For N > 1 launch with torchrun; every rank runs the full workload (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from softmax_attention_backward_gb300 import workloads as W  # noqa: E402

METRIC = "attention fwd+bwd TFLOP/s (bf16, 1 GB300) and % of dense BF16 tensor peak"
DEFAULT_WORKLOAD = "gqa_causal_b4_h32x8_s4096_d128"
EXTRA_DENSE = ("mha_causal_b8_h32_s1024_d64", "thd_varlen_causal_h16_d128")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dense_flops(w):
    """Algorithmic FLOPs: forward 4*B*H*S^2*D (x0.5 causal), backward 2.5x forward."""
    if w.kind == "thd":
        f = 4.0 * w.heads_q * w.head_dim * sum(n * n for n in w.lengths) * (0.5 if w.causal else 1)
    else:
        f = 4.0 * w.batch * w.heads_q * w.seqlen ** 2 * w.head_dim * (0.5 if w.causal else 1.0)
    return f, 2.5 * f


def source_sha(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def profiled_traffic(kernel, workload, src_rel):
    """dram bytes per launch from a committed ncu summary, if the kernel source
    has not changed since it was captured (else None)."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    sha = source_sha(src_rel)
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        text = open(os.path.join(pdir, fn)).read()
        fields = dict(re.findall(r"^\s*[-*]?\s*([a-z_0-9]+):\s*`?([^`\n]+)`?\s*$", text, re.M))
        if (fields.get("kernel") == kernel and fields.get("workload") == workload
                and fields.get("source_sha256") == sha and "dram_bytes_per_launch" in fields):
            return float(fields["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """Samples nvidia-smi every 50 ms while active; keeps samples inside marks."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        self.samples, self.t0, self.t1 = [], None, None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [s for t, s in self.samples if self.t0 - 0.06 <= t <= self.t1 + 0.06]
        if not inside and self.samples:   # timed region shorter than the period
            mid = 0.5 * (self.t0 + self.t1)
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - mid))[1]]
        sm, smax, reasons = [], [], set()
        for s in inside:
            try:
                sm.append(float(s[0]))
                smax.append(float(s[1]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(self.NAMES, s[3:7]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def reduce_max(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------
# oracle (CPU) leg
# ----------------------------------------------------------------------------
def oracle_units(w):
    """Independent samples of a workload for the oracle, with their FLOPs
    (fwd+bwd): one query head of one batch entry (its O, LSE, dQ and its share of
    dK/dV) for a dense problem, one sequence of a THD problem."""
    causal = 0.5 if w.causal else 1.0
    if w.kind == "thd":
        per = [3.5 * 4.0 * w.heads_q * w.head_dim * L * L * causal for L in w.lengths]
        return [(n, per[n]) for n in range(len(w.lengths))]
    per = 3.5 * 4.0 * w.seqlen * w.seqlen * w.head_dim * causal
    return [((b, h), per) for b in range(w.batch) for h in range(w.heads_q)]


def oracle_unit_rate(w, x, budget_s, start=0):
    """Times the fp64 oracle over independent samples until `budget_s` is spent
    (at least one).  Returns (TFLOP/s, samples done, seconds)."""
    import oracle
    units = oracle_units(w)
    if w.kind != "thd":
        q, k, v, do = (x[n].double() for n in ("q", "k", "v", "do"))
        mask = oracle.causal_mask(w.seqlen, w.seqlen) if w.causal else \
            oracle.full_mask(w.seqlen, w.seqlen)
        grp = w.heads_q // w.heads_kv
    done, flops, t0 = 0, 0.0, time.perf_counter()
    while True:
        u, f = units[(start + done) % len(units)]
        if w.kind == "thd":
            oracle.thd_backward(x["q"], x["k"], x["v"], x["do"], x["cu_seqlens"], w.scale, w.causal,
                                seqs=[u])
        else:
            b, h = u
            oracle.head_backward(q[b, :, h], k[b, :, h // grp], v[b, :, h // grp], do[b, :, h],
                                 w.scale, mask)
        done += 1
        flops += f
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return flops / el / 1e12, done, el


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    torch.set_num_threads(len(os.sched_getaffinity(0)))
    x = W.make_inputs(w)
    cores = torch.get_num_threads()
    for i in range(args.warmup):
        oracle_unit_rate(w, x, 0.0, start=i)
    times, units, flops = [], 0, 0.0
    for i in range(args.steps):
        rate, n, el = oracle_unit_rate(w, x, 0.0, start=args.warmup + i)
        times.append(el)
        units += n
        flops += rate * el * 1e12
    total = sum(times)
    value = flops / total / 1e12
    what = "sequence" if w.kind == "thd" else "query head (one batch entry)"
    sample = f"{units} samples of {w.name}, one {what} per step, fp64 oracle fwd+bwd"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, world):
    c = {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "heads_q": w.heads_q,
         **({"lengths": w.lengths, "capacity": w.capacity} if w.kind == "thd" else {}),
         "heads_kv": w.heads_kv, "head_dim": w.head_dim, "causal": w.causal, "dq_mode": "atomic",
         "l2": "flushed between timed steps (256 MiB write)",
         "parallelism": "replicas" if world == 1 else f"replicas x{world}"}
    return c


def cpu_baseline(w, seconds):
    torch.set_num_threads(len(os.sched_getaffinity(0)))
    x = W.make_inputs(w)
    rate, units, el = oracle_unit_rate(w, x, seconds)
    what = "sequences" if w.kind == "thd" else "query heads"
    return {"value": rate, "unit": "TFLOP/s", "cores": torch.get_num_threads(), "kind": "oracle",
            "sample": f"{units} {what} of {w.name} (fwd+bwd, fp64) in {el:.1f} s"}


# ----------------------------------------------------------------------------
# our leg: one dense workload
# ----------------------------------------------------------------------------
def tflops(flops, ms):
    return flops / (ms * 1e-3) / 1e12


def dense_pass_bytes(w):
    """Algorithmic bytes of the two memory-bound passes (atomic dQ mode).
    Preprocess: reads O and dO, writes Delta and clears the fp32 accumulator row,
    for every valid row-head.  Postprocess: reads the accumulator and writes bf16
    dQ for every valid row-head, and writes the exact zeros of THD padding rows of
    dQ, dK and dV."""
    D = w.head_dim
    if w.kind == "thd":
        valid = sum(w.lengths)
        pad = w.capacity - valid
    else:
        valid, pad = w.batch * w.seqlen, 0
    rh = valid * w.heads_q
    pre = rh * (2 * D * 2 + 4 + 4 * D)
    post = rh * (4 * D + 2 * D) + pad * (w.heads_q + 2 * w.heads_kv) * D * 2
    return pre, post


def bench_dense(args, w, dev, flush, world, rank, sampler=None, e2e=False):
    """Times K steps of fwd + preprocess + bwd + postprocess (atomic dQ; then split
    dQ unless --no-split) and returns the per-workload block of the JSON line."""
    import softmax_attention_backward_gb300 as A
    x = W.make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    if w.kind == "thd":
        lse = torch.empty(w.heads_q, w.capacity, dtype=torch.float32, device=dev)
    else:
        lse = torch.empty(w.batch, w.heads_q, w.seqlen, dtype=torch.float32, device=dev)
    delta = torch.empty_like(lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    kw = dict(causal=w.causal, scale=w.scale)
    if w.kind == "thd":
        kw.update(cu_seqlens=x["cu_seqlens"].to(dev), max_seqlen=max(w.lengths))
    ws = {}
    modes = (A.ATTN_DQ_ATOMIC,) if args.no_split else (A.ATTN_DQ_ATOMIC, A.ATTN_DQ_SPLIT)
    for mode in modes:
        n = A.attn_bwd_workspace_size(q, k, mode=mode, **kw)
        ws[mode] = torch.empty(n, dtype=torch.uint8, device=dev)
    f_fwd, f_bwd = dense_flops(w)
    stream = torch.cuda.current_stream()

    def step(mode, ev=None):
        if ev:
            ev[0].record(stream)
        A.attn_fwd(q, k, v, out=o, lse=lse, **kw)
        if ev:
            ev[1].record(stream)
        A.attn_bwd_preprocess(q, k, o, do, mode=mode, workspace=ws[mode], delta=delta, **kw)
        if ev:
            ev[2].record(stream)
        A.attn_bwd(q, k, v, do, lse, delta, mode=mode, workspace=ws[mode], dk=dk, dv=dv, **kw)
        if ev:
            ev[3].record(stream)
        A.attn_bwd_postprocess(q, k, dk, dv, mode=mode, workspace=ws[mode], dq=dq, **kw)
        if ev:
            ev[4].record(stream)

    def timed(mode, steps, smp=None):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
        barrier(world)
        torch.cuda.synchronize()
        if smp:
            smp.mark_start()
        for i in range(steps):
            flush.zero_()
            step(mode, evs[i])
        torch.cuda.synchronize()
        if smp:
            smp.mark_end()
        barrier(world)
        r = {}
        for key, a, b in (("total", 0, 4), ("fwd", 0, 1), ("bwd", 1, 4), ("pre", 1, 2),
                          ("main", 2, 3), ("post", 3, 4)):
            r[key] = reduce_max(sum(e[a].elapsed_time(e[b]) for e in evs) / steps, world)
        return r

    for _ in range(args.warmup):
        for mode in modes:
            step(mode)
    torch.cuda.synchronize()
    t_at = timed(A.ATTN_DQ_ATOMIC, args.steps, sampler)
    t_sp = None if args.no_split else timed(A.ATTN_DQ_SPLIT, args.steps)
    del ws
    ws_split_bytes = 0 if args.no_split else A.attn_bwd_workspace_size(
        q, k, mode=A.ATTN_DQ_SPLIT, **kw)

    pk, pk_kind = peaks()
    peak, hbm = pk["bf16_tflops"], pk["hbm_gbs"]
    pre_b, post_b = dense_pass_bytes(w)
    src = "softmax_attention_backward_gb300/csrc/"
    D = w.head_dim
    # the dominant kernel: head_dim 64 and 128 have kernels of their own
    bwd_kernel, bwd_src = (("attn_bwd_kernel<64>", "attn_bwd.cu") if D == 64
                           else ("attn_bwd128_kernel", "attn_bwd_d128.cu"))
    blk = {
        "workload": w.name,
        "fwd_bwd_tflops": tflops(f_fwd + f_bwd, t_at["total"]),
        "pct_of_peak": 100.0 * tflops(f_fwd + f_bwd, t_at["total"]) / peak,
        "fwd_tflops": tflops(f_fwd, t_at["fwd"]), "bwd_tflops": tflops(f_bwd, t_at["bwd"]),
        "ms_per_step": t_at["total"],
        "ms_breakdown": {"fwd": t_at["fwd"], "bwd_preprocess": t_at["pre"],
                         "bwd_main": t_at["main"], "bwd_postprocess": t_at["post"]},
        "flops": {"fwd": f_fwd, "bwd": f_bwd},
        "split": None if t_sp is None else {
            "fwd_bwd_tflops": tflops(f_fwd + f_bwd, t_sp["total"]),
            "bwd_tflops": tflops(f_bwd, t_sp["bwd"]), "ms_per_step": t_sp["total"],
            "ms_breakdown": {"fwd": t_sp["fwd"], "bwd_preprocess": t_sp["pre"],
                             "bwd_main": t_sp["main"], "bwd_postprocess": t_sp["post"]},
            "workspace_bytes": ws_split_bytes},
        "roofline": {"kernel": bwd_kernel, "bound": "tensor",
                     "achieved": tflops(f_bwd, t_at["main"]), "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops(f_bwd, t_at["main"]) / peak,
                     "peak_kind": f"{pk_kind} bf16 burst",
                     "traffic": profiled_traffic(bwd_kernel.split("<")[0], w.name, src + bwd_src),
                     "flops_per_launch": f_bwd},
        "fwd_roofline": {"kernel": f"attn_fwd_kernel<{D}>", "bound": "tensor",
                         "achieved": tflops(f_fwd, t_at["fwd"]), "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops(f_fwd, t_at["fwd"]) / peak,
                         "peak_kind": f"{pk_kind} bf16 burst",
                         "traffic": profiled_traffic("attn_fwd_kernel", w.name,
                                                     src + "attn_fwd.cu"),
                         "flops_per_launch": f_fwd},
        "hbm_passes": {
            name: {"kernel": kern, "bound": "hbm", "us": 1e3 * ms, "bytes": b,
                   "achieved": b / ms / 1e6, "peak": hbm, "unit": "GB/s",
                   "frac": b / ms / 1e6 / hbm, "peak_kind": f"{pk_kind} copy",
                   "traffic": profiled_traffic(kern, w.name, src + "attn_bwd_aux.cu")}
            for name, kern, ms, b in (
                ("bwd_preprocess", "attn_bwd_preprocess_kernel", t_at["pre"], pre_b),
                ("bwd_postprocess", "attn_dq_finalize_kernel", t_at["post"], post_b))},
        "launches_per_step": 5 if w.kind == "thd" else 4,
    }
    if not e2e:
        return blk
    blk["e2e"] = bench_e2e(args, A, dev, x, (q, k, v, do), (o, lse, delta, dq, dk, dv), kw,
                           f_fwd + f_bwd, world)
    return blk


def bench_e2e(args, A, dev, x, ins, outs, kw, flops, world):
    """End to end through the public API: pinned host inputs -> device -> results
    -> host, every step.  Three streams overlap step i's compute with the
    host->device copy of step i+1's inputs and the device->host copy of step
    i-1's gradients (inputs and gradients double-buffered on the device and on
    the host)."""
    q, k, v, do = ins
    o, lse, delta, dq, dk, dv = outs
    stream = torch.cuda.current_stream()
    ws = torch.empty(A.attn_bwd_workspace_size(q, k, mode=A.ATTN_DQ_ATOMIC, **kw),
                     dtype=torch.uint8, device=dev)
    hin = [[x[n].pin_memory() for n in ("q", "k", "v", "do")]]
    hin.append([t.clone().pin_memory() for t in hin[0]])
    dins = [[q, k, v, do], [torch.empty_like(t) for t in (q, k, v, do)]]
    douts = [[dq, dk, dv], [torch.empty_like(t) for t in (dq, dk, dv)]]
    hout = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
            for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in hin[0])
    d2h = sum(t.numel() * t.element_size() for t in hout[0])
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = torch.cuda.Event
    in_ready, in_free, out_ready, out_free = ([ev(), ev()] for _ in range(4))
    for e_ in in_free + out_free:
        e_.record(stream)

    def e2e_step(i):
        b = i & 1
        qi, ki, vi, doi = dins[b]
        dqi, dki, dvi = douts[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(in_free[b])
            for d_, h_ in zip(dins[b], hin[b]):
                d_.copy_(h_, non_blocking=True)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_free[b])
        A.attn_fwd(qi, ki, vi, out=o, lse=lse, stream=stream, **kw)
        A.attn_bwd_preprocess(qi, ki, o, doi, mode=A.ATTN_DQ_ATOMIC, workspace=ws, delta=delta,
                              stream=stream, **kw)
        A.attn_bwd(qi, ki, vi, doi, lse, delta, mode=A.ATTN_DQ_ATOMIC, workspace=ws, dk=dki,
                   dv=dvi, stream=stream, **kw)
        A.attn_bwd_postprocess(qi, ki, dki, dvi, mode=A.ATTN_DQ_ATOMIC, workspace=ws, dq=dqi,
                               stream=stream, **kw)
        in_free[b].record(stream)
        out_ready[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(out_ready[b])
            for h_, d_ in zip(hout[b], douts[b]):
                h_.copy_(d_, non_blocking=True)
            out_free[b].record(s_out)

    for i in range(max(1, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_stream(s_out)
    e_end.record(stream)
    torch.cuda.synchronize()
    ms_e2e = reduce_max(e_start.elapsed_time(e_end) / args.steps, world)
    # the last step's gradients must have reached the host intact
    for h_, d_ in zip(hout[(args.steps - 1) & 1], douts[(args.steps - 1) & 1]):
        assert torch.equal(h_, d_.cpu())
    return {"value": world * tflops(flops, ms_e2e), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
            "overlap": "h2d(i+1) | compute(i) | d2h(i-1) on three streams"}


def run_ours(args, w, world, rank, local):
    import softmax_attention_backward_gb300 as A
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    A.lib()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sampler = ClockSampler(f"GPU-{torch.cuda.get_device_properties(dev).uuid}") if rank == 0 else None
    head = bench_dense(args, w, dev, flush, world, rank, sampler=sampler, e2e=True)
    clocks = sampler.stop() if sampler else None
    torch.cuda.empty_cache()

    extra = {}
    if not args.no_extras:
        configs = {}
        for name in EXTRA_DENSE:
            if name != w.name:
                configs[name] = bench_dense(args, W.get_workload(name), dev, flush, world, rank)
                torch.cuda.empty_cache()
        extra["configs"] = configs
        if rank == 0 and not args.no_sparse:
            extra["sparse"] = bench_sparse(args, dev, flush)
            torch.cuda.empty_cache()
        if rank == 0:
            extra["csa_compressor"] = bench_csa(args, dev, flush)
            torch.cuda.empty_cache()
            extra["dsa_indexer"] = bench_indexer(args, dev, flush)
            torch.cuda.empty_cache()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": world * head["fwd_bwd_tflops"], "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(w, world),
        "pct_of_peak": head["pct_of_peak"],
        "fwd_tflops": head["fwd_tflops"], "bwd_tflops": head["bwd_tflops"],
        "ms_breakdown": head["ms_breakdown"], "split": head["split"],
        "roofline": head["roofline"], "fwd_roofline": head["fwd_roofline"],
        "hbm_passes": head["hbm_passes"],
        "cpu_baseline": cpu_baseline(w, args.cpu_seconds) if args.cpu_seconds > 0 else None,
        "clocks": clocks,
        "e2e": head["e2e"],
        "gpu_launches": head["launches_per_step"] * args.steps,
        **extra,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# top-k sparse workload
# ----------------------------------------------------------------------------
def sparse_logical_bytes(T, H, idx):
    """Logical bytes of the sparse path: gathered KV rows (576 bf16 once per
    token and selected key), Q, O, idx; backward adds dO, dQ and 576 fp32
    atomic adds (4 bytes each) per selected key."""
    pairs = int((idx >= 0).sum().item())
    q_b, o_b = T * H * 576 * 2, T * H * 512 * 2
    idx_b = idx.numel() * 4
    gather = pairs * 576 * 2
    fwd = q_b + gather + idx_b + o_b + T * H * 4
    bwd = q_b + gather + idx_b + 2 * o_b + T * H * 4 + T * H * 576 * 2 + pairs * 576 * 4
    return fwd, bwd, pairs


def bench_sparse(args, dev, flush):
    import softmax_attention_backward_gb300 as A
    w = W.get_workload("sparse_topk2048_t8192_h64")
    x = W.make_inputs(w)
    q, kv, do, idx = (x[n].to(dev) for n in ("q", "kv", "do", "idx"))
    o = torch.empty(w.seqlen, w.heads_q, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.seqlen, w.heads_q, dtype=torch.float32, device=dev)
    dq, dkv = torch.empty_like(q), torch.empty_like(kv)
    ws = torch.empty(A.sparse_attn_bwd_workspace_size(q, idx), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, 10))
    for _ in range(3):
        A.sparse_attn_fwd(q, kv, idx, scale=w.scale, out=o, lse=lse)
        A.sparse_attn_bwd(q, kv, idx, o, do, lse, scale=w.scale, workspace=ws, dq=dq, dkv=dkv)
    f_ms, b_ms = [], []
    for _ in range(steps):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        A.sparse_attn_fwd(q, kv, idx, scale=w.scale, out=o, lse=lse)
        e[1].record(stream)
        A.sparse_attn_bwd(q, kv, idx, o, do, lse, scale=w.scale, workspace=ws, dq=dq, dkv=dkv)
        e[2].record(stream)
        torch.cuda.synchronize()
        f_ms.append(e[0].elapsed_time(e[1]))
        b_ms.append(e[1].elapsed_time(e[2]))
    # deterministic dKV (private slabs summed in slab order): same inputs, its own
    # workspace; bitwise repeat
    # checked on the last two runs
    del ws
    wsd = torch.empty(A.sparse_attn_bwd_deterministic_workspace_size(q, idx), dtype=torch.uint8,
                      device=dev)
    dkv_prev = torch.empty_like(kv)
    d_ms = []
    for i in range(2 + steps):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e[0].record(stream)
        A.sparse_attn_bwd_deterministic(q, kv, idx, o, do, lse, scale=w.scale, workspace=wsd,
                                        dq=dq, dkv=dkv)
        e[1].record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            d_ms.append(e[0].elapsed_time(e[1]))
        if i == 1 + steps - 1:
            dkv_prev.copy_(dkv)
    repeat_equal = bool(torch.equal(dkv_prev, dkv))
    ws_det = wsd.numel()
    del wsd
    fb, bb, pairs = sparse_logical_bytes(w.seqlen, w.heads_q, x["idx"])
    fm, bm = sum(f_ms) / steps, sum(b_ms) / steps
    dm = sum(d_ms) / len(d_ms)
    pk, pk_kind = peaks()
    hbm = pk["hbm_gbs"]
    flops_f = pairs * w.heads_q * 2 * (576 + 512)
    flops_b = pairs * w.heads_q * 2 * (3 * 576 + 2 * 512)
    src = "softmax_attention_backward_gb300/csrc/"
    return {"workload": w.name, "steps": steps, "fwd_ms": fm, "bwd_ms": bm,
            "fwd_logical_gbs": fb / fm / 1e6, "bwd_logical_gbs": bb / bm / 1e6,
            "fwd_frac_hbm": fb / fm / 1e6 / hbm, "bwd_frac_hbm": bb / bm / 1e6 / hbm,
            "fwd_tflops": flops_f / fm / 1e9, "bwd_tflops": flops_b / bm / 1e9,
            "roofline": {"kernel": "sparse_bwd_tc_kernel (+ preprocess, cast)", "bound": "hbm",
                         "achieved": bb / bm / 1e6, "peak": hbm, "unit": "GB/s",
                         "frac": bb / bm / 1e6 / hbm, "peak_kind": f"{pk_kind} copy",
                         "bytes": "logical (gathered KV rows once per token, fp32 dKV adds)",
                         "traffic": profiled_traffic("sparse_bwd_tc_kernel", w.name,
                                                     src + "sparse_bwd_tc.cu")},
            "bwd_deterministic_ms": dm, "bwd_deterministic_bitwise_repeat": repeat_equal,
            "bwd_deterministic_workspace_bytes": ws_det,
            "valid_pairs": pairs}


# ----------------------------------------------------------------------------
# CSA compressor gated pooling (HBM-bound)
# ----------------------------------------------------------------------------
# Kernel times the compressor page reports on one B200 (nsys kernel sums, after
# its forward vectorization and backward zero-write commits; the backward
# includes its dAPE zero fill).  Context only: other hardware.
CSA_PAGE_B200_US = {"csa_1x8192_d128": (4.5, 12.8), "csa_3x8192_d128": (10.0, 22.2),
                    "csa_1x8192_d512": (12.4, 22.8), "csa_3x8192_d512": (35.0, 66.0)}


def csa_bytes(x, ratio, coff):
    """Algorithmic bytes: the forward reads kv and score at every (token, column)
    some window reads, ape, and writes out; the backward reads the same plus
    dout and writes every dkv / dscore position and dape."""
    D = x["kv"].shape[1] // coff
    cu, cc = x["cu_seqlens"].tolist(), x["cu_seqlens_comp"].tolist()
    used = 0
    for n in range(len(cu) - 1):
        nb = cc[n + 1] - cc[n]
        used += nb * ratio * D if coff == 1 else max(0, 2 * nb - 1) * ratio * D
    ape = x["ape"].numel() * 4
    out = x["comp_capacity"] * D * 2
    fwd = used * 4 + ape + out
    bwd = used * 4 + ape + out + x["kv"].numel() * 2 * 2 + ape
    return fwd, bwd


def bench_csa(args, dev, flush):
    import softmax_attention_backward_gb300 as A
    hbm = peaks()[0]["hbm_gbs"]
    pk_kind = peaks()[1]
    res = {}
    iters = max(5, min(args.steps, 20))
    for name, c in W.CSA_WORKLOADS.items():
        x = W.csa_inputs(c["lengths"], c["head_dim"], c["ratio"], c["coff"], c["seed"])
        g = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
        kw = dict(ratio=c["ratio"], coff=c["coff"])
        out = torch.empty(x["comp_capacity"], c["head_dim"], dtype=torch.bfloat16, device=dev)
        dkv, dsc, dape = torch.empty_like(g["kv"]), torch.empty_like(g["score"]), \
            torch.empty_like(g["ape"])
        ws = torch.empty(A.csa_compressor_bwd_workspace_size(
            g["kv"], g["cu_seqlens"], g["cu_seqlens_comp"], comp_capacity=x["comp_capacity"],
            **kw), dtype=torch.uint8, device=dev)

        def fwd():
            A.csa_compressor_fwd(g["kv"], g["score"], g["ape"], g["cu_seqlens"],
                                 g["cu_seqlens_comp"], comp_capacity=x["comp_capacity"], out=out,
                                 **kw)

        def bwd():
            A.csa_compressor_bwd(g["kv"], g["score"], g["ape"], g["dout"], g["cu_seqlens"],
                                 g["cu_seqlens_comp"], workspace=ws, dkv=dkv, dscore=dsc,
                                 dape=dape, **kw)

        times = {key: _time(fn, flush, iters) for key, fn in (("fwd", fwd), ("bwd", bwd))}
        fb, bb = csa_bytes(x, c["ratio"], c["coff"])
        page = CSA_PAGE_B200_US[name]
        res[name] = {
            "fwd_us": 1e3 * times["fwd"], "bwd_us": 1e3 * times["bwd"],
            "fwd_gbs": fb / times["fwd"] / 1e6, "bwd_gbs": bb / times["bwd"] / 1e6,
            "fwd_frac_hbm": fb / times["fwd"] / 1e6 / hbm,
            "bwd_frac_hbm": bb / times["bwd"] / 1e6 / hbm,
            "bytes": {"fwd": fb, "bwd": bb},
            "page_b200_us": {"fwd": page[0], "bwd": page[1]},
        }
    return {"ratio": 4, "coff": 2, "iters": iters, "timing": "median of CUDA-graph replays, L2 flushed before each",
            "peak": hbm, "peak_kind": f"{pk_kind} copy", "launches_per_bwd": 2,
            "roofline": {"kernel": "csa_bwd_kernel<4,2> (+ dape reduce) at csa_3x8192_d512",
                         "bound": "hbm", "achieved": res["csa_3x8192_d512"]["bwd_gbs"],
                         "peak": hbm, "unit": "GB/s",
                         "frac": res["csa_3x8192_d512"]["bwd_frac_hbm"],
                         "traffic": profiled_traffic(
                             "csa_bwd_kernel", "csa_3x8192_d512",
                             "softmax_attention_backward_gb300/csrc/csa_compressor.cu")},
            "shapes": res}


# ----------------------------------------------------------------------------
# DSA lightning indexer (logits, top-k, backward) and the sparse KL loss
# ----------------------------------------------------------------------------
def _time(fn, flush, iters):
    """Median device time of fn's launches after an L2 flush, replayed from a
    CUDA graph captured once: the host work of the Python binding stays out of
    the timed region (for a few-microsecond kernel it takes longer than the
    flush, and the GPU would sit idle inside the events waiting for the launch)."""
    stream = torch.cuda.current_stream()
    for _ in range(3):
        fn()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    torch.cuda.synchronize()
    ms = []
    for _ in range(iters):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    return statistics.median(ms)


def bench_indexer(args, dev, flush):
    import softmax_attention_backward_gb300 as A
    c = W.INDEXER_WORKLOAD
    T, H, K = c["tokens"], c["heads"], c["topk"]
    x = W.indexer_inputs(T, H, c["seed"], topk=K)
    q, k, w, g = (x[n].to(dev) for n in ("q", "k", "w", "grad"))
    logits = torch.empty(T, A.logits_ld(T), dtype=torch.float32, device=dev)
    idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    length = torch.empty(T, dtype=torch.int32, device=dev)
    scores = torch.empty(T, K, dtype=torch.float32, device=dev)
    dq, dk, dw = torch.empty_like(q), torch.empty_like(k), torch.empty_like(w)
    iters = max(5, min(args.steps, 20))
    pk, pk_kind = peaks()
    peak, hbm = pk["bf16_tflops"], pk["hbm_gbs"]
    t_fwd = _time(lambda: A.dsa_indexer_fwd(q, k, w, logits=logits), flush, iters)
    t_topk = _time(lambda: A.dsa_topk(logits, K, heads=H, idx=idx, length=length, scores=scores),
                   flush, iters)
    t_bwd = _time(lambda: A.dsa_indexer_bwd(q, k, w, idx, g, dq=dq, dk=dk, dw=dw), flush, iters)
    pairs_causal = T * (T + 1) // 2                  # (query, key) pairs the logits cover
    sel = int((idx >= 0).sum().item())               # selected (query, key) pairs
    f_fwd = 2.0 * pairs_causal * H * W.INDEXER_D
    f_bwd = 3 * 2.0 * sel * H * W.INDEXER_D
    b_topk = pairs_causal * 4 + T * K * 8 + T * 4    # visible logits read; idx, scores, length
    # sparse KL on the sparse attention workload (the indexer's training signal)
    ws, xs = W.get_workload("sparse_topk2048_t8192_h64"), None
    xs = W.make_inputs(ws)
    gq, gkv, gidx = xs["q"].to(dev), xs["kv"].to(dev), xs["idx"].to(dev)
    _, lse = A.sparse_attn_fwd(gq, gkv, gidx, scale=ws.scale)
    sc = torch.randn(gidx.shape, generator=torch.Generator().manual_seed(9)).to(dev)
    loss = torch.empty(ws.seqlen, dtype=torch.float32, device=dev)
    kgrad = torch.empty_like(sc)
    t_kl = _time(lambda: A.dsa_sparse_kl(gq, gkv, lse, gidx, sc, scale=ws.scale, loss=loss,
                                         grad=kgrad), flush, iters)
    kl_pairs = int((xs["idx"] >= 0).sum().item())
    f_kl = 2.0 * kl_pairs * ws.heads_q * 576
    tf = lambda f, ms: f / (ms * 1e-3) / 1e12
    return {
        "workload": c["name"], "iters": iters, "timing": "median of CUDA-graph replays, L2 flushed before each",
        "fwd": {"kernel": "dsa_indexer_logits_kernel", "us": 1e3 * t_fwd, "tflops": tf(f_fwd, t_fwd),
                "frac": tf(f_fwd, t_fwd) / peak, "flops": f_fwd},
        "topk": {"kernel": "dsa_topk_kernel", "us": 1e3 * t_topk, "gbs": b_topk / t_topk / 1e6,
                 "frac_hbm": b_topk / t_topk / 1e6 / hbm, "bytes": b_topk},
        "bwd": {"kernel": "dsa_indexer_bwd_kernel (+ zero, cast)", "us": 1e3 * t_bwd,
                "tflops": tf(f_bwd, t_bwd), "frac": tf(f_bwd, t_bwd) / peak, "flops": f_bwd,
                "selected_pairs": sel},
        "sparse_kl": {"kernel": "dsa_sparse_kl_kernel", "workload": ws.name, "us": 1e3 * t_kl,
                      "tflops": tf(f_kl, t_kl), "frac": tf(f_kl, t_kl) / peak, "flops": f_kl},
        "peak": {"bf16_tflops": peak, "hbm_gbs": hbm, "kind": f"{pk_kind} (bf16 burst, copy)"},
        "roofline": {"kernel": "dsa_indexer_logits_kernel", "bound": "tensor",
                     "achieved": tf(f_fwd, t_fwd), "peak": peak, "unit": "TFLOP/s",
                     "frac": tf(f_fwd, t_fwd) / peak,
                     "traffic": profiled_traffic("dsa_indexer_logits_kernel", c["name"],
                                                 "softmax_attention_backward_gb300/csrc/dsa_indexer.cu")},
    }


def run_leg(args, local):
    """One extra leg alone (sparse, CSA compressor or indexer), printed as its own
    JSON object; used by the profiling commands, not a bench line."""
    import softmax_attention_backward_gb300 as A
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    A.lib()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    fn = {"sparse": bench_sparse, "csa": bench_csa, "indexer": bench_indexer}[args.leg]
    print(json.dumps({"leg": args.leg, "result": fn(args, dev, flush)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-extras", action="store_true",
                    help="time only --workload (no other dense workloads, no sparse)")
    ap.add_argument("--no-sparse", action="store_true")
    ap.add_argument("--no-split", action="store_true", help="time only the atomic dQ mode")
    ap.add_argument("--leg", choices=["all", "sparse", "csa", "indexer"], default="all",
                    help="run one extra leg alone and print its block (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    w = W.get_workload(args.workload)
    if w.kind == "sparse":
        raise SystemExit("the sparse workload is timed inside every default run (key 'sparse')")
    if args.impl == "reference":
        run_reference(args, w, world, rank)
    elif args.leg != "all":
        run_leg(args, local)
    else:
        run_ours(args, w, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
