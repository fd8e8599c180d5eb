#!/usr/bin/env python
"""Benchmark of the fused relative-position attention on GB300.

One step = the whole hot path on one batch: forward (bias built in-kernel, varlen, online
softmax) and backward (preprocess, main kernel with the table gradient, finalize), all through
the library's C ABI. Reports bf16 attention TFLOP/s (4*L^2*d per head and document for the
forward, halved when causal; 2.5x that for the backward) and the fraction of the measured
tensor-core peak. Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|INDEX] [--impl reference]
Under torchrun each rank runs its own replica of the workload (independent problems, no
collective on the data path: weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "bf16 attention TFLOP/s fwd & fwd+bwd (T5-bias, varlen) vs tensor-core peak"
# the largest single-GPU workload: long-context T5 encoder, 1 x 16384 tokens, 12 heads, d 64
DEFAULT_WORKLOAD = 4
L2_FLUSH_BYTES = 256 << 20  # > 129 MB of L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def max_over_ranks(x, device):
    """The largest value of x over the ranks of the default process group (the slowest replica
    sets the job's time); x itself without one."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(step_flops, world, ms):
    """Whole-job throughput: every replica does step_flops per step of ms milliseconds."""
    return step_flops * world / ms / 1e9


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=str(DEFAULT_WORKLOAD))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true",
                    help="timed steps only: no e2e, clocks, CPU baseline or extra workloads "
                         "(for profiler launch lists)")
    ap.add_argument("--next-rows", action="store_true",
                    help="only the cross-attention, decode and RoPE figures, as one JSON line (for "
                         "profiling those kernels)")
    ap.add_argument("--aux-kernels", action="store_true",
                    help="only the RMSNorm and cross-entropy figures, as one JSON line (for "
                         "profiling those kernels)")
    return ap.parse_args()


def pick_workload(spec):
    from attention_relative_position_gb300 import workloads as wl
    if spec.isdigit():
        return wl.WORKLOADS[int(spec)]
    return wl.by_name(spec)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def workload_config(w, world, l2_note):
    return {
        "workload": w.name,
        "description": w.description,
        "num_docs": len(w.seqlens),
        "tokens_per_gpu": w.total_tokens,
        "global_tokens": w.total_tokens * world,
        "max_seqlen": w.max_seqlen,
        "num_heads": w.num_heads,
        "head_dim": w.head_dim,
        "t5_bias": (None if w.t5 is None else
                    {"num_buckets": w.t5[0], "max_distance": w.t5[1], "bidirectional": w.t5[2]}),
        "alibi": w.alibi,
        "causal": w.causal,
        "softmax_scale": w.scale,
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        "l2": l2_note,
    }


# -------------------------------------------------------------------------------------------
# clocks sampled by nvidia-smi while the timed loop runs
# -------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                n += 1
                for name, val in zip(names, parts[4:8]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


# -------------------------------------------------------------------------------------------
# the GPU arm
# -------------------------------------------------------------------------------------------
def lib_kwargs(w, x):
    t5 = w.t5 or (0, 0, True)
    return dict(bias_table=x["table"], alibi_slopes=x["slopes"], causal=w.causal,
                softmax_scale=w.scale, num_buckets=t5[0], max_distance=t5[1],
                bidirectional=t5[2])


class Runner:
    """Device-resident inputs, outputs and workspace for one workload; step() enqueues the whole
    hot path with CUDA events between the kernels."""

    def __init__(self, w, device):
        import torch
        import attention_relative_position_gb300 as fa
        from attention_relative_position_gb300 import workloads as wl
        self.torch, self.fa, self.w = torch, fa, w
        self.x = wl.make_inputs(w, device=device)
        x = self.x
        self.kw = lib_kwargs(w, x)
        self.out = torch.empty_like(x["q"])
        self.lse = torch.empty((w.num_heads, w.total_tokens), dtype=torch.float32, device=device)
        self.dq = torch.empty_like(x["q"])
        self.dk = torch.empty_like(x["q"])
        self.dv = torch.empty_like(x["q"])
        self.dtab = torch.empty_like(x["table"]) if x["table"] is not None else None
        nws = fa.fat_attn_bwd_workspace_size(w.total_tokens, w.num_heads, w.head_dim,
                                             len(w.seqlens), w.max_seqlen)
        self.ws = torch.empty(nws, dtype=torch.uint8, device=device)
        nfws = fa.fat_attn_fwd_workspace_size(w.total_tokens, len(w.seqlens), w.max_seqlen,
                                              w.num_heads, w.head_dim)
        self.fws = torch.empty(nfws, dtype=torch.uint8, device=device) if nfws else False
        # kernels one step launches: forward (+ split last wave and its merge), backward
        # preprocess, main (+ split last wave), finalize
        bws_min = fa.fat_attn_bwd_workspace_size(w.total_tokens, w.num_heads, w.head_dim)
        self.launches_per_step = 4 + (0 if w.causal else (2 if nfws else 0) +
                                      (1 if nws > bws_min else 0))
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.stream = torch.cuda.current_stream(device)

    def step(self):
        """One pass of the hot path through the public calls (forward, then the fused backward,
        whose main and finishing grids overlap the set-up of the grid before them)."""
        fa, x, w = self.fa, self.x, self.w
        fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, out=self.out,
                        lse=self.lse, workspace=self.fws, stream=self.stream, **self.kw)
        fa.fat_attn_bwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, self.out,
                        self.lse, x["dout"], workspace=self.ws, dq=self.dq, dk=self.dk,
                        dv=self.dv, dbias_table=self.dtab, stream=self.stream, **self.kw)

    def step_staged(self, events):
        """The same work as step(), backward as its three stage calls with CUDA events between
        the kernels (per-kernel times; no overlap between the grids)."""
        fa, x, w = self.fa, self.x, self.w
        events[0].record(self.stream)
        fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, out=self.out,
                        lse=self.lse, workspace=self.fws, stream=self.stream, **self.kw)
        between = None
        if events is not None:
            def between(i):
                if i >= 0:
                    events[i + 2].record(self.stream)
                else:
                    events[1].record(self.stream)
        fa.fat_attn_bwd_stages(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, self.out,
                               self.lse, x["dout"], self.ws, self.dq, self.dk, self.dv,
                               dbias_table=self.dtab, stream=self.stream, between=between,
                               **self.kw)

    def flush_l2(self):
        self.flush.zero_()



def time_steps(r, steps, flush=True):
    """Device times (ms, one entry per step; summarised by their median) of `steps` steps, L2 flushed between steps (not timed): "step" from
    steps through the public calls, each bracketed by CUDA events on the launching stream;
    the per-kernel times from as many steps run stage by stage with events between kernels."""
    torch = r.torch
    per = {"fwd": [], "bwd_pre": [], "bwd_main": [], "bwd_fin": [], "step": [], "step_staged": []}
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        if flush:
            r.flush_l2()
        evs[i][0].record(r.stream)
        r.step()
        evs[i][1].record(r.stream)
    torch.cuda.synchronize()
    per["step"] = [e[0].elapsed_time(e[1]) for e in evs]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for i in range(steps):
        if flush:
            r.flush_l2()
        r.step_staged(evs[i])
    torch.cuda.synchronize()
    for e in evs:
        t = [e[j].elapsed_time(e[j + 1]) for j in range(4)]
        per["fwd"].append(t[0])
        per["bwd_pre"].append(t[1])
        per["bwd_main"].append(t[2])
        per["bwd_fin"].append(t[3])
        per["step_staged"].append(sum(t))
    return per


def _packed(tensors, device, pin=False):
    """One flat byte buffer holding the given tensors (256-byte aligned) and views into it with
    the tensors' shapes and dtypes, so that a whole set moves with one copy."""
    import torch
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    flat = torch.empty(max(total, 1), dtype=torch.uint8, device=device, pin_memory=pin)
    views = [flat[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for o, t in zip(offs, tensors)]
    return flat, views


def e2e_steps(w, r, steps, nbuf=2):
    """Same metric through the public API from pinned host buffers: every step copies its
    inputs host->device, runs forward + backward, and copies out, dq, dk, dv (and the table
    gradient) back to host. Steps are pipelined as a training loop would run them: `nbuf` sets
    of device buffers and three streams, so the inputs of step i+1 are copied in and the results
    of step i-1 copied out while step i computes; each direction moves one packed buffer per
    step. The timed region runs from the first step's input copy to the last step's result
    copy."""
    torch, fa = r.torch, r.fa
    x = r.x
    names_in = [n for n in ("q", "k", "v", "dout", "cu_seqlens", "table", "slopes")
                if x[n] is not None]
    host_in_flat, host_in_views = _packed([x[n] for n in names_in], "cpu", pin=True)
    for v_, n in zip(host_in_views, names_in):
        v_.copy_(x[n].cpu())
    dev_in = []
    for _ in range(nbuf):
        flat, views = _packed([x[n] for n in names_in], x["q"].device)
        dev_in.append((flat, dict(zip(names_in, views))))
    out_names = ["out", "dq", "dk", "dv"] + (["dtab"] if r.dtab is not None else [])
    like = {"out": r.out, "dq": r.dq, "dk": r.dk, "dv": r.dv, "dtab": r.dtab}
    dev_out = []
    for _ in range(nbuf):
        flat, views = _packed([like[n] for n in out_names], x["q"].device)
        dev_out.append((flat, dict(zip(out_names, views))))
    host_out = [_packed([like[n] for n in out_names], "cpu", pin=True)[0] for _ in range(nbuf)]
    lse = [torch.empty_like(r.lse) for _ in range(nbuf)]
    ws = [torch.empty_like(r.ws) for _ in range(nbuf)]
    h2d = sum(x[n].numel() * x[n].element_size() for n in names_in)
    d2h = sum(like[n].numel() * like[n].element_size() for n in out_names)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_cmp = r.stream
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]    # inputs of the buffer set copied in
    ev_cmp = [torch.cuda.Event() for _ in range(nbuf)]   # compute done (inputs free, outputs ready)
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]   # outputs copied out (outputs free)
    t5 = w.t5 or (0, 0, True)

    def one(i):
        b = i % nbuf
        (in_flat, din), (out_flat, dout_) = dev_in[b], dev_out[b]
        with torch.cuda.stream(s_in):
            if i >= nbuf:
                s_in.wait_event(ev_cmp[b])
            in_flat.copy_(host_in_flat, non_blocking=True)
            ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        if i >= nbuf:
            s_cmp.wait_event(ev_out[b])
        kw = dict(alibi_slopes=din.get("slopes"), causal=w.causal, softmax_scale=w.scale,
                  num_buckets=t5[0], max_distance=t5[1], bidirectional=t5[2],
                  bias_table=din.get("table"))
        out, l_ = fa.fat_attn_fwd(din["q"], din["k"], din["v"], din["cu_seqlens"], w.max_seqlen,
                                  out=dout_["out"], lse=lse[b], stream=s_cmp, **kw)
        fa.fat_attn_bwd(din["q"], din["k"], din["v"], din["cu_seqlens"], w.max_seqlen, out, l_,
                        din["dout"], workspace=ws[b], dq=dout_["dq"], dk=dout_["dk"],
                        dv=dout_["dv"], dbias_table=dout_.get("dtab"), stream=s_cmp, **kw)
        ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[b])
            host_out[b].copy_(out_flat, non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(2 * nbuf):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        one(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return ms, h2d, d2h


def traffic_for(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
        ent = table[kernel_key]
        src = os.path.join(ROOT, "attention_relative_position_gb300", "csrc", ent["source"])
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return float(ent["dram_bytes_per_launch"]) if sha == ent["source_sha"] else None
    except Exception:
        return None


def cpu_baseline(w, seconds=10.0):
    """The fp64 oracle, as it stands, on the host cores over a bounded sample of the workload:
    whole (document, head) pairs, forward + backward, until `seconds` have elapsed."""
    import numpy as np
    import oracle
    from attention_relative_position_gb300 import workloads as wl
    x = wl.make_inputs(w, device="cpu")
    t5 = w.t5 or (0, 0, True)
    pb = oracle.Problem(wl.bf16_bits(x["q"]), wl.bf16_bits(x["k"]), wl.bf16_bits(x["v"]),
                        x["cu_seqlens"].numpy(),
                        table=x["table"].numpy() if x["table"] is not None else None,
                        num_buckets=t5[0], max_distance=t5[1], bidirectional=t5[2],
                        slopes=x["slopes"].numpy() if x["slopes"] is not None else None,
                        causal=w.causal, scale=w.scale, d_from_bf16_out=True)
    dout = wl.bf16_bits(x["dout"])
    lens = np.diff(x["cu_seqlens"].numpy())
    pairs = [(i, h) for i in range(len(lens)) for h in range(w.num_heads) if lens[i] > 0]
    flops, done, t0 = 0.0, 0, time.perf_counter()
    for doc, h in pairs:
        L = int(lens[doc])
        rows = list(range(L))
        oracle.attn_fwd_rows(pb, doc, h, rows)
        oracle.attn_bwd_rows(pb, dout, doc, h, rows, rows, want_dtable=w.t5 is not None)
        f = 4.0 * L * L * w.head_dim * 3.5
        flops += f / 2 if w.causal else f
        done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{done} of {len(pairs)} (document, head) pairs of {w.name}, forward + "
                      f"backward of every row, {dt:.1f} s",
            "seconds": dt}


def _guarded(fn, *args):
    """fn(*args), or an error record: a side figure must not cost the benchmark line."""
    try:
        return fn(*args)
    except Exception as e:
        return {"error": f"{type(e).__name__}: {e}"[:200]}


def hbm_bytes(w):
    """Algorithmic HBM bytes of one launch of each kernel: the forward reads Q, K, V (and the
    table) and writes O and lse; the backward preprocess reads O and dO, writes D and zeroes the
    fp32 dQ accumulator (and the table gradient); the finish reads that accumulator and writes
    dq in bf16."""
    T, H, d = w.total_tokens, w.num_heads, w.head_dim
    x = T * H * d
    tab = w.t5[0] * H * 4 if w.t5 else 0
    return {"fwd": 3 * x * 2 + tab + x * 2 + T * H * 4,
            "bwd_pre": 2 * x * 2 + T * H * 4 + x * 4 + tab,
            "bwd_fin": x * 4 + x * 2}


def hbm_figures(w, per, peak_gbs):
    """GB/s of the memory-bound kernels (algorithmic bytes / median CUDA-event time) and their
    fraction of the measured copy bandwidth; the forward's figure matters for short sequences,
    where it is latency-bound rather than tensor-bound."""
    b = hbm_bytes(w)
    res = {}
    for k in ("fwd", "bwd_pre", "bwd_fin"):
        ms = statistics.median(per[k])
        gbs = b[k] / ms / 1e6
        res[k + "_us"] = round(ms * 1e3, 2)
        res[k + "_gbs"] = round(gbs, 1)
        res[k + "_gbs_frac"] = round(gbs / peak_gbs, 4)
    res["peak_gbs"] = peak_gbs
    return res


def graph_step(r, f):
    """The step (forward + fused backward) captured in a CUDA graph after warm-up on the capture
    stream (kernel attributes and tensor maps are prepared then), replayed and timed with CUDA
    events: the device time without the host's per-launch cost."""
    import torch
    s = torch.cuda.Stream()
    old = r.stream
    r.stream = s
    try:
        with torch.cuda.stream(s):
            for _ in range(3):
                r.step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            r.step()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            ms = _time_ms(torch, g.replay, reps=50, warm=5)
    finally:
        r.stream = old
    bits = r.fa.fat_attn_get_device_error()
    if bits:
        raise RuntimeError(f"device error word {bits}")
    return {"step_us": round(ms * 1e3, 2), "fwd_bwd_tflops": round(3.5 * f / ms / 1e9, 3),
            "how": "forward + fused backward captured once in a CUDA graph, replayed"}


def quick_other(w, device, peaks, steps=10):
    r = Runner(w, device)
    for _ in range(3):
        r.step()
    per = time_steps(r, steps)
    f = w.fwd_flops()
    fwd_ms = statistics.median(per["fwd"])
    step_ms = statistics.median(per["step"])
    main_ms = statistics.median(per["bwd_main"])
    res = {"fwd_tflops": f / fwd_ms / 1e9, "fwd_bwd_tflops": 3.5 * f / step_ms / 1e9,
           "bwd_main_tflops": 2.5 * f / main_ms / 1e9}
    res.update({k + "_frac": v / peaks["bf16_tflops"] for k, v in list(res.items())})
    res = {k: round(v, 4) for k, v in res.items()}
    res["ms_per_step"] = round(step_ms, 4)
    res["hbm"] = _guarded(hbm_figures, w, per, peaks["hbm_gbs"])
    if w.total_tokens <= 8192:  # launch-bound: the same step captured once and replayed
        res["cuda_graph"] = _guarded(graph_step, r, f)
    if w.total_tokens <= 1024:  # latency-bound: beside the launch floor of this stream
        import torch
        one = torch.zeros(1, device=device)
        floor = _time_ms(torch, lambda: one.zero_(), reps=50, warm=5)
        res["latency"] = {"fwd_us": round(statistics.median(per["fwd"]) * 1e3, 2),
                          "step_us": round(step_ms * 1e3, 2),
                          "launches_per_step": r.launches_per_step,
                          "launch_floor_us": round(floor * 1e3, 2),
                          "floor": "CUDA-event time of one one-element kernel on the same stream"}
    del r
    return res


def _time_ms(torch, fn, reps=10, warm=3):
    """Median CUDA-event time (ms) of fn() on the current stream, after warm-up calls."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times)


def _time_graph_ms(torch, fn, inner=10, reps=20):
    """Median device time (ms) of one fn() when `inner` calls are captured in one CUDA graph and
    replayed: the GPU time without the host's per-launch cost (warm-up on the capture stream
    first, so kernel attributes and tensor maps are prepared outside the capture)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(inner):
            fn()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        ms = _time_ms(torch, g.replay, reps=reps, warm=3)
    return ms / inner


def aux_kernels(device, peaks):
    """The report's other fused kernels (RMSNorm forward/backward, cross-entropy with z-loss and
    its gradient in one pass): HBM GB/s of algorithmic bytes over the median CUDA-event time,
    inputs larger than L2, and the oracle's rate on a bounded sample."""
    import numpy as np
    import torch
    import attention_relative_position_gb300 as fa
    from attention_relative_position_gb300 import workloads as wl
    res = {}
    rows, dim = 131072, 1024  # 256 MiB of bf16 activations
    g = torch.Generator(device=device).manual_seed(4242)
    x = torch.randn(rows, dim, device=device, generator=g).to(torch.bfloat16)
    dy = torch.randn(rows, dim, device=device, generator=g).to(torch.bfloat16)
    w = 1.0 + 0.1 * torch.randn(dim, device=device, generator=g)
    y, rstd = fa.fat_rmsnorm_fwd(x, w)
    dx, dw = torch.empty_like(x), torch.empty_like(w)
    t_f = _time_ms(torch, lambda: fa.fat_rmsnorm_fwd(x, w, y=y, rstd=rstd))
    t_b = _time_ms(torch, lambda: fa.fat_rmsnorm_bwd(x, w, rstd, dy, dx=dx, dweight=dw))
    b_f = rows * dim * 2 * 2 + rows * 4 + dim * 4             # x in, y out, rstd, w
    b_b = rows * dim * 2 * 3 + rows * 4 + dim * 4 * 2         # x, dy in, dx out, rstd, w, dw
    xs, ws, dys = wl.make_norm_inputs(2048, dim, seed=7)
    from oracle import norm_ce as nc
    t0 = time.perf_counter()
    nc.rmsnorm_fwd(wl.bf16_bits(xs), ws.numpy(), 1e-6)
    nc.rmsnorm_bwd(wl.bf16_bits(xs), ws.numpy(), wl.bf16_bits(dys), 1e-6)
    t_o = time.perf_counter() - t0
    res["rmsnorm"] = {"rows": rows, "dim": dim,
                      "fwd_us": round(t_f * 1e3, 2), "fwd_gbs": round(b_f / t_f / 1e6, 1),
                      "fwd_frac": round(b_f / t_f / 1e6 / peaks["hbm_gbs"], 4),
                      "bwd_us": round(t_b * 1e3, 2), "bwd_gbs": round(b_b / t_b / 1e6, 1),
                      "bwd_frac": round(b_b / t_b / 1e6 / peaks["hbm_gbs"], 4),
                      "oracle_fwd_bwd_gbs": round(2048 * dim * 2 * 5 / t_o / 1e9, 3),
                      "oracle_sample": f"2048 x {dim} rows, forward + backward, {t_o:.2f} s"}
    del x, dy, y, dx
    rows, vocab = 8192, 32768  # 512 MiB of bf16 logits
    z = (2.0 * torch.randn(rows, vocab, device=device, generator=g)).to(torch.bfloat16)
    t = torch.randint(0, vocab, (rows,), device=device, generator=g, dtype=torch.int32)
    loss, lse, dz = fa.fat_cross_entropy(z, t, z_loss=1e-4, grad_scale=1.0 / rows)
    t_c = _time_ms(torch, lambda: fa.fat_cross_entropy(z, t, z_loss=1e-4, grad_scale=1.0 / rows,
                                                       loss=loss, lse=lse, dlogits=dz))
    b_c = rows * vocab * 2 * 2 + rows * (4 + 4 + 4)
    zs, ts = wl.make_ce_inputs(64, vocab, seed=8)
    t0 = time.perf_counter()
    nc.cross_entropy_fwd(wl.bf16_bits(zs), ts.numpy(), 1e-4)
    nc.cross_entropy_bwd(wl.bf16_bits(zs), ts.numpy(), 1e-4, 1.0 / 64)
    t_o = time.perf_counter() - t0
    res["cross_entropy"] = {"rows": rows, "vocab": vocab, "z_loss": 1e-4,
                            "us": round(t_c * 1e3, 2), "gbs": round(b_c / t_c / 1e6, 1),
                            "frac": round(b_c / t_c / 1e6 / peaks["hbm_gbs"], 4),
                            "oracle_gbs": round(64 * vocab * 2 * 2 / t_o / 1e9, 3),
                            "oracle_sample": f"64 x {vocab} rows, loss + gradient, {t_o:.2f} s"}
    res["peak_gbs"] = peaks["hbm_gbs"]
    return res


def next_rows(device, peaks):
    """Measurements of the generalised rows: T5 decoder cross-attention forward + backward
    (TFLOP/s), a decode step over long key caches with and without key splits (HBM GB/s of the
    cache read), and the RoPE rotation (HBM GB/s)."""
    import torch
    import attention_relative_position_gb300 as fa
    from attention_relative_position_gb300 import workloads as wl
    res = {}
    # cross-attention: 8 documents, 512 decoder queries over 1024 encoder keys, 12 heads, d 64
    xw = wl.XWorkload("xattn_b8_q512_k1024_h12_d64", (512,) * 8, (1024,) * 8, 12, 12, 64,
                      qkv_std=0.5, seed=2001)
    x = wl.make_xinputs(xw, device=device)
    mq, mk = xw.max_seqlen_q, xw.max_seqlen_k

    def xstep():
        o, l = fa.fat_xattn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"],
                                mq, mk)
        fa.fat_xattn_bwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], mq, mk,
                         o, l, x["dout"])

    t_fwd = _time_ms(torch, lambda: fa.fat_xattn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                                                     x["cu_seqlens_k"], mq, mk))
    t_step = _time_ms(torch, xstep)
    f = xw.fwd_flops()
    res["cross_attention"] = {"workload": xw.name, "fwd_tflops": round(f / t_fwd / 1e9, 2),
                              "fwd_bwd_tflops": round(3.5 * f / t_step / 1e9, 2),
                              "fwd_frac": round(f / t_fwd / 1e9 / peaks["bf16_tflops"], 4)}
    del x
    # decode: one query per document over its cache, causal, unidirectional T5 bias
    for name, n, lk, hq, hkv, d in (("decode_b8_k8192_h8_d128", 8, 8192, 8, 8, 128),
                                    ("decode_b32_k4096_gqa16x4_d128", 32, 4096, 16, 4, 128)):
        dw = wl.XWorkload(name, (1,) * n, (lk,) * n, hq, hkv, d, 1.0, (32, 128, False),
                          causal=True, scale=d ** -0.5, seed=2002)
        x = wl.make_xinputs(dw, device=device)
        kw = dict(bias_table=x["table"], num_buckets=32, max_distance=128, bidirectional=False,
                  causal=True, softmax_scale=dw.scale)
        ns = fa.fat_xattn_splitkv_num_splits(x["q"], x["k"], x["cu_seqlens_q"], 1, lk)
        ws = torch.empty(1 << 26, dtype=torch.uint8, device=device)
        t1 = _time_ms(torch, lambda: fa.fat_xattn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                                                      x["cu_seqlens_k"], 1, lk, **kw))
        split = lambda: fa.fat_xattn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], 1, lk, num_splits=ns, workspace=ws,
                                         **kw)
        tn = _time_ms(torch, split)
        tg = _time_graph_ms(torch, split)
        cache = 2 * n * lk * hkv * d * 2  # K and V, bf16
        res[name] = {"splits": ns, "unsplit_us": round(t1 * 1e3, 2),
                     "split_us": round(tn * 1e3, 2),
                     "split_gbs": round(cache / tn / 1e6, 1),
                     "split_graph_us": round(tg * 1e3, 2),
                     "split_graph_gbs": round(cache / tg / 1e6, 1),
                     "split_graph_frac": round(cache / tg / 1e6 / peaks["hbm_gbs"], 4),
                     "bytes": "the K and V cache read once",
                     "graph": "split forward + merge captured 10 times in one CUDA graph"}
        del x, ws
    # RoPE on 8 documents of the 16K T5 shape (q: 131072 x 12 x 64 bf16, 201 MB, beyond L2),
    # positions local to each document
    g = torch.Generator(device=device).manual_seed(2003)
    q = torch.randn(8 * 16384, 12, 64, device=device, generator=g).to(torch.bfloat16)
    cu = torch.arange(0, 8 * 16384 + 1, 16384, dtype=torch.int32, device=device)
    out = torch.empty_like(q)
    rope = lambda: fa.fat_rope_apply(q, cu, 16384, out=out)
    t_r = _time_ms(torch, rope)
    t_g = _time_graph_ms(torch, rope)
    b = 2 * q.numel() * 2
    res["rope"] = {"shape": "8 x 16384 x 12 x 64", "us": round(t_r * 1e3, 2),
                   "gbs": round(b / t_r / 1e6, 1), "frac": round(b / t_r / 1e6 / peaks["hbm_gbs"], 4),
                   "graph_us": round(t_g * 1e3, 2), "graph_gbs": round(b / t_g / 1e6, 1),
                   "bytes": "q read and written once"}
    del q, out
    res["peaks"] = {"bf16_tflops": peaks["bf16_tflops"], "hbm_gbs": peaks["hbm_gbs"]}
    return res


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from attention_relative_position_gb300 import _build
    if rank == 0:
        _build.build()
    if args.aux_kernels:
        device = f"cuda:{local_rank}"
        torch.cuda.set_device(device)
        if rank == 0:
            print(json.dumps({"aux_kernels": aux_kernels(device, load_peaks()[0])}), flush=True)
        return
    if args.next_rows:
        device = f"cuda:{local_rank}"
        torch.cuda.set_device(device)
        if rank == 0:
            print(json.dumps({"next_rows": next_rows(device, load_peaks()[0])}), flush=True)
        return
    if world > 1:
        dist.barrier()
    device = f"cuda:{local_rank}"
    torch.cuda.set_device(device)
    w = pick_workload(args.workload)
    steps = args.steps if args.steps is not None else (300 if w.fwd_flops() < 1e11 else 30)
    warmup = max(args.warmup, 1)
    peaks, peak_src = load_peaks()
    r = Runner(w, device)
    for _ in range(warmup):
        r.step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if not args.quick else None
    if sampler:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    per = time_steps(r, steps, flush=not args.quick)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t0
    clocks = sampler.stop() if sampler else None
    bits = r.fa.fat_attn_get_device_error()
    if bits:
        raise RuntimeError(f"device error word {bits}")
    med = {k: statistics.median(v) for k, v in per.items()}
    step_ms = max_over_ranks(med["step"], device)
    f = w.fwd_flops()
    value = job_tflops(3.5 * f, world, step_ms)  # TFLOP/s
    # the backward runs as the persistent kernel for d = 64 and documents of <= 64 key tiles,
    # else as one CTA per key tile
    persistent = w.head_dim == 64 and (w.max_seqlen + 127) // 128 <= 64
    bwd_name = "fat_bwd_kernel" if persistent else "fat_bwd_tiles_kernel"
    # the forward runs as persistent one-tile CTAs for d = 64, documents of <= 2048 rows and at
    # least three 128-row blocks per resident CTA (two per SM), else as a grid
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    blocks = (w.total_tokens // 128 + len(w.seqlens)) * w.num_heads
    fwd_pers = w.head_dim == 64 and w.max_seqlen <= 2048 and blocks >= 3 * 2 * sms
    fwd_name = "fat_fwd_pers_kernel" if fwd_pers else "fat_fwd_kernel"
    kernels = {"fwd": (fwd_name, f, med["fwd"], "fat_attn_fwd.cu"),
               "bwd_main": (bwd_name, 2.5 * f, med["bwd_main"], "fat_attn_bwd.cu")}
    dom = max(kernels, key=lambda k: kernels[k][2])
    kname, kflops, kms, ksrc = kernels[dom]
    achieved = kflops / kms / 1e9
    peak = peaks["bf16_tflops"]
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1)-type inputs of the workload's shapes; no dataset)",
        "config": workload_config(w, world, "flushed between timed steps (256 MiB write, "
                                            "outside the timed kernels)"),
        "fwd_tflops": round(f / med["fwd"] / 1e9, 3),
        "bwd_tflops": round(2.5 * f / (med["bwd_pre"] + med["bwd_main"] + med["bwd_fin"])
                            / 1e9, 3),
        "per_kernel_ms": {k: round(v, 5) for k, v in med.items()},
        "timing": "median of the per-step CUDA-event times",
        "roofline": {"kernel": f"{kname}<{w.head_dim}>", "bound": "tensor",
                     "achieved": round(achieved, 3), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_src} bf16 dense (burst; kernel timed alone)",
                     "traffic": traffic_for(f"{kname}<{w.head_dim}>@{w.name}"),
                     "algorithmic_flops_per_launch": kflops},
        "hbm": _guarded(hbm_figures, w, per, peaks["hbm_gbs"]),
        "gpu_launches": steps * r.launches_per_step,
        "timed_wall_s": round(wall, 4),
    }
    if clocks is not None:
        line["clocks"] = clocks
    if not args.quick:
        e_steps = max(3, min(steps, 20))
        ems, h2d, d2h = e2e_steps(w, r, e_steps)
        ems = max_over_ranks(ems, device)
        line["e2e"] = {"value": round(job_tflops(3.5 * f, world, ems), 3), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(ems, 4),
                       "pipelining": "2 buffer sets: step i+1 copied in and step i-1 copied "
                                     "out while step i computes; one packed copy per "
                                     "direction per step"}
        if rank == 0 and world == 1:
            from attention_relative_position_gb300 import workloads as wl
            others = {}
            for idx in range(len(wl.WORKLOADS)):
                ow = wl.WORKLOADS[idx]
                if ow.name != w.name:
                    try:  # one side measurement must not cost the line
                        others[ow.name] = quick_other(ow, device, peaks)
                    except Exception as e:
                        others[ow.name] = {"error": f"{type(e).__name__}: {e}"[:200]}
                        continue
                    try:  # the oracle beside it, on a ~3 s sample
                        cb = cpu_baseline(ow, seconds=3.0)
                        cb["full_workload_s_extrapolated"] = round(
                            3.5 * ow.fwd_flops() / (cb["value"] * 1e12), 1)
                        others[ow.name]["cpu_baseline"] = cb
                    except Exception as e:
                        others[ow.name]["cpu_baseline"] = {
                            "error": f"{type(e).__name__}: {e}"[:200]}
            line["other_workloads"] = others
            line["aux_kernels"] = _guarded(aux_kernels, device, peaks)
            line["next_rows"] = _guarded(next_rows, device, peaks)
            line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from attention_relative_position_gb300 import workloads as wl
    oracle.build()
    w = pick_workload(args.workload)
    steps = args.steps if args.steps is not None else 3
    warmup = args.warmup
    x = wl.make_inputs(w, device="cpu")
    t5 = w.t5 or (0, 0, True)
    pb = oracle.Problem(wl.bf16_bits(x["q"]), wl.bf16_bits(x["k"]), wl.bf16_bits(x["v"]),
                        x["cu_seqlens"].numpy(),
                        table=x["table"].numpy() if x["table"] is not None else None,
                        num_buckets=t5[0], max_distance=t5[1], bidirectional=t5[2],
                        slopes=x["slopes"].numpy() if x["slopes"] is not None else None,
                        causal=w.causal, scale=w.scale, d_from_bf16_out=True)
    dout = wl.bf16_bits(x["dout"])
    lens = np.diff(x["cu_seqlens"].numpy())
    pairs = [(i, h) for i in range(len(lens)) for h in range(w.num_heads) if lens[i] > 0]

    def one(k):  # one bounded sample: the k-th (document, head) pair, forward + backward
        doc, h = pairs[k % len(pairs)]
        L = int(lens[doc])
        rows = list(range(L))
        oracle.attn_fwd_rows(pb, doc, h, rows)
        oracle.attn_bwd_rows(pb, dout, doc, h, rows, rows, want_dtable=w.t5 is not None)
        f = 3.5 * 4.0 * L * L * w.head_dim
        return f / 2 if w.causal else f

    # warm-up: the oracle has no cache or compiled code to warm, so each warm-up step is one
    # forward row (it only touches the library and the input pages)
    for k in range(warmup):
        doc, h = pairs[k % len(pairs)]
        oracle.attn_fwd_rows(pb, doc, h, [0])
    t0 = time.perf_counter()
    flops = sum(one(k) for k in range(steps))
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": round(dt / steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, world, "host run (no GPU)"),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "kind": "oracle",
                         "cores": oracle.num_threads(),
                         "sample": f"each step: one (document, head) pair of {w.name}, "
                                   f"forward + backward of every row, fp64"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
