#!/usr/bin/env python3
"""Benchmark of one MLA decode step (cache append + absorbed decode) on GB300.

A step is one pass of the whole path over one batch: mla_cache_append (new row per sequence)
then mla_decode_attn (absorb, split attention over every cached row, combine + W_UV
up-projection). The default workload is the largest single-GPU one: ragged paged decode
(B=64 sequences of U{128..32768} rows, H=128, kv_lora 512, rope 64, bf16, 64-row pages with a
shuffled page table). The same line carries, under "also", the attention kernel's roofline
fraction on the single-sequence (B=1, H=16, 4096 rows) and batched (B=32, H=128, 4096 rows)
workloads, measured in the same run, and under "layer_projections" the layer's front end
(mla_front_end: Q chain or q projection + kv_a) and o_proj (mla_o_proj) per call on V2-Lite- and
V3-shaped layers. Prints ONE JSON line (--proj-only: one line per projection record).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Timing: inputs resident in HBM; each step uses the next of R rotating input copies whose total
exceeds 2x L2, so no step reads another's data from L2; the timed K steps are replayed as CUDA
graphs with CUDA events on the launching stream; the attention kernel of the first step of
every graph is bracketed by events inside the graph (an event between two kernels makes their
overlapped launch a plain one, so the other steps run without). N > 1 (torchrun) runs independent replicas per GPU (the
sequences are independent: no data-path collective) and reports the max over ranks.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MLA decode: KV-cache rows/s, achieved TFLOP/s & HBM GB/s vs roofline"
DEFAULT_WORKLOAD = "ragged_paged_b64"
# attention-only sub-records measured in the same run: workload -> timed steps
ALSO_WORKLOADS = {"v2lite_b1_t4096": 4000, "v3_b32_t4096": 400}
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ------------------------------------------------------------------------------------------------
# algorithmic work of one step
# ------------------------------------------------------------------------------------------------

def step_work(prob):
    """Algorithmic FLOPs and bytes of one step, and of the attention stage alone.

    FLOPs: absorb 2HNC per sequence, attention (QK over the C+R row and PV over the C latent)
    rows*H*(2(C+R)+2C), up-projection 2HCV per sequence, plus the kv_a GEMV when the append
    projects. Bytes: every attended cache row once (shared by all heads), kv_b once, q, out,
    lse, page table, append input and output (and W_kva, x when projecting)."""
    wl = prob.wl
    B, H, C, N, R, V = wl.B, wl.H, wl.C, wl.N, wl.R, wl.V
    e = 2 if wl.act == "bf16" else 4
    rows = int(np.sum(prob.seq_lens))
    if wl.kv_b == "q8_0":
        kvb = H * (N + V) * (C // 32) * 34
    elif wl.kv_b == "q4_affine":
        kvb = H * (N + V) * (C // 2 + (C // 64) * 4)
    else:
        kvb = H * (N + V) * C * (2 if wl.kv_b == "bf16" else 4)
    attn_flops = rows * H * (2 * (C + R) + 2 * C)
    attn_bytes = rows * (C + R) * e
    flops = B * 2 * H * N * C + attn_flops + B * 2 * H * C * V
    pages = 0 if prob.page_table is None else int(np.sum((prob.seq_lens + wl.page_size - 1) // wl.page_size))
    byts = attn_bytes + kvb + B * H * (N + R) * e + B * H * (V + 1) * 4 + 4 * (pages + 2 * B)
    if wl.append == "gemv":
        flops += B * 2 * (C + R) * wl.hidden
        byts += (C + R) * wl.hidden * e + B * wl.hidden * e
    else:
        byts += B * (C + R) * 4
    decode_flops, decode_bytes = flops, byts   # mla_decode_attn alone (kernel 3 runs it in one launch)
    if wl.append == "gemv":
        flops += B * 2 * (C + R) * wl.hidden
        byts += (C + R) * wl.hidden * e + B * wl.hidden * e
    else:
        byts += B * (C + R) * 4
    byts += B * (C + R) * e  # the appended rows
    return dict(rows=rows, flops=flops, bytes=byts, attn_flops=attn_flops, attn_bytes=attn_bytes,
                decode_flops=decode_flops, decode_bytes=decode_bytes)


def input_bytes(prob):
    n = prob.pool.nbytes + prob.kv_b.nbytes + prob.q.nbytes
    for a in (prob.kva_rows, prob.x, prob.w_kva, prob.page_table):
        if a is not None:
            n += a.nbytes
    return n


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------

_SMI_FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, uuid: str):
        self.uuid = uuid
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={_SMI_FIELDS}", "--format=csv,noheader",
                                       "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()

    def samples(self, t0: float, t1: float):
        out = []
        try:
            lines = open(self.f.name).read().strip().splitlines()
        except OSError:
            return out
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm = float(parts[2].split()[0])
                smax = float(parts[3].split()[0])
            except ValueError:
                continue
            if t0 <= ts <= t1:
                out.append(dict(uuid=parts[1], sm=sm, smax=smax, hw=parts[6], hwt=parts[7], swt=parts[8],
                                pcap=parts[9]))
        mine = [s for s in out if s["uuid"] == self.uuid]
        if mine or len({s["uuid"] for s in out}) > 1:
            return mine
        return out  # only one GPU visible to nvidia-smi: it is ours


def summarize_clocks(samples, window):
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
    reasons = set()
    for s in samples:
        for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                        ("pcap", "sw_power_cap")):
            if s[k].lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(s["sm"] for s in samples), "sm_max_mhz": max(s["smax"] for s in samples),
            "reasons": sorted(reasons), "samples": len(samples), "window": window}


# ------------------------------------------------------------------------------------------------
# events that can live inside a CUDA graph
# ------------------------------------------------------------------------------------------------

class _CudartEvent:
    """A timing event recorded with cudaEventRecordExternal, so that it becomes an event-record
    node when recorded during stream capture (for torch builds without external events)."""
    _rt = None

    @classmethod
    def _lib(cls):
        if cls._rt is None:
            import ctypes
            cls._rt = ctypes.CDLL("libcudart.so.13")   # the runtime torch has already loaded
        return cls._rt

    def __init__(self):
        import ctypes
        self._c = ctypes
        self.ev = ctypes.c_void_p()
        if self._lib().cudaEventCreateWithFlags(ctypes.byref(self.ev), 0) != 0:
            raise RuntimeError("cudaEventCreateWithFlags failed")

    def record(self, stream):
        if self._lib().cudaEventRecordWithFlags(self.ev, self._c.c_void_p(stream.cuda_stream), 1) != 0:
            raise RuntimeError("cudaEventRecordWithFlags failed")

    def synchronize(self):
        self._lib().cudaEventSynchronize(self.ev)

    def elapsed_time(self, other):
        ms = self._c.c_float()
        if self._lib().cudaEventElapsedTime(self._c.byref(ms), self.ev, other.ev) != 0:
            raise RuntimeError("cudaEventElapsedTime failed")
        return ms.value


def graph_event(torch):
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:  # torch without external events: record through the runtime directly
        return _CudartEvent()


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# attention kernel of a plan (mla_plan_info.kernel) -> its source file and kernel name
KERNEL_FILE = {0: "attn_simt", 1: "attn_tc", 2: "attn_pair", 3: "decode_small"}


def kernel_source_sha(kernel: int) -> str:
    f = os.path.join(ROOT, "mla_latent_cache_absorb_gb300", "csrc", KERNEL_FILE[kernel] + ".cu")
    return hashlib.sha256(open(f, "rb").read()).hexdigest()[:16]


def ncu_traffic(kernel: int, workload: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary, if it
    was taken on the current kernel source."""
    try:
        d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    except (OSError, ValueError):
        return None
    ent = d.get(f"{KERNEL_FILE[kernel]}:{workload}")
    if not ent or ent.get("source_sha") != kernel_source_sha(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


def aggregate_over_ranks(total_ms, world, rows_per_step, steps, device):
    """Whole-job throughput: every rank processed rows_per_step * steps rows; the job took
    as long as the slowest rank. Returns (max time in ms, rows per second)."""
    tmax = float(total_ms)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([tmax], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        tmax = float(t.item())
    return tmax, world * rows_per_step * steps / (tmax / 1e3)


def workload_config(wl, prob, work):
    """The workload's own description (the same dict in both arms)."""
    return {
        "workload": wl.name, "B": wl.B, "H": wl.H, "kv_lora": wl.C, "qk_nope": wl.N, "qk_rope": wl.R,
        "v_head": wl.V, "rows_per_step": work["rows"], "kv_b": wl.kv_b, "act": wl.act,
        "paged": bool(wl.page_size), "append": wl.append, "parallelism": "replicas (independent sequences)",
    }


def run_ours(args, rank, world, device, workload, K, W, with_e2e=True, with_clocks=True):
    import torch

    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300 import synth
    from mla_latent_cache_absorb_gb300.runner import DeviceStep

    wl = synth.WORKLOADS[workload]
    prob = synth.make_problem(wl)
    work = step_work(prob)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 2 ** 20)
    per_copy = input_bytes(prob)
    R = max(1, min(64, math.ceil(2.2 * l2 / per_copy)))
    stream = torch.cuda.Stream(device=device)
    steps = [DeviceStep(prob, device=device, stream=stream)]
    for _ in range(R - 1):
        steps.append(DeviceStep(prob, device=device, stream=stream))
    st, plan = L.mla_decode_plan(steps[0].cfg, wl.B)
    L.check(st, "mla_decode_plan")
    launches_per_step = (2 if wl.append == "gemv" else 1) + (1 if plan.kernel == 3 else 3)

    def one_step(ds, s, ev=None):
        # the user's calls: mla_cache_append, then mla_decode_attn; a step whose attention is
        # bracketed by events enqueues the same kernels through the three step calls instead
        L.check(ds.append(s), "mla_cache_append")
        if ev is None:
            L.check(ds.decode(s), "mla_decode_attn")
            return
        if plan.kernel == 3:   # one launch: the whole decode is the bracketed kernel
            ev[0].record(s)
            L.check(ds.decode(s), "mla_decode_attn")
            ev[1].record(s)
            return
        L.check(ds.absorb(s), "mla_decode_absorb")
        ev[0].record(s)
        L.check(ds.partial(s), "mla_decode_partial")
        ev[1].record(s)
        L.check(ds.combine(s), "mla_decode_combine")

    # graphs of G steps (whole passes over the R copies, at least 16 steps), two of them to
    # double-buffer the in-graph attention events, plus a tail graph for K mod G steps. Only
    # the first step of each graph has its attention launch bracketed by events: an event
    # between two kernels turns their programmatic (overlapped) launch into a plain one.
    G = R * max(1, math.ceil(16 / R)) if R > 1 else max(1, min(64, K))
    G = max(1, min(G, max(R, 64)))
    torch.cuda.synchronize(device)

    def capture(n, with_events):
        g = torch.cuda.CUDAGraph()
        evs = [(graph_event(torch), graph_event(torch))] if with_events else None
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            s = torch.cuda.current_stream(device)
            for i in range(n):
                one_step(steps[i % R], s, evs[0] if (evs and i == 0) else None)
        return g, evs

    with torch.cuda.stream(stream):
        # eager warm-up (W steps) also checks every call once outside capture
        for i in range(W):
            one_step(steps[i % R], stream)
        torch.cuda.synchronize(device)
        for ds in steps:
            for ws in (ds.ws_append, ds.ws_decode):
                e, seq = L.mla_get_device_error(ws, stream)
                L.check(e, f"device error (seq {seq})")
        gA, evA = capture(G, True)
        gB, evB = capture(G, True)
        tail = K % G
        gT, evT = capture(tail, True) if tail else (None, None)
        n_full = K // G
        # one untimed replay of every graph: uploads them and warms their first launch, so the
        # timed region holds steady-state replays only
        for g in (gA, gB, gT):
            if g is not None:
                g.replay()
        torch.cuda.synchronize(device)

        sampler = None
        if with_clocks:
            sampler = ClockSampler(str(props.uuid) if hasattr(props, "uuid") else "")
            if not str(sampler.uuid).startswith("GPU-") and sampler.uuid:
                sampler.uuid = "GPU-" + sampler.uuid
            sampler.start()
            time.sleep(0.3)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        wall0 = time.time()
        t_start.record(stream)
        attn_ms = []
        pending = []
        graphs = [(gA, evA), (gB, evB)]
        for r in range(n_full):
            g, ev = graphs[r % 2]
            if len(pending) == 2:  # reuse of this graph's events: read the previous replay first
                ev_old = pending.pop(0)
                ev_old[-1][1].synchronize()
                attn_ms.extend(a.elapsed_time(b) for a, b in ev_old)
            g.replay()
            pending.append(ev)
        if gT is not None:
            gT.replay()
            pending.append(evT)
        t_end.record(stream)
        for ev in pending:
            ev[-1][1].synchronize()
            attn_ms.extend(a.elapsed_time(b) for a, b in ev)
        t_end.synchronize()
        wall1 = time.time()
        if world > 1:
            torch.distributed.barrier()
        total_ms = t_start.elapsed_time(t_end)
        clocks = None
        if sampler is not None:
            clk = sampler.samples(wall0, wall1)
            window = "timed"
            if len(clk) < 3 and args.clock_window_s > 0:
                # the timed region was shorter than the sampler's period: sample the same graphs
                # for about a second right after it (untimed) and say so
                wa = time.time()
                while time.time() - wa < args.clock_window_s:
                    gA.replay()
                    gB.replay()
                    torch.cuda.synchronize(device)
                clk = sampler.samples(wa, time.time())
                window = "adjacent"
            sampler.stop()
            clocks = summarize_clocks(clk, window)

        # end to end through the public calls: pinned host inputs in, results out, every step
        e2e = None
        if with_e2e:
            e2e = run_e2e(torch, L, steps, prob, stream, device, K, W, work)

    tmax, value = aggregate_over_ranks(total_ms, world, work["rows"], K, device)
    ms_per_step = tmax / K
    attn_avg_ms = sum(attn_ms) / len(attn_ms)
    hbm, tf_burst, tf_sust, src = peaks()
    # the bracketed kernel's algorithmic work: the attention (kernels 0-2), or the whole decode
    # (kernel 3: absorb, attention, merge and W_UV in one launch)
    k_bytes = work["decode_bytes"] if plan.kernel == 3 else work["attn_bytes"]
    k_flops = work["decode_flops"] if plan.kernel == 3 else work["attn_flops"]
    attn_gbs = k_bytes / (attn_avg_ms / 1e3) / 1e9
    step_s = ms_per_step / 1e3
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.act, "data": "synthetic (seeded generator; random-init kv_b)",
        "config": workload_config(wl, prob, work),
        "run": {
            "l2": f"rotating {R} input copies ({R * per_copy / 2 ** 20:.0f} MB, L2 {l2 / 2 ** 20:.0f} MB)",
            "timing": f"CUDA graphs of {G} steps (each replayed once untimed first), events on the "
                      f"launching stream; the attention launch of each graph's first step bracketed "
                      f"by in-graph events",
            "gpus": f"replicas x{world}" if world > 1 else "single GPU",
            "attention_kernel": {0: "cuda-core", 1: "tcgen05, one CTA per head group",
                                 2: "tcgen05, SM pairs (clusters of two CTAs)",
                                 3: "one launch: absorb and merge with W_UV on the CUDA cores, chunk attention on warp-level bf16 tensor-core steps"}[plan.kernel],
            "heads_per_cta": plan.heads_per_cta, "splits": plan.splits,
            "rows_per_split": plan.rows_per_split,
        },
        "tflops": work["flops"] / step_s / 1e12,
        "hbm_gbs": work["bytes"] / step_s / 1e9,
        "step_roofline_frac": max(work["flops"] / (tf_burst * 1e12), work["bytes"] / (hbm * 1e9)) / step_s,
        "roofline": {
            "kernel": f"{KERNEL_FILE[plan.kernel]} ({'whole decode' if plan.kernel == 3 else 'split attention'})",
            "bound": "hbm", "achieved": attn_gbs, "peak": hbm, "unit": "GB/s", "frac": attn_gbs / hbm,
            "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback",
            "bytes_per_launch": k_bytes, "avg_launch_us": attn_avg_ms * 1e3,
            "traffic": ncu_traffic(plan.kernel, wl.name),
            "tensor_tflops": k_flops / (attn_avg_ms / 1e3) / 1e12 if plan.kernel in (1, 2) else None,
            "kernel_tflops": k_flops / (attn_avg_ms / 1e3) / 1e12,
        },
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "e2e": e2e,
    }
    del steps
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()
    return line


# layer-projection sub-records measured in the same run: (workload, weight format) -> timed steps
PROJ_BENCH = {("v3_proj_b4", "bf16"): 100, ("v3_proj_b64", "bf16"): 60, ("v3_proj_b4", "q4_affine"): 100,
              ("v3_proj_b4", "q8_0"): 100, ("v2lite_proj_b1", "bf16"): 400}


def weight_bytes(a):
    return 0 if a is None else int(a.nbytes)


def proj_work(pp):
    """Algorithmic bytes and FLOPs of mla_front_end and of mla_o_proj: every weight byte once,
    the inputs and outputs once (the Q chain's q_lat rows written, normalised in place and read
    back), 2 FLOPs per weight element and sequence."""
    wl = pp.wl
    B, act = wl.B, (2 if wl.act == "bf16" else 4)
    qk = wl.N + wl.R
    fe_w = weight_bytes(pp.w_q_a) + weight_bytes(pp.w_q) + weight_bytes(pp.w_kva)
    fe_b = fe_w + B * wl.hidden * act + B * wl.H * qk * act + B * (wl.C + wl.R) * 4
    fe_f = 2 * B * ((wl.q_lora * wl.hidden + wl.H * qk * wl.q_lora) if wl.q_lora else wl.H * qk * wl.hidden)
    fe_f += 2 * B * (wl.C + wl.R) * wl.hidden
    if wl.q_lora:
        fe_b += weight_bytes(pp.q_a_norm_w) + 4 * B * wl.q_lora * 4
    o_b = weight_bytes(pp.w_o) + B * wl.H * wl.V * 4 + B * wl.hidden * 4
    o_f = 2 * B * wl.hidden * wl.H * wl.V
    return {"front_end": (fe_b, fe_f), "o_proj": (o_b, o_f)}


def run_proj(device, name, fmt, K, W):
    """Time mla_front_end and mla_o_proj on one projection workload: R device copies of the
    weights (more than 2.2x L2 in all), CUDA graphs of whole passes over the copies, each call
    bracketed by in-graph events on the launching stream."""
    import torch

    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300 import synth
    from mla_latent_cache_absorb_gb300.runner import DeviceProj

    wl = synth.PROJ_WORKLOADS[name].with_(w=fmt)
    pp = synth.make_proj_problem(wl)
    work = proj_work(pp)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 2 ** 20)
    per_copy = work["front_end"][0] + work["o_proj"][0]
    R = max(1, min(32, math.ceil(2.2 * l2 / per_copy)))
    stream = torch.cuda.Stream(device=device)
    copies = [DeviceProj(pp, device=device, stream=stream) for _ in range(R)]
    G = R * max(1, math.ceil(8 / R))
    with torch.cuda.stream(stream):
        for i in range(W):
            L.check(copies[i % R].front_end(), "mla_front_end")
            L.check(copies[i % R].o_proj(), "mla_o_proj")
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        evs = [(graph_event(torch), graph_event(torch), graph_event(torch)) for _ in range(G)]
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            s = torch.cuda.current_stream(device)
            for i in range(G):
                dp = copies[i % R]
                evs[i][0].record(s)
                L.check(dp.front_end(stream=s), "mla_front_end")
                evs[i][1].record(s)
                L.check(dp.o_proj(stream=s), "mla_o_proj")
                evs[i][2].record(s)
        g.replay()
        torch.cuda.synchronize(device)
        fe_ms, o_ms = [], []
        for _ in range(max(1, K // G)):
            g.replay()
            evs[-1][2].synchronize()
            fe_ms.extend(e[0].elapsed_time(e[1]) for e in evs)
            o_ms.extend(e[1].elapsed_time(e[2]) for e in evs)
    hbm = peaks()[0]
    out = {"workload": wl.name, "weights": fmt, "B": wl.B, "hidden": wl.hidden, "q_lora": wl.q_lora,
           "launches_per_step": copies[0].launches(), "steps": len(fe_ms)}
    for key, ms in (("front_end", fe_ms), ("o_proj", o_ms)):
        t = statistics.median(ms) / 1e3
        b, f = work[key]
        out[key] = {"median_us": t * 1e6, "bytes": b, "gbs": b / t / 1e9, "hbm_frac": b / t / 1e9 / hbm,
                    "tflops": f / t / 1e12}
    del copies
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()
    return out


# multi-token decode sub-records: (workload, query tokens) -> timed calls
MULTI_BENCH = {("v2lite_b1_t4096", 4): 2000, ("v3_b32_t4096", 2): 200, ("v3_b32_t4096", 4): 100}


def run_multi_tokens(device, name, tokens, K, W):
    """Time mla_decode_attn_multi (T query tokens per sequence over the cached rows) against T
    one-token mla_decode_attn calls on the same cache: CUDA graphs over R input copies (more than
    2.2x L2 in all), events around each graph."""
    import torch

    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300 import synth
    from mla_latent_cache_absorb_gb300.runner import DeviceStep

    wl = synth.WORKLOADS[name].with_(tokens=tokens)
    prob = synth.make_problem(wl)
    Lb = prob.seq_lens.astype(np.int64)
    # rows each token attends, summed (token i of b: L_b - T + 1 + i), and distinct rows read
    token_rows = int(sum(int(l) * tokens - tokens * (tokens - 1) // 2 for l in Lb))
    row_bytes = (wl.C + wl.R) * (2 if wl.act == "bf16" else 4)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 2 ** 20)
    per_copy = input_bytes(prob)
    R = max(1, min(32, math.ceil(2.2 * l2 / per_copy)))
    stream = torch.cuda.Stream(device=device)
    copies = [DeviceStep(prob, device=device, stream=stream) for _ in range(R)]
    G = R * max(1, math.ceil(16 / R))

    def timed(call):
        with torch.cuda.stream(stream):
            for i in range(W):
                L.check(call(copies[i % R], stream), "warm-up")
            torch.cuda.synchronize(device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                s = torch.cuda.current_stream(device)
                for i in range(G):
                    L.check(call(copies[i % R], s), "captured call")
            g.replay()
            torch.cuda.synchronize(device)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n = max(1, K // G)
            e0.record(stream)
            for _ in range(n):
                g.replay()
            e1.record(stream)
            e1.synchronize()
            return e0.elapsed_time(e1) / (n * G)

    def multi(ds, s):
        return ds.decode_multi(s)

    def singles(ds, s):
        # the T tokens one call each (token i: its query, position and length), as without
        # multi-token decode
        st = 0
        for i in range(tokens):
            st = st or L.mla_decode_attn(ds.cfg, ds.q_tok[i], ds.kv_b, ds.cache, ds.len_tok[i], ds.pos_tok[i],
                                         ds.out_tok, ds.lse_tok, wl.B, ds.ws_tok, ds.ws_tok.numel(), s)
        return st

    for ds in copies:
        ds.q_tok = [ds.q[:, i].contiguous() for i in range(tokens)]
        ds.len_tok = [(ds.seq_lens - (tokens - 1 - i)).contiguous() for i in range(tokens)]
        ds.pos_tok = [(ds.positions + i).contiguous() for i in range(tokens)]
        ds.out_tok = torch.empty((wl.B, wl.H, wl.V), dtype=torch.float32, device=device)
        ds.lse_tok = torch.empty((wl.B, wl.H), dtype=torch.float32, device=device)
        st, n = L.mla_decode_workspace_size(ds.cfg, wl.B)
        L.check(st, "mla_decode_workspace_size")
        ds.ws_tok = torch.zeros(n, dtype=torch.uint8, device=device)
    ms_multi = timed(multi)
    ms_single = timed(singles)
    st, plan = L.mla_decode_plan(copies[0].cfg, wl.B)
    del copies
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()
    hbm = peaks()[0]
    distinct = int(Lb.sum()) * row_bytes
    return {"workload": wl.name, "tokens": tokens, "B": wl.B, "H": wl.H, "token_rows_per_call": token_rows,
            "us_per_call": ms_multi * 1e3, "token_rows_per_s": token_rows / (ms_multi / 1e3),
            "cache_gbs_distinct_rows": distinct / (ms_multi / 1e3) / 1e9,
            "cache_hbm_frac": distinct / (ms_multi / 1e3) / 1e9 / hbm,
            "us_as_one_token_calls": ms_single * 1e3, "speedup_vs_one_token_calls": ms_single / ms_multi,
            "one_token_attention_kernel": plan.kernel}


def run_e2e(torch, L, steps, prob, stream, device, K, W, work):
    """Same metric through the public calls with host buffers: every step copies its inputs
    (query, kv_a rows, positions, lengths) from one pinned host buffer into the step's device
    inputs with one copy, calls mla_cache_append + mla_decode_attn, and copies out + lse back
    with one copy; launched eagerly (no graph)."""
    R = len(steps)
    names = ["q", "kv_in", "positions", "len_before", "seq_lens"]

    def packed(ds, tensors, dev):
        """one 256-byte-aligned byte buffer holding `tensors` (name -> tensor) back to back,
        plus views of it with their shapes and dtypes"""
        offs, off = {}, 0
        for k, t in tensors.items():
            offs[k] = off
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(off, dtype=torch.uint8, device=dev)
        if dev == "cpu":
            buf = buf.pin_memory()
        views = {k: buf[offs[k]:offs[k] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                 for k, t in tensors.items()}
        return buf, views

    # every device step gets its inputs and outputs re-homed into one packed buffer each
    dev_in, dev_out = [], []
    for ds in steps:
        b_in, v_in = packed(ds, {k: getattr(ds, k) for k in names}, device)
        for k in names:
            v_in[k].copy_(getattr(ds, k))
            setattr(ds, k, v_in[k])
        b_out, v_out = packed(ds, {"out": ds.out, "lse": ds.lse}, device)
        ds.out, ds.lse = v_out["out"], v_out["lse"]
        dev_in.append(b_in)
        dev_out.append(b_out)
    ds0 = steps[0]
    host_in, hv = packed(ds0, {k: getattr(ds0, k) for k in names}, "cpu")
    for k in names:
        hv[k].copy_(getattr(ds0, k))
    host_out, _ = packed(ds0, {"out": ds0.out, "lse": ds0.lse}, "cpu")
    h2d = sum(getattr(ds0, k).numel() * getattr(ds0, k).element_size() for k in names)
    d2h = ds0.out.numel() * 4 + ds0.lse.numel() * 4

    def one(i):
        ds = steps[i % R]
        dev_in[i % R].copy_(host_in, non_blocking=True)
        L.check(ds.append(stream), "mla_cache_append")
        L.check(ds.decode(stream), "mla_decode_attn")
        host_out.copy_(dev_out[i % R], non_blocking=True)

    for i in range(W):
        one(i)
    torch.cuda.synchronize(device)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(K):
        one(i)
    b.record(stream)
    b.synchronize()
    ms = a.elapsed_time(b)
    return {"value": work["rows"] * K / (ms / 1e3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / K,
            "launch": "eager, one call each per step; one packed copy in and one out per step"}


# ------------------------------------------------------------------------------------------------
# the CPU oracle: cpu_baseline leg and the reference arm
# ------------------------------------------------------------------------------------------------

def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# The oracle runs in spawned worker processes, one sequence-step per task, each worker with one
# BLAS thread, so `cores` is the number of processes that actually ran it. A task carries only
# its sequence's rows (in logical order), so the workers never hold the whole cache.
_OW = {}


def _oracle_worker_init(wl, shared):
    _OW["wl"] = wl
    _OW["shared"] = shared


def _oracle_task(task):
    """One sequence's whole step (append + decode over `heads` heads) on the oracle, as a
    one-sequence contiguous problem holding that sequence's rows. Returns rows credited."""
    from mla_latent_cache_absorb_gb300 import synth
    from oracle import step as OS
    rows, q, kva, x, pos, L, nheads = task
    wl = _OW["wl"].with_(B=1, page_size=0)
    sh = _OW["shared"]
    prob = synth.Problem(wl=wl, q=q, pool=rows, page_table=None, rows_per_seq=rows.shape[0], max_pages=0,
                         positions=np.array([pos], np.int32), seq_lens=np.array([L], np.int32),
                         norm_w=sh["norm_w"], kv_b=sh["kv_b"], kva_rows=kva, x=x, w_kva=sh["w_kva"])
    OS.run_step(prob, seqs=[0], heads=np.arange(nheads))
    return float(L) * nheads / _OW["wl"].H


class OracleSampler:
    """A pool of spawned processes that time the oracle over bounded samples of a workload."""

    def __init__(self, prob, workers=None):
        import multiprocessing as mp
        self.prob = prob
        self.workers = workers or host_cores()
        shared = {"norm_w": prob.norm_w, "kv_b": prob.kv_b, "w_kva": prob.w_kva}
        keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in keep:
            os.environ[k] = "1"   # inherited by the spawned workers only
        try:
            self.pool = mp.get_context("spawn").Pool(self.workers, _oracle_worker_init, (prob.wl, shared))
        finally:
            for k, v in keep.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def task(self, b, nheads):
        from oracle import mla_oracle as O
        p, wl = self.prob, self.prob.wl
        L = int(p.seq_lens[b])
        phys = O.physical_row(b, np.arange(L), p.page_table, wl.page_size, p.rows_per_seq)
        kva = None if p.kva_rows is None else p.kva_rows[b:b + 1]
        x = None if p.x is None else p.x[b:b + 1]
        return (p.pool[phys], p.q[b:b + 1], kva, x, int(p.positions[b]), L, nheads)

    def run(self, seqs, nheads):
        """Wall time of computing the given sequence-steps in parallel; rows credited."""
        tasks = [self.task(b, nheads) for b in seqs]
        t0 = time.perf_counter()
        rows = sum(self.pool.map(_oracle_task, tasks, chunksize=1))
        return rows, time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(prob, seconds):
    """The oracle on all host cores over a bounded sample: one round of one sequence-step per
    worker to size the sample, then enough rounds to take about `seconds`."""
    wl = prob.wl
    smp = OracleSampler(prob)
    try:
        nxt = 0

        def seqs(n):
            nonlocal nxt
            out = [(nxt + i) % wl.B for i in range(n)]
            nxt += n
            return out

        r0, t0 = smp.run(seqs(smp.workers), wl.H)
        rounds = max(1, int(seconds / max(t0, 1e-3)))
        rows, dt = smp.run(seqs(rounds * smp.workers), wl.H)
    finally:
        smp.close()
    return {"value": rows / dt, "unit": "rows/s", "cores": smp.workers, "kind": "oracle",
            "sample": f"{rounds * smp.workers} oracle sequence-steps (append + decode of one sequence, all "
                      f"{wl.H} heads; sequences taken in order, wrapping), {rows:.0f} rows in {dt:.1f} s, fp64 "
                      f"numpy in {smp.workers} processes with one BLAS thread each, after one sizing round"}


def run_reference(args, budget_s=150.0):
    """The oracle as it stands, timed on the host cores. Each step is a bounded sample of the
    workload: one sequence-step per worker process (the next sequences in order), all heads when
    that fits the time budget (budget_s over all warm-up and timed steps), else the first heads
    only; rows are credited in proportion to the heads computed."""
    from mla_latent_cache_absorb_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    prob = synth.make_problem(wl)
    work = step_work(prob)
    smp = OracleSampler(prob)
    try:
        nw = smp.workers
        _, t_one = smp.run(list(range(min(nw, wl.B))), wl.H)
        per_step = budget_s / (args.steps + args.warmup)
        hs = wl.H if t_one <= per_step else max(1, int(wl.H * per_step / t_one))
        k = [0]

        def step():
            seqs = [(k[0] * nw + i) % wl.B for i in range(nw)]
            k[0] += 1
            return smp.run(seqs, hs)

        for _ in range(args.warmup):
            step()
        rows, dt = 0.0, 0.0
        for _ in range(args.steps):
            r, t = step()
            rows += r
            dt += t
    finally:
        smp.close()
    value = rows / dt
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator)",
        "config": workload_config(wl, prob, work),
        "cpu_baseline": {"value": value, "unit": "rows/s", "kind": "oracle", "cores": nw,
                         "sample": f"{args.steps} steps of {nw} oracle sequence-steps each ({hs} of {wl.H} "
                                   f"heads, append + decode, one per worker process with one BLAS thread) "
                                   f"after {args.warmup} warm-up steps, {rows:.0f} rows credited in {dt:.1f} s"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-also", action="store_true", help="skip the attention sub-records")
    ap.add_argument("--no-proj", action="store_true", help="skip the layer-projection sub-records")
    ap.add_argument("--proj-only", action="store_true", help="print only the layer-projection records")
    ap.add_argument("--no-multi", action="store_true", help="skip the multi-token decode sub-records")
    ap.add_argument("--multi-only", action="store_true", help="print only the multi-token decode records")
    ap.add_argument("--proj-filter", default=None,
                    help="with --proj-only: one 'workload:format' record (e.g. v3_proj_b4:bf16)")
    ap.add_argument("--clock-window-s", type=float, default=1.2,
                    help="seconds of untimed replays to sample clocks when the timed region is too short")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if args.steps is None:
            args.steps = 20
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    if args.steps is None:
        args.steps = 20000 if args.workload == "v2lite_b1_t4096" else 200
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.multi_only:
        for (name, t), k in MULTI_BENCH.items():
            print(json.dumps(run_multi_tokens(device, name, t, k, args.warmup)), flush=True)
        return
    if args.proj_only:
        for (name, fmt), k in PROJ_BENCH.items():
            if args.proj_filter and args.proj_filter != f"{name}:{fmt}":
                continue
            print(json.dumps(run_proj(device, name, fmt, k, args.warmup)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    line = run_ours(args, rank, world, device, args.workload, args.steps, args.warmup,
                    with_e2e=not args.no_e2e, with_clocks=True)
    if not args.no_also:
        also = {}
        for wname, k in ALSO_WORKLOADS.items():
            if wname == args.workload:
                continue
            sub = run_ours(args, rank, world, device, wname, k, args.warmup, with_e2e=False, with_clocks=False)
            also[wname] = {"kernel": sub["roofline"]["kernel"],
                           "roofline_frac": sub["roofline"]["frac"], "avg_launch_us": sub["roofline"]["avg_launch_us"],
                           "attn_gbs": sub["roofline"]["achieved"], "ms_per_step": sub["ms_per_step"],
                           "rows_per_s": sub["value"], "steps": k, "heads_per_cta": sub["run"]["heads_per_cta"]}
            line["gpu_launches"] += sub["gpu_launches"]
        line["also"] = {"what": "attention kernel of other workloads, same run, same timing method "
                                "(not part of value or ms_per_step; their launches are counted in gpu_launches)",
                        **also}
    if not args.no_proj:
        recs = [run_proj(device, name, fmt, k, args.warmup) for (name, fmt), k in PROJ_BENCH.items()]
        for r in recs:
            line["gpu_launches"] += r["launches_per_step"] * r["steps"]
        line["layer_projections"] = {
            "what": "mla_front_end (q chain or q projection + kv_a) and mla_o_proj per call, median of "
                    "in-graph events, weights rotating over copies > 2.2x L2 (not part of value)",
            "records": recs}
    if not args.no_multi:
        recs = [run_multi_tokens(device, name, t, k, args.warmup) for (name, t), k in MULTI_BENCH.items()]
        for (name, t), r in zip(MULTI_BENCH, recs):
            line["gpu_launches"] += 3 * (1 + t) * MULTI_BENCH[(name, t)]
        line["multi_token"] = {
            "what": "mla_decode_attn_multi (T tokens per sequence, causal) per call vs the same tokens as T "
                    "one-token calls; CUDA graphs, inputs rotating over copies > 2.2x L2 (not part of value)",
            "records": recs}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from mla_latent_cache_absorb_gb300 import synth
        line["cpu_baseline"] = cpu_baseline(synth.make_problem(synth.WORKLOADS[args.workload]), args.cpu_seconds)
    else:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
