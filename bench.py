"""Benchmark: batch-1 ternary decode over the 30-layer BitNet-b1.58-2B4T-shaped
stack (210 projections, 2.08e9 weights, 521 MB of .trit v1 planes).

One step = one decode token: quantise the 210 fresh fp32 activation vectors
and compute the 210 ternary products, in one persistent launch (the fused
kernel), inputs resident in HBM.  Weights are synthetic, seeded, drawn with per-layer
zero fractions uniform in [0.385, 0.508]; the 521 MB of planes exceed the
129 MB L2, so every step streams them from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores instead (a bounded sample of the same workload per step).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("batch-1 ternary GEMV HBM GB/s (% of GB300 peak) and tok/s over 30-layer stack")
WORKLOAD = "bitnet-2b4t-30layer-ternary-decode-batch1"
SEED = 2
FALLBACK_HBM_GBS = 6800.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over all ranks of the process group (x itself when there is
    no group or one rank): every replica's time, the job's time is the slowest."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_rates(step_bytes: int, steps: int, total_ms: float, world: int):
    """Whole-job GB/s and tok/s of `world` replicas that each ran `steps` steps
    of `step_bytes` in (at most) total_ms."""
    secs = total_ms * 1e-3
    return world * step_bytes * steps / secs / 1e9, world * steps / secs


# ---- clocks -----------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, wait_first: float = 0.0):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.wait_first = wait_first

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # nvidia-smi takes a moment to start: wait (bounded) for its first line
            # so that the samples cover what follows
            t0 = time.time()
            while self.wait_first and not self.lines and time.time() - t0 < self.wait_first:
                time.sleep(0.05)
            self.skip = len(self.lines)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines[getattr(self, "skip", 0):]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- workload -----------------------------------------------------------------

def build_stack(device, layers: int):
    import numpy as np
    import torch

    import synth
    from bit_plane_select_gb300.stack import TernaryStack

    st = TernaryStack(device)
    for layer, idx, name, N, K in synth.stack_items(layers):
        w = synth.stack_weights(SEED, layer, idx)
        st.add(torch.from_numpy(w), float(synth.w_scale(w)), M=1, name=f"L{layer}.{name}")
    st.finalize()
    for i, (layer, idx, name, N, K) in enumerate(synth.stack_items(layers)):
        st.x[i].copy_(torch.from_numpy(synth.projection_acts(SEED, layer, idx, 1)))
    torch.cuda.synchronize()
    return st


def read_probe_gbs(dev, gib: int = 2, reps: int = 5):
    """Same-run read rate of the device memory: trit_read_probe over a buffer far
    larger than L2, best of `reps` launches timed with CUDA events."""
    import torch

    import bit_plane_select_gb300 as t
    nbytes = gib << 30
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    buf.fill_(1)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    t.trit_read_probe(buf, sink)
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        t.trit_read_probe(buf, sink)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1)
        best = ms if best is None or ms < best else best
    del buf
    torch.cuda.empty_cache()
    return round(nbytes / (best * 1e-3) / 1e9, 1)


def source_hash(paths):
    """Hash of the kernel sources' code: comments and blank lines are left out,
    so that a comment edit does not retire the DRAM counters taken on the same
    code."""
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for line in text.splitlines():
            code = re.sub(r"//.*$", "", line).rstrip()
            if code.strip():
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


GEMV_SOURCES = ["bit_plane_select_gb300/csrc/trit_gemv.cu",
                "bit_plane_select_gb300/csrc/trit_internal.cuh"]


def committed_traffic(bytes_per_launch_expected):
    """DRAM bytes per launch of the product kernel from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "select_accumulate_stack30.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_hash") != source_hash(GEMV_SOURCES):
        return None
    return d.get("dram_bytes_per_launch")


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()

    st = build_stack(dev, args.layers)
    stream = torch.cuda.current_stream(dev)

    # warm-up
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    st.err.zero_()

    K = args.steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # The step is exactly one launch, so the launches are timed as a whole: an
    # event pair around every launch would separate consecutive launches and
    # stop the next token's set-up from overlapping the current one's tail.
    with ClockSampler(local) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(K):
            st.step()                      # one fused launch: quantise + 210 products
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    err = int(st.err.item())

    # context: one launch alone, bracketed by its own events (no overlap)
    I = max(1, min(K, 200))
    evi = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(I)]
    for i in range(I):
        evi[i][0].record(stream)
        st.step()
        evi[i][1].record(stream)
    torch.cuda.synchronize()
    isolated_ms = sorted(evi[i][0].elapsed_time(evi[i][1]) for i in range(I))[I // 2]

    # context: the two-launch path (quantise, then multiply) on the same data
    T = max(1, min(K, args.two_launch_steps))
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(T)]
    for _ in range(3):
        st.step_two_launch()
    torch.cuda.synchronize()
    for i in range(T):
        ev2[i][0].record(stream)
        st.quantize()
        ev2[i][1].record(stream)
        st.products()
        ev2[i][2].record(stream)
    torch.cuda.synchronize()
    two_quant = sum(ev2[i][0].elapsed_time(ev2[i][1]) for i in range(T)) / T
    two_prod = sum(ev2[i][1].elapsed_time(ev2[i][2]) for i in range(T)) / T

    total_ms = max_over_ranks(total_ms, dev)

    ms_per_step = total_ms / K
    step_bytes = st.fused_bytes()
    value, tok_s = replica_rates(step_bytes, K, total_ms, world)     # whole job
    peak, peak_kind = peaks()

    # dominant (only) kernel of the step: the fused quantise-and-multiply launch;
    # its average duration over the timed region is the region / K (one launch
    # per step, gaps between launches included)
    kern_avg_ms = total_ms / K
    achieved = step_bytes / (kern_avg_ms * 1e-3) / 1e9
    traffic = committed_traffic(step_bytes)
    probe_gbs = read_probe_gbs(dev)

    # e2e: host fp32 activations in, host y_i32 + y_f32 out, every step.  Two
    # buffer sets (twin stacks over the same planes) and three streams: the
    # copy in of step i+1 and the copy out of step i-1 run while step i
    # computes; every step still moves its own inputs and outputs.
    sts = [st, st.twin()]
    x_host = st.x_arena.cpu().pin_memory()
    y_host = [torch.empty_like(st.y_arena, device="cpu").pin_memory() for _ in range(2)]
    f_host = [torch.empty_like(st.f_arena, device="cpu").pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for k in range(2):
        ev_out[k].record(s_out)

    def e2e_step(i):
        k = i & 1
        b = sts[k]
        s_in.wait_event(ev_out[k])                # this slot's previous outputs are home
        with torch.cuda.stream(s_in):
            b.x_arena.copy_(x_host, non_blocking=True)
        ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        b.step(stream)
        ev_comp[k].record(stream)
        s_out.wait_event(ev_comp[k])
        with torch.cuda.stream(s_out):
            y_host[k].copy_(b.y_arena, non_blocking=True)
            f_host[k].copy_(b.f_arena, non_blocking=True)
        ev_out[k].record(s_out)

    E = max(1, min(K, args.e2e_steps))
    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(E):
        e2e_step(i)
    stream.wait_stream(s_out)
    stream.wait_stream(s_in)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / E, dev)
    # the serial form for context: copy in, step, copy out on one stream
    for _ in range(3):
        st.x_arena.copy_(x_host, non_blocking=True)
        st.step()
        y_host[0].copy_(st.y_arena, non_blocking=True)
        f_host[0].copy_(st.f_arena, non_blocking=True)
    torch.cuda.synchronize()
    S = max(1, min(E, 500))
    e0.record(stream)
    for _ in range(S):
        st.x_arena.copy_(x_host, non_blocking=True)
        st.step()
        y_host[0].copy_(st.y_arena, non_blocking=True)
        f_host[0].copy_(st.f_arena, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    serial_ms = e0.elapsed_time(e1) / S
    h2d = st.x_arena.numel() * 4
    d2h = st.y_arena.numel() * 4 + st.f_arena.numel() * 4

    # seconds-long, clock-sampled pass of the same step, the issue rates the
    # batch floors use, and the other four configurations (single GPU runs)
    rates = measure_issue_rates(dev)
    sus = sustained_pass(st, local, stream, step_bytes, peak)
    configs = None
    if world == 1 and not args.no_configs:
        torch.cuda.empty_cache()
        configs = {"config0": gpu_config0(dev, stream, peak),
                   "config1": gpu_config1(dev, stream, peak),
                   "config2": "this line (value, roofline, e2e)"}
        torch.cuda.empty_cache()
        configs["config3"] = gpu_config3(st.planes, st.specs, dev, stream, peak,
                                         sus["clocks"]["sm_mhz"], rates)
        torch.cuda.empty_cache()
        configs["config4"] = gpu_config4(dev, stream, args.layers, max(5, min(20, K)), 3)
        torch.cuda.empty_cache()
        # config 2's token in dependency order (beside this line's independent step)
        forms, _, oerr = decode_ordered(dev, stream, args.layers, 500, 5, ("paired",))
        configs["config2_ordered"] = dict(forms["paired"], err_flag=oerr, mlp_form="paired",
                                          timing="CUDA graph of one token replayed 500 times")
        torch.cuda.empty_cache()
    timed_clk = clk.summary()
    clocks = dict(sus["clocks"])
    clocks["sampled_during"] = (f"the sustained pass: {sus['launches']} back-to-back launches of this "
                                f"step ({sus['seconds']} s) in this run; the {K}-step timed region lasts "
                                f"{total_ms:.1f} ms, under nvidia-smi's 200 ms period")
    clocks["timed_region_samples"] = timed_clk["samples"]

    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "tok_per_s": round(tok_s, 1),
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8",
        "data": "synthetic",
        "config": {
            "workload": WORKLOAD,
            "layers": args.layers,
            "projections": len(st.specs),
            "batch": 1,
            "weights": st.weights,
            "plane_bytes": st.plane_bytes,
            "algorithmic_bytes_per_step": step_bytes,
            "l2": "inputs larger than L2: 521 MB of planes streamed per step (L2 129 MB)",
            "parallelism": f"replicas{world}" if world > 1 else "single",
        },
        "roofline": {
            "kernel": "select_accumulate_kernel<1>, fused quantise + 210 products "
                      "(trit_quant_gemv_many, one launch per token)",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": step_bytes,
            "avg_launch_us": round(kern_avg_ms * 1e3, 3),
            "avg_launch_from": "CUDA events around the K back-to-back launches of the timed "
                               "region, divided by K",
            "isolated_launch_us": round(isolated_ms * 1e3, 3),
            "probe_read_gbs": probe_gbs,
            "frac_of_probe": round(achieved / probe_gbs, 4) if probe_gbs else None,
            "probe": "trit_read_probe over a 2 GiB buffer in the same run, best of 5 "
                     "(plain coalesced 16-byte reads)",
            "sustained": {k: v for k, v in sus.items() if k != "clocks"},
        },
        "issue_rates": {k: v["lanes_per_clk"] for k, v in rates.items()},
        "two_launch_path": {
            "quant_us": round(two_quant * 1e3, 3),
            "product_us": round(two_prod * 1e3, 3),
            "product_gbs": round(st.product_bytes() / (two_prod * 1e-3) / 1e9, 1),
            "steps": T,
        },
        "e2e": {
            "value": round(step_bytes / (e2e_ms * 1e-3) / 1e9 * world, 1),
            "unit": "GB/s",
            "tok_per_s": round(world / (e2e_ms * 1e-3), 1),
            "ms_per_step": round(e2e_ms, 5),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "steps": E,
            "pipelining": "two buffer sets; copy in of step i+1 and copy out of step i-1 "
                          "overlap step i",
            "serial_ms_per_step": round(serial_ms, 5),
        },
        "gpu_launches": K,
        "err_flag": err,
        "clocks": clocks,
    }
    if configs is not None:
        out["configs"] = configs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_layers)
        out["cpu_baseline"]["all_cores"] = cpu_baseline_all_cores(args.cpu_layers)
        out["cpu_baseline"]["configs"] = cpu_baseline_configs()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---- the other configurations, measured in the default run ------------------

L2_BYTES = 129 * 1024 * 1024   # GB300 L2; rotating copies span at least 4x this


def _events_ms(fn, n, stream):
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def sustained_pass(st, gpu: int, stream, step_bytes: int, peak: float, seconds: float = 2.5):
    """Back-to-back fused decode launches for about `seconds`, with nvidia-smi
    sampling the clocks throughout (the K-step region is too short to sample)."""
    import torch
    ms_one = _events_ms(lambda i: st.step(), 50, stream) / 50
    n = max(1000, int(seconds / (ms_one * 1e-3)))
    with ClockSampler(gpu, wait_first=3.0) as clk:
        total_ms = _events_ms(lambda i: st.step(), n, stream)
    ms = total_ms / n
    gbs = step_bytes / (ms * 1e-3) / 1e9
    return {"launches": n, "seconds": round(total_ms * 1e-3, 3), "us_per_step": round(ms * 1e3, 3),
            "achieved": round(gbs, 1), "frac": round(gbs / peak, 4), "tok_per_s": round(1e3 / ms, 1),
            "clocks": clk.summary()}


def gpu_config0(dev, stream, peak: float):
    """Config 0: one 2560 x 2560 product at batch 1, int8 activations, over
    rotating copies of the planes spanning >= 4x L2.  Two forms: one call per
    product (trit_gemv, scale by value; launch-latency bound) and every copy in
    one list call (trit_gemm_many: the stream rate)."""
    import torch

    import bit_plane_select_gb300 as t
    import synth
    w, x = synth.config0()
    ws = float(synth.w_scale(w))
    planes0, _ = t.trit_pack(torch.from_numpy(w).to(dev), ws)
    xq, xsc, _ = t.trit_quant_act(torch.from_numpy(x).to(dev))
    xs_host = float(xsc.item())
    nb = planes0.numel()
    copies = -(-4 * L2_BYTES // nb)
    planes = [planes0.clone() for _ in range(copies)]
    y = torch.empty(2560, dtype=torch.int32, device=dev)
    f = torch.empty(2560, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    per = nb + 2560 + 4 + 8 * 2560          # planes + int8 x + scale + y_i32 + y_f32
    call = lambda i: t.trit_gemv(planes[i % copies], ws, xq[0], xs_host, 2560, y, f, err)
    for i in range(copies):
        call(i)
    n = 4 * copies
    ms = _events_ms(call, n, stream) / n
    ys = [torch.empty((1, 2560), dtype=torch.int32, device=dev) for _ in range(copies)]
    fs = [torch.empty((1, 2560), dtype=torch.float32, device=dev) for _ in range(copies)]
    plist = t.ProjList([(planes[i], ws, xq, xsc, 2560, ys[i], fs[i]) for i in range(copies)])
    t.trit_gemm_many(plist, err)
    reps = 20
    ms_all = _events_ms(lambda i: t.trit_gemm_many(plist, err), reps, stream) / reps
    same = all(torch.equal(ys[i][0], y) for i in range(0, copies, 37))
    gbs_call = per / (ms * 1e-3) / 1e9
    gbs_all = per * copies / (ms_all * 1e-3) / 1e9
    return {"workload": "single ternary GEMV 2560x2560, batch 1, int8 activations",
            "rotating_copies": copies, "bytes_per_product": per,
            "per_call": {"us": round(ms * 1e3, 3), "GBs": round(gbs_call, 1),
                         "frac_of_peak": round(gbs_call / peak, 4), "calls": n},
            "one_list_call": {"us_per_product": round(ms_all * 1e3 / copies, 3),
                              "GBs": round(gbs_all, 1), "frac_of_peak": round(gbs_all / peak, 4),
                              "products_per_call": copies},
            "outputs_identical_across_copies": bool(same), "err_flag": int(err.item())}


def gpu_config1(dev, stream, peak: float):
    """Config 1: one BitNet-shaped layer (seven products) at batch 1, fp32
    activations quantised in the same launch (trit_quant_gemv_many), over
    rotating copies of the layer's planes spanning >= 4x L2."""
    import torch

    import bit_plane_select_gb300 as t
    import synth
    layer = synth.config1()
    packed = []
    for name, w, x in layer:
        ws = float(synth.w_scale(w))
        pl, _ = t.trit_pack(torch.from_numpy(w).to(dev), ws)
        packed.append((pl, ws, torch.from_numpy(x.reshape(-1)).to(dev), w.shape[0], w.shape[1]))
    nb = sum(p[0].numel() for p in packed)
    copies = -(-4 * L2_BYTES // nb)
    outs = [(torch.empty(N, dtype=torch.int32, device=dev), torch.empty(N, dtype=torch.float32, device=dev))
            for _, _, _, N, _ in packed]
    lists = []
    for c in range(copies):
        ents = []
        for (pl, ws, x, N, K), (y, f) in zip(packed, outs):
            ents.append((pl if c == 0 else pl.clone(), ws, x, None, None, y, f))
        lists.append(t.QProjList(ents))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    step = lambda i: t.trit_quant_gemv_many(lists[i % copies], err)
    for i in range(copies):
        step(i)
    n = 10 * copies
    ms = _events_ms(step, n, stream) / n
    per = sum(pl.numel() + 4 * K + ((K + 63) // 64) * 64 + 4 + 8 * N for pl, _, _, N, K in packed)
    gbs = per / (ms * 1e-3) / 1e9
    return {"workload": "one BitNet-2B4T-shaped layer (7 projections), batch 1, fused quantise + product",
            "rotating_copies": copies, "bytes_per_layer": per, "us_per_layer": round(ms * 1e3, 3),
            "GBs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "launches_per_layer": 1,
            "err_flag": int(err.item())}


# ---- the CPU oracle ---------------------------------------------------------

def oracle_sample(layers, rows_frac=1.0, shard=0, nshards=1):
    """Pack (untimed) the sampled projections with the oracle; returns a list of
    (payload, w_scale, x fp32, K, rows) items (every nshards-th projection from
    `shard` on)."""
    import numpy as np

    import oracle
    import synth

    items = []
    for i, (layer, idx, name, N, K) in enumerate(synth.stack_items(layers)):
        if i % nshards != shard:
            continue
        w = synth.stack_weights(SEED, layer, idx)
        n = max(1, int(round(N * rows_frac)))
        items.append((oracle.pack(w[:n]), float(synth.w_scale(w)),
                      synth.projection_acts(SEED, layer, idx, 1), K, n))
    return items


def oracle_step(items):
    import oracle
    for payload, ws, x, K, n in items:
        q, s, _ = oracle.quant(x)
        oracle.gemm(payload, ws, q, s, K)


def cpu_baseline(layers):
    """The oracle as it stands, single-threaded, on the first `layers` layers of
    the same stack; scaled to the full 30-layer token."""
    import synth
    items = oracle_sample(layers)
    weights = sum(N * K for _, _, _, N, K in synth.stack_items(layers))
    passes = 0
    t = time.perf_counter()
    while True:                            # whole passes, about 10 s of CPU work
        oracle_step(items)
        passes += 1
        if time.perf_counter() - t >= 10.0 or passes >= 8:
            break
    dt = (time.perf_counter() - t) / passes
    full = sum(N * K for _, _, _, N, K in synth.stack_items(synth.LAYERS))
    token_s = dt * full / weights
    plane_b = weights / 4
    return {"value": round(plane_b / dt / 1e9, 3), "unit": "GB/s",
            "tok_per_s": round(1.0 / token_s, 4), "cores": 1, "kind": "oracle",
            "sample": f"layers 0..{layers - 1} of the 30-layer stack ({len(items)} projections, "
                      f"{weights} weights), quantise + product, {passes} passes of "
                      f"{dt:.2f} s each"}


def cpu_baseline_configs(seconds: float = 2.0):
    """The oracle, single-threaded, on the two small workloads: one 2560 x 2560
    product (P(0) = 0.4219) and one layer (seven products); quantise + product,
    whole passes for about `seconds` each."""
    import oracle
    import synth
    w0, x0 = synth.config0()
    cases = {"single_product_2560x2560": [(oracle.pack(w0), float(synth.w_scale(w0)), x0, 2560, 2560)],
             "one_layer_7_products": [(oracle.pack(w), float(synth.w_scale(w)), x, w.shape[1], w.shape[0])
                                      for _, w, x in synth.config1()]}
    out = {}
    for name, items in cases.items():
        weights = sum(n * K for _, _, _, K, n in items)
        passes, t = 0, time.perf_counter()
        while True:
            oracle_step(items)
            passes += 1
            if time.perf_counter() - t >= seconds:
                break
        dt = (time.perf_counter() - t) / passes
        out[name] = {"weights_per_s": round(weights / dt), "plane_gbs": round(weights / 4 / dt / 1e9, 4),
                     "cores": 1, "passes": passes, "s_per_pass": round(dt, 4)}
    return out


def _oracle_shard(layers, shard, nshards, seconds, barrier, q):
    items = oracle_sample(layers, shard=shard, nshards=nshards)
    import synth
    weights = sum(N * K for i, (_, _, _, N, K) in enumerate(synth.stack_items(layers))
                  if i % nshards == shard)
    barrier.wait()
    passes, t = 0, time.perf_counter()
    while True:
        oracle_step(items)
        passes += 1
        if time.perf_counter() - t >= seconds:
            break
    q.put((passes * weights, time.perf_counter() - t))


def cpu_baseline_all_cores(layers, seconds: float = 8.0):
    """The same oracle on every host core: the stack's projections dealt round
    robin to one spawned process per core, each running whole passes over its
    share for about `seconds`; throughput = weights processed / slowest time."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    ctx = mp.get_context("spawn")
    barrier, q = ctx.Barrier(cores + 1), ctx.Queue()
    procs = [ctx.Process(target=_oracle_shard, args=(layers, i, cores, seconds, barrier, q))
             for i in range(cores)]
    for pr in procs:
        pr.start()
    barrier.wait()
    res = [q.get() for _ in procs]
    for pr in procs:
        pr.join()
    done = sum(w for w, _ in res)
    wall = max(dt for _, dt in res)
    import synth
    full = sum(N * K for _, _, _, N, K in synth.stack_items(synth.LAYERS))
    return {"value": round(done / 4 / wall / 1e9, 3), "unit": "GB/s",
            "tok_per_s": round(done / full / wall, 4), "cores": cores, "kind": "oracle",
            "sample": f"layers 0..{layers - 1}, projections dealt round robin to {cores} "
                      f"processes, about {seconds:.0f} s of whole passes each"}


def run_reference(args):
    """The CPU oracle timed on the host cores, each step a bounded sample of the
    token: a fixed fraction of every projection's rows."""
    import synth
    rank, world, local = dist_env()
    if rank != 0:
        return
    budget_s = args.reference_budget
    steps = args.steps + args.warmup
    full = sum(N * K for _, _, _, N, K in synth.stack_items(synth.LAYERS))
    # calibrate: one projection
    cal = oracle_sample(1, rows_frac=0.05)
    t = time.perf_counter()
    oracle_step(cal)
    cal_s = (time.perf_counter() - t) / sum(n * K for _, _, _, K, n in cal)
    frac = min(1.0, budget_s / steps / (cal_s * full))
    frac = max(frac, 1.0 / 2560)
    items = oracle_sample(synth.LAYERS, rows_frac=frac)
    w_sample = sum(n * K for _, _, _, K, n in items)
    b_sample = sum(n * ((K + 63) // 64) * 16 + K + 4 + 8 * n for _, _, _, K, n in items)
    for _ in range(args.warmup):
        oracle_step(items)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(items)
    dt = (time.perf_counter() - t) / args.steps
    value = b_sample / dt / 1e9
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "tok_per_s": round(w_sample / full / dt, 6),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": synth.LAYERS, "batch": 1},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{frac:.5f} of the rows of each of the 210 projections "
                                   f"({w_sample} weights) per step, quantise + product"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ---- other workloads (extra lines; the default run is the decode stack) --------

def _timed(fn, steps, warmup, stream):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_prefill(args):
    """Config 4 alone: prefill TFLOP/s at M = 512 and 2048."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    r = gpu_config4(dev, torch.cuda.current_stream(dev), args.layers, args.steps, args.warmup)
    M = max(r["by_M"])
    best = r["by_M"][M]
    print(json.dumps({"metric": "prefill ternary GEMM TFLOP/s (30 layers x gate/up/down, tensor cores)",
                      "value": best["tflops"], "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
                      "warmup": args.warmup, "higher_is_better": True,
                      "dtype": "int8 (fp16 tensor operands, fp32 accumulation)", "data": "synthetic",
                      "config": {"workload": f"prefill-gate-up-down-{args.layers}layers-M{M}"},
                      "roofline": {"bound": "tensor", "achieved": best["tflops"],
                                   "peak": r["peak_tflops"]["bf16_sustained"], "unit": "TFLOP/s",
                                   "frac": best["frac_of_sustained_peak"],
                                   "peak_kind": r["peak_tflops"]["kind"] + " (bf16 sustained)"},
                      "clocks": best["clocks"], "detail": r}), flush=True)


def run_batch_sweep(args):
    """Config 3 alone: batched decode over the 30-layer stack at every M of the sweep."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    st = build_stack(dev, args.layers)
    peak, peak_kind = peaks()
    rates = measure_issue_rates(dev)
    sus = sustained_pass(st, 0, stream, st.fused_bytes(), peak, seconds=2.0)
    r = gpu_config3(st.planes, st.specs, dev, stream, peak, sus["clocks"]["sm_mhz"], rates)
    top = max(r["by_M"])
    print(json.dumps({"metric": "batched ternary decode over the 30-layer stack", "unit": "tok/s",
                      "value": r["by_M"][top]["tok_per_s"],
                      "config": {"workload": "bitnet-2b4t-30layer-batch-sweep"},
                      "clocks": sus["clocks"], "issue_rates": rates, "detail": r}), flush=True)


MMA_CYCLES_M128 = 101.4   # tcgen05.mma cta_group::1 kind::f16, M = 128, N <= 128: measured back to back

# ---- issue rates (trit_issue_probe) -------------------------------------------

ISSUE_KINDS = ("dp4a", "dp4a.su", "lop3", "prmt", "shf", "imad", "iadd", "shfl", "lds32",
               "lds128", "dp4a+lop3")


def issue_rates(rec, threads: int, iters: int, per_iter: int = 32) -> dict:
    """Per-SM completion rates from a trit_issue_probe record ([CTAs, 3] of SM
    id, start clock, end clock): for every SM, the instructions its CTAs issued
    (32 * iters per thread) over the span from the earliest start to the latest
    end (SM clocks).  Returns lanes (thread-instructions) per SM-clock: the
    median over SMs, and the lowest and highest."""
    per_sm = {}
    for smid, t0, t1 in rec:
        n, lo, hi = per_sm.get(int(smid), (0, None, None))
        lo = int(t0) if lo is None else min(lo, int(t0))
        hi = int(t1) if hi is None else max(hi, int(t1))
        per_sm[int(smid)] = (n + 1, lo, hi)
    rates = sorted(n * threads * per_iter * iters / max(hi - lo, 1) for n, lo, hi in per_sm.values())
    return {"lanes_per_clk": round(statistics.median(rates), 2), "min": round(rates[0], 2),
            "max": round(rates[-1], 2), "sms": len(rates)}


def measure_issue_rates(dev, iters: int = 2048, threads: int = 256, ctas_per_sm: int = 4) -> dict:
    """Every probe kind at ctas_per_sm x threads per SM (32 warps), each thread
    issuing 32 * iters instructions in eight chains."""
    import torch

    import bit_plane_select_gb300 as t
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {}
    for kind in ISSUE_KINDS:
        t.trit_issue_probe(kind, sms * ctas_per_sm, threads, 16, dev)      # warm the kernel
        rec = t.trit_issue_probe(kind, sms * ctas_per_sm, threads, iters, dev)
        torch.cuda.synchronize(dev)
        r = issue_rates(rec.cpu().numpy(), threads, iters, 64 if kind == "dp4a+lop3" else 32)
        if kind == "lds32":
            r["bytes_per_clk"] = round(4 * r["lanes_per_clk"], 1)
        if kind == "lds128":
            r["bytes_per_clk"] = round(16 * r["lanes_per_clk"], 1)
        out[kind] = r
    return out


def run_issue(args):
    """The integer and shared-memory issue rates the decode kernels are built
    from, in lanes per SM-clock (clock64 spans, so independent of the clock)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    with ClockSampler(0) as clk:
        rates = measure_issue_rates(dev)
    print(json.dumps({"metric": "issue rates, lanes per SM-clock", "unit": "lanes/clk/SM",
                      "value": rates["dp4a"]["lanes_per_clk"], "by_kind": rates,
                      "config": {"workload": "trit_issue_probe, 4 CTAs x 256 threads per SM, "
                                             "8 chains per thread"},
                      "clocks": clk.summary()}), flush=True)


# Per (weight row, beat) instruction counts of the dp4a path for a chunk of mt
# staged activation rows, as the kernel is built: the code words (10 logic),
# the P1 check (3) and the masks into weight classes (16 / 20 / 28 logic for
# 4 / 2 / 1 classes: classes 4, 2, 2 at 2, 4, 8 staged rows), 16 dp4a per
# activation row, and the staged activations read from shared memory -- 64
# bytes per activation row and beat, shared by the lane's two weight rows.
DP4A_LOGIC = {2: 10 + 3 + 16, 4: 10 + 3 + 20, 8: 10 + 3 + 20}
DP4A_ROWS_PER_LANE = 2


def batch_floors(M: int, shapes, nbytes: int, peak_gbs: float, sm_count: int, sm_mhz,
                 rates: dict | None = None) -> dict:
    """Lower bounds on one batched step over `shapes` ((N, K) per product) with
    M activation rows, for the path the library takes at that M:
      hbm: the step's algorithmic bytes at the measured copy peak;
      dp4a path (2 <= M <= 12): rows in chunks of 8, the remainder staged as 2,
        4 or 8 rows; per weight row-beat and chunk of mt staged rows: 16 mt dp4a
        (the dp4a pipe), DP4A_LOGIC[mt] logic instructions (the logic pipe),
        64 mt / DP4A_ROWS_PER_LANE bytes of staged activations (shared memory),
        16 mt + DP4A_LOGIC[mt] + 2 mt instructions issued; each at the rate
        `rates` gives (trit_issue_probe, lanes per SM-clock), the bound being
        the largest;
      tensor path (13 <= M <= 128): four M = 128 MMAs per 128 weight rows and
        beat at MMA_CYCLES_M128 each, one MMA stream per SM.
    With no sampled clock (sm_mhz None) the compute floors are None."""
    rates = rates or {}
    dp4a = rates.get("dp4a", {}).get("lanes_per_clk", 64.0)
    lop = rates.get("lop3", {}).get("lanes_per_clk", 64.0)
    lds = rates.get("lds128", {}).get("bytes_per_clk", 128.0)
    out = {"hbm_floor_ms": nbytes / (peak_gbs * 1e9) * 1e3}
    row_beats = sum(N * ((K + 63) // 64) for N, K in shapes)
    other = 0.0
    if 2 <= M <= 12:
        r = M % 8
        chunks = [8] * (M // 8) + ([] if r == 0 else [2 if r <= 2 else 4 if r <= 4 else 8])
        out["path"] = "dp4a"
        out["chunks"] = chunks
        if sm_mhz:
            f = sm_mhz * 1e6 * sm_count
            per = {"dp4a": sum(16 * mt for mt in chunks) / dp4a,
                   "logic": sum(DP4A_LOGIC[mt] for mt in chunks) / lop,
                   "shared": sum(64 * mt / DP4A_ROWS_PER_LANE for mt in chunks) / lds,
                   "issue": sum(16 * mt + DP4A_LOGIC[mt] + 2 * mt for mt in chunks) / 128.0}
            out["alu_floors_ms"] = {k: row_beats * v / f * 1e3 for k, v in per.items()}
            out["alu_floor_ms"] = max(out["alu_floors_ms"].values())
            other = out["alu_floor_ms"]
    elif 13 <= M <= 128:
        tiles = sum(((N + 127) // 128) * ((K + 63) // 64) for N, K in shapes)
        out["path"] = "tensor (weights as the 128-row operand)"
        if sm_mhz:
            out["mma_floor_ms"] = tiles * 4 * MMA_CYCLES_M128 / (sm_count * sm_mhz * 1e6) * 1e3
            other = out["mma_floor_ms"]
    else:
        out["path"] = "dp4a (M = 1)" if M == 1 else "tensor (pair tiles)"
    out["bound"] = "hbm" if out["hbm_floor_ms"] >= other else ("alu" if M <= 12 else "mma")
    out["floor_ms"] = max(out["hbm_floor_ms"], other)
    return out


def gpu_config3(planes, specs, dev, stream, peak: float, sm_mhz, rates, steps: int = 60):
    """Config 3: batched decode over the given 30-layer planes (the config-2
    stack) at every M of the sweep -- M seeded activation rows per projection
    (seed 3), quantised outside the timed region -- then the same products on a
    copy of the planes with 0.1% of the beats given both bits at one position:
    the flag must be raised and every row without such a beat must equal the
    clean planes' output."""
    import torch

    import bit_plane_select_gb300 as t
    import synth
    Mmax = max(synth.BATCH_SWEEP)
    items = list(synth.stack_items(len(specs) // len(synth.PROJECTIONS)))
    xs, qs, ss, ys, fs = [], [], [], [], []
    for (layer, idx, name, N, K) in items:
        xs.append(torch.from_numpy(synth.projection_acts(3, layer, idx, Mmax)).to(dev))
        qs.append(torch.empty((Mmax, t.k_pad(K)), dtype=torch.int8, device=dev))
        ss.append(torch.empty(Mmax, dtype=torch.float32, device=dev))
        ys.append(torch.empty((Mmax, N), dtype=torch.int32, device=dev))
        fs.append(torch.empty((Mmax, N), dtype=torch.float32, device=dev))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    t.trit_quant_act_many(t.ActList(list(zip(xs, qs, ss))), err)
    shapes = [(N, K) for _, N, K, _, _ in specs]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def plist(M, pl):
        return t.ProjList([(pl[i], specs[i][4], qs[i][:M], ss[i][:M], specs[i][2], ys[i][:M], fs[i][:M])
                           for i in range(len(specs))])

    by_m = {}
    for M in synth.BATCH_SWEEP:
        pm = plist(M, planes)
        for _ in range(3):
            t.trit_gemm_many(pm, err)
        n = max(5, steps // M)
        ms = _events_ms(lambda i: t.trit_gemm_many(pm, err), n, stream) / n
        nbytes = sum(t.payload_bytes(N, K) + M * (t.k_pad(K) + 4 + 8 * N) for N, K in shapes)
        fl = batch_floors(M, shapes, nbytes, peak, sms, sm_mhz, rates)
        comp = fl.get("alu_floor_ms", fl.get("mma_floor_ms"))
        by_m[M] = {"us_per_step": round(ms * 1e3, 2), "tok_per_s": round(M / (ms * 1e-3), 1),
                   "GBs": round(nbytes / (ms * 1e-3) / 1e9, 1), "path": fl["path"], "bound": fl["bound"],
                   "hbm_floor_us": round(fl["hbm_floor_ms"] * 1e3, 2),
                   "compute_floor_us": round(comp * 1e3, 2) if comp else None,
                   "frac_of_floor": round(fl["floor_ms"] / ms, 4), "err_flag": int(err.item())}
        if "alu_floors_ms" in fl:
            by_m[M]["alu_floors_us"] = {k: round(v * 1e3, 2) for k, v in fl["alu_floors_ms"].items()}
    # corruption run
    clean = {}
    for M in (1, 4, 32):
        t.trit_gemm_many(plist(M, planes), err)
        torch.cuda.synchronize()
        clean[M] = [y[:M].clone() for y in ys]
    bad_planes, bad_rows = [], []
    for i, (layer, idx, name, N, K) in enumerate(items):
        B = (K + 63) // 64
        beats, bits = synth.corrupt_positions(3, layer, idx, N * B)
        pl = planes[i].clone().view(-1, 16)
        b_t = torch.from_numpy(beats).to(dev)
        for plane in (0, 1):
            byte = torch.from_numpy(plane * 8 + bits // 8).to(dev)
            val = torch.from_numpy((1 << (bits % 8)).astype("uint8")).to(dev)
            pl[b_t, byte] |= val
        bad_planes.append(pl.view_as(planes[i]))
        bad_rows.append(torch.from_numpy(beats // B).to(dev))
    corrupt = {}
    for M in (1, 4, 32):
        e2 = torch.zeros(1, dtype=torch.int32, device=dev)
        t.trit_gemm_many(plist(M, bad_planes), e2)
        torch.cuda.synchronize()
        same = True
        for i in range(len(specs)):
            keep = torch.ones(specs[i][1], dtype=torch.bool, device=dev)
            keep[bad_rows[i]] = False
            same &= bool(torch.equal(ys[i][:M][:, keep], clean[M][i][:, keep]))
        corrupt[M] = {"flag": int(e2.item()), "flag_p1_raised": bool(int(e2.item()) & t.ERR_P1),
                      "other_rows_identical": same}
    del bad_planes
    torch.cuda.empty_cache()
    return {"workload": "batched decode M in {1,2,4,8,16,32,64} over the config-2 30-layer planes",
            "activations": "seeded N(0,1) / relu(z)^2 rows (seed 3), quantised before timing",
            "by_M": by_m, "corruption_0.1pct": corrupt,
            "floors_from": {"issue_rates": "trit_issue_probe in this run" if rates else "assumed",
                            "sm_mhz": sm_mhz, "mma_cycles_m128": MMA_CYCLES_M128}}


def gpu_config4(dev, stream, layers: int, steps: int, warmup: int):
    """Config 4: prefill GEMMs -- M tokens through gate/up/down of `layers`
    layers (distinct weights, P(0) = 0.4219): fp32 activations quantised, then
    one trit_gemm_many over the products (tensor-core path), per M."""
    import torch

    import bit_plane_select_gb300 as t
    import synth
    items = list(synth.prefill_items(layers))
    planes, wss = [], []
    for layer, idx, name, N, K in items:
        w = synth.projection_weights(4, layer, idx)
        ws = float(synth.w_scale(w))
        pl, _ = t.trit_pack(torch.from_numpy(w).to(dev), ws)
        planes.append(pl)
        wss.append(ws)
    Mmax = max(synth.PREFILL_M)
    xs = [torch.from_numpy(synth.projection_acts(4, layer, idx, Mmax)).to(dev)
          for layer, idx, name, N, K in items]
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        burst, sustained, kind = float(pk["bf16_tflops"]), float(pk["bf16_tflops_sustained"]), "measured"
    except Exception:
        burst, sustained, kind = 1900.0, 1700.0, "fallback"
    results = {}
    for M in synth.PREFILL_M:
        acts, projs, keep = [], [], []
        for i, (layer, idx, name, N, K) in enumerate(items):
            x = xs[i][:M].contiguous()
            q = torch.empty((M, t.k_pad(K)), dtype=torch.int8, device=dev)
            sc = torch.empty(M, dtype=torch.float32, device=dev)
            y = torch.empty((M, N), dtype=torch.int32, device=dev)
            fo = torch.empty((M, N), dtype=torch.float32, device=dev)
            acts.append((x, q, sc))
            projs.append((planes[i], wss[i], q, sc, K, y, fo))
            keep.append((x, q, sc, y, fo))
        alist, plist = t.ActList(acts), t.ProjList(projs)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        flops = sum(2 * M * N * K for _, _, _, N, K in items)
        ms_q = _timed(lambda: t.trit_quant_act_many(alist, err), steps, warmup, stream)
        # at least `steps`, and about a second of back-to-back GEMM lists so that
        # nvidia-smi (200 ms period) samples the clocks under this load
        ms_est = _timed(lambda: t.trit_gemm_many(plist, err), 3, warmup, stream)
        n = max(steps, int(1.0 / (ms_est * 1e-3)))
        with ClockSampler(dev.index or 0, wait_first=3.0) as clk:
            ms_g = _timed(lambda: t.trit_gemm_many(plist, err), n, 1, stream)
        tf = flops / (ms_g * 1e-3) / 1e12
        results[M] = {"gemm_ms": round(ms_g, 4), "quant_ms": round(ms_q, 4), "tflops": round(tf, 1),
                      "frac_of_sustained_peak": round(tf / sustained, 4),
                      "frac_of_burst_peak": round(tf / burst, 4),
                      "tok_per_s": round(M / ((ms_g + ms_q) * 1e-3), 1), "err_flag": int(err.item()),
                      "steps": n, "clocks": clk.summary()}
        del alist, plist, keep, acts, projs
        torch.cuda.empty_cache()
    del xs, planes
    torch.cuda.empty_cache()
    return {"workload": f"prefill gate/up/down x {layers} layers ({len(items)} GEMMs), tensor cores",
            "peak_tflops": {"bf16_sustained": sustained, "bf16_burst": burst, "kind": kind,
                            "note": "kind::f16 (the exact fp16 path used) has the bf16 nominal rate"},
            "by_M": results}


def run_bitcos(args):
    """Row f4: the 30-layer stack at batch 1 with the weights in the BITCOS
    form (presence bitmap + compacted signs, 2 - z bits per weight) against the
    same weights as 2-bit planes, both from int8 activation codes, in one run.
    A step is one token through the 210 products."""
    import numpy as np
    import torch

    import __graft_entry__
    import synth
    import bit_plane_select_gb300 as t
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    items = list(synth.stack_items(args.layers))
    bents, pents, keep = [], [], []
    bytes_bitcos = bytes_planes = nnz = weights = 0
    for layer, idx, name, N, K in items:
        w = synth.stack_weights(SEED, layer, idx)
        ws = float(synth.w_scale(w))
        W = t.BitcosWeights(*t.trit_bitcos_pack(w), K, dev)
        planes, _ = t.trit_pack(torch.from_numpy(w).to(dev), ws)
        x = torch.from_numpy(synth.projection_acts(SEED, layer, idx, 1)).to(dev)
        q, sc, _ = t.trit_quant_act(x)
        y = torch.empty(N, dtype=torch.int32, device=dev)
        f = torch.empty(N, dtype=torch.float32, device=dev)
        y2 = torch.empty((1, N), dtype=torch.int32, device=dev)
        f2 = torch.empty((1, N), dtype=torch.float32, device=dev)
        bents.append((W, ws, q[0], sc, y, f))
        pents.append((planes, ws, q, sc, K, y2, f2))
        keep.append((W, planes, q, sc, y, f, y2, f2))
        kp = t.k_pad(K)
        bytes_bitcos += W.nbytes + kp + 4 + 8 * N
        bytes_planes += planes.numel() + kp + 4 + 8 * N
        nnz += int(np.count_nonzero(w))
        weights += N * K
    blist, plist = t.BitcosList(bents), t.ProjList(pents)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    steps = max(3, args.steps // 10)
    with ClockSampler(0) as clk:
        ms_b = _timed(lambda: t.trit_bitcos_gemv_many(blist), steps, args.warmup, stream)
    clocks = clk.summary()
    ms_p = _timed(lambda: t.trit_gemm_many(plist, err), steps, args.warmup, stream)
    same = all(torch.equal(k[4], k[6][0]) and torch.equal(k[5].view(torch.int32), k[7][0].view(torch.int32))
               for k in keep)
    peak, peak_kind = peaks()
    gbs = bytes_bitcos / (ms_b * 1e-3) / 1e9
    print(json.dumps({
        "metric": "BITCOS batch-1 ternary decode over the 30-layer stack",
        "unit": "tok/s", "value": round(1e3 / ms_b, 1), "ms_per_step": round(ms_b, 4),
        "higher_is_better": True, "dtype": "int8", "data": "synthetic",
        "config": {"workload": "bitnet-2b4t-30layer-bitcos-batch1", "layers": args.layers,
                   "zero_density": round(1 - nnz / weights, 4),
                   "bits_per_weight": round(8 * bytes_bitcos / weights, 4),
                   "l2": "inputs larger than L2"},
        "planes_same_run": {"ms_per_step": round(ms_p, 4), "tok_per_s": round(1e3 / ms_p, 1),
                            "bytes_per_step": bytes_planes},
        "speedup_vs_planes": round(ms_p / ms_b, 3),
        "identical_to_planes": bool(same),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                     "bytes_per_step": bytes_bitcos},
        "clocks": clocks, "err_flag": int(err.item())}), flush=True)


def run_mlp(args):
    """The MLP blocks of the 30-layer stack at batch 1 (row f1), one token
    through every layer, three ways with the same bits: "paired" -- gate and
    up in one launch that also publishes the max|t| partials, then the down
    product forming the IntMlp codes from them (trit_mlp_gate_up,
    trit_mlp_down: two launches per layer); "fused" -- gate/up, then every CTA
    of the down launch forming the codes with its own max|t| pass (two); and
    "three_launch" -- gate/up, the standalone IntMlp quantiser, the down product
    of its int8 codes.  Beside them the same 90 products with no dependency:
    all gate/up in one launch, all down products (int8 codes) in another."""
    import torch

    import __graft_entry__
    import synth
    import bit_plane_select_gb300 as t
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    names = [p[0] for p in synth.PROJECTIONS]
    ig, iu, idn = names.index("gate"), names.index("up"), names.index("down")
    K, N = synth.PROJECTIONS[ig][2], synth.PROJECTIONS[ig][1]      # 2560, 6912
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    paired, fused, three, keep, block_entries = [], [], [], [], []
    indep_gu, indep_dn = [], []
    plane_bytes = 0
    for layer in range(args.layers):
        pl, ws = [], []
        for idx in (ig, iu, idn):
            w = synth.stack_weights(SEED, layer, idx)
            ws.append(float(synth.w_scale(w)))
            pl.append(t.trit_pack(torch.from_numpy(w).to(dev), ws[-1])[0])
            plane_bytes += pl[-1].numel()
        x = torch.from_numpy(synth.projection_acts(SEED, layer, ig, 1)).to(dev).reshape(-1)
        a_g = torch.empty(N, dtype=torch.int32, device=dev)
        a_u = torch.empty(N, dtype=torch.int32, device=dev)
        xs = torch.empty(1, dtype=torch.float32, device=dev)
        h = torch.empty(t.k_pad(N), dtype=torch.int8, device=dev)
        hs = torch.empty(1, dtype=torch.float32, device=dev)
        y = torch.empty(K, dtype=torch.int32, device=dev)
        yf = torch.empty(K, dtype=torch.float32, device=dev)
        tmax = torch.empty(t.trit_mlp_tmax_bytes(N), dtype=torch.uint8, device=dev)
        gu_e = [(pl[0], ws[0], x, None, xs, a_g, None), (pl[1], ws[1], x, None, None, a_u, None)]
        gu = t.QProjList(gu_e, planes_ready=True)
        dn = t.MlpProjList([(pl[2], ws[2], a_g, a_u, xs, ws[0], ws[1], None, None, y, yf)])
        dn3_e = [(pl[2], ws[2], h, hs, N, y, yf)]
        dn3 = t.ProjList(dn3_e, planes_ready=True)
        blk = (pl[0], pl[1], pl[2], ws[0], ws[1], ws[2], x, xs, a_g, a_u, tmax, None, None, y, yf)
        paired.append(t.MlpBlockList([blk], planes_ready=True))
        block_entries.append(blk)
        fused.append((gu, dn))
        three.append((gu, a_g, a_u, ws[0], ws[1], xs, h, hs, dn3))
        indep_gu += gu_e
        indep_dn += dn3_e
        keep.append((pl, x, a_g, a_u, xs, h, hs, y, yf, tmax))
    torch.cuda.synchronize(dev)   # the planes are complete before any launch below
    indep = (t.QProjList(indep_gu, planes_ready=True), t.ProjList(indep_dn, planes_ready=True))
    all_blocks = t.MlpBlockList(block_entries, planes_ready=True)

    def step_paired():
        for bl in paired:
            t.trit_mlp_gate_up(bl, err)
            t.trit_mlp_down(bl, err)

    def step_fused():
        for gu, dn in fused:
            t.trit_quant_gemv_many(gu, err)
            t.trit_intmlp_gemv_many(dn, err)

    def step_three():
        for gu, a_g, a_u, wg, wu, xs, h, hs, dn3 in three:
            t.trit_quant_gemv_many(gu, err)
            t.trit_intmlp_quant(a_g, a_u, wg, wu, xs, h, hs)
            t.trit_gemm_many(dn3, err)

    def step_indep():
        t.trit_quant_gemv_many(indep[0], err)
        t.trit_gemm_many(indep[1], err)

    def step_batched():   # the 30 independent blocks in one call each (8 blocks per launch)
        t.trit_mlp_gate_up(all_blocks, err)
        t.trit_mlp_down(all_blocks, err)

    steps = max(20, args.steps // 100)
    eager = {name: _timed(fn, steps, args.warmup, stream)
             for name, fn in (("paired", step_paired), ("fused", step_fused),
                              ("three_launch", step_three))}

    # the launches of one step captured in a CUDA graph: replay time is device
    # time, free of the per-call host work of the eager loop above
    def graph_ms(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return _timed(g.replay, steps, args.warmup, stream)

    ms = {"paired": graph_ms(step_paired), "fused": graph_ms(step_fused),
          "three_launch": graph_ms(step_three)}
    ms_i = graph_ms(step_indep)
    ms_b = graph_ms(step_batched)
    launches = {"paired": 2, "fused": 2, "three_launch": 3}
    act_bytes = args.layers * (K * 4 + 4 + 2 * N * 4 * 2 + K * 8)
    nbytes = plane_bytes + act_bytes
    ms_p = ms["paired"]
    out = {"metric": "MLP blocks of the 30-layer stack, batch 1 (gate+up with max|t| partials; "
                     "IntMlp codes + down)",
           "unit": "tok/s", "value": round(1e3 / ms_p, 1),
           "ms_per_step": round(ms_p, 4), "GBs": round(nbytes / (ms_p * 1e-3) / 1e9, 1),
           "launches_per_step": 2 * args.layers, "timing": "CUDA graph of one step, replayed",
           "forms": {k: {"ms_per_step": round(v, 4), "tok_per_s": round(1e3 / v, 1),
                         "launches_per_step": launches[k] * args.layers,
                         "eager_ms_per_step": round(eager[k], 4)} for k, v in ms.items()},
           "independent_products": {"ms_per_step": round(ms_i, 4), "launches_per_step": 2,
                                    "what": "the same 60 gate/up and 30 down products with no "
                                            "dependency between them: two launches"},
           "chain_over_independent": round(ms_p / ms_i, 2),
           "blocks_batched": {"ms_per_step": round(ms_b, 4), "tok_per_s": round(1e3 / ms_b, 1),
                              "launches_per_step": 2 * ((args.layers + 7) // 8),
                              "over_independent": round(ms_b / ms_i, 2),
                              "what": "the blocks are independent of one another in this "
                                      "workload: trit_mlp_gate_up and trit_mlp_down over all of "
                                      "them (up to 8 per launch), every block's gate/up -> down "
                                      "dependency kept"},
           "algorithmic_bytes_per_step": nbytes, "err_flag": int(err.item()),
           "config": {"workload": "bitnet-2b4t-30layer-mlp-batch1", "layers": args.layers,
                      "gate_up": [N, K], "down": [K, N]}}
    print(json.dumps(out), flush=True)


def decode_ordered(dev, stream, layers, steps, warmup, forms=None):
    """The dependency-ordered decode of one token over the stack: per layer
    qkv -> o -> gate/up -> IntMlp + down, each launch reading what the one
    before it wrote (the per-matvec ordering of "Tritium ..." -- Why it does not
    scale), timed as a CUDA graph of one token replayed, for each MLP form."""
    import torch

    import synth
    from bit_plane_select_gb300.stack import LayerChain
    names = [p[0] for p in synth.PROJECTIONS]
    weights = []
    for layer in range(layers):
        lw = {}
        for i, n in enumerate(names):
            w = synth.stack_weights(SEED, layer, i)
            lw[n] = (torch.from_numpy(w), float(synth.w_scale(w)))
        weights.append(lw)
    chain = LayerChain(weights, dev)
    for layer in range(layers):
        chain.x[layer].copy_(torch.from_numpy(synth.projection_acts(SEED, layer, 0, 1)[0]))
    del weights
    out = {}
    for form in forms or LayerChain.MLP_FORMS:
        chain.mlp_form = form
        for _ in range(3):
            chain.step()
        torch.cuda.synchronize()
        # the launches of one token captured in a CUDA graph and replayed
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chain.step()
        ms = _timed(g.replay, steps, warmup, stream)
        eager = _timed(chain.step, max(20, steps // 10), warmup, stream)
        out[form] = {"us_per_token": round(ms * 1e3, 2), "tok_per_s": round(1e3 / ms, 1),
                     "launches_per_token": chain.launches_per_step,
                     "us_per_launch": round(ms * 1e3 / chain.launches_per_step, 3),
                     "eager_us_per_token": round(eager * 1e3, 2)}
        del g
    return out, chain.step_bytes(), int(chain.err.item())


def run_decode_ordered(args):
    """The dependency-ordered decode of one token over the 30-layer stack in
    its three MLP forms (paired: gate/up publishing max|t| partials, then the
    down product forming the IntMlp codes from them, 4 launches per layer;
    split: a quantiser launch between, 5; fused: max|t| in every down CTA, 4)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    steps = max(50, min(args.steps, 2000))
    with ClockSampler(0) as clk:
        forms, nbytes, err = decode_ordered(dev, stream, args.layers, steps, args.warmup)
    best = min(forms, key=lambda k: forms[k]["us_per_token"])
    ms = forms[best]["us_per_token"] * 1e-3
    peak, peak_kind = peaks()
    out = {"metric": "dependency-ordered batch-1 decode over the 30-layer stack", "unit": "tok/s",
           "value": round(1e3 / ms, 1), "us_per_token": round(ms * 1e3, 2),
           "GBs": round(nbytes / (ms * 1e-3) / 1e9, 1),
           "frac_of_hbm_peak": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4), "peak": peak,
           "peak_kind": peak_kind, "mlp_form": best, "forms": forms,
           "launches_per_token": forms[best]["launches_per_token"],
           "us_per_launch": forms[best]["us_per_launch"],
           "algorithmic_bytes_per_token": nbytes,
           "timing": f"CUDA graph of one token replayed {steps} times", "err_flag": err,
           "clocks": clk.summary(),
           "config": {"workload": "bitnet-2b4t-30layer-decode-ordered-batch1", "layers": args.layers,
                      "order": "per layer: [q,k,v] <- x; [o] <- q; [gate,up] <- o; IntMlp + [down] "
                               "<- gate,up (paired: max|t| partials from the gate/up launch; split: "
                               "a quantiser launch between; fused: max|t| in every down CTA)"}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=30)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--two-launch-steps", type=int, default=500)
    ap.add_argument("--cpu-layers", type=int, default=30)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip configs 0, 1, 3 and 4 in the default run")
    ap.add_argument("--reference-budget", type=float, default=90.0)
    ap.add_argument("--workload", choices=["decode", "prefill", "batch", "mlp", "bitcos", "issue",
                                           "decode-ordered"],
                    default="decode",
                    help="decode (default): the 30-layer batch-1 stack; prefill, batch, mlp and "
                         "bitcos print extra lines for the other configurations")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "prefill":
        run_prefill(args)
    elif args.workload == "batch":
        run_batch_sweep(args)
    elif args.workload == "mlp":
        run_mlp(args)
    elif args.workload == "bitcos":
        run_bitcos(args)
    elif args.workload == "issue":
        run_issue(args)
    elif args.workload == "decode-ordered":
        run_decode_ordered(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
