#!/usr/bin/env python3
"""Benchmark of the MoE expert layer on GB300 (one JSON line on rank 0).

A step is one pass of the whole layer (route -> grouped gate/up GEMM with
SiLU*up -> grouped down GEMM -> combine) over one batch of the pages-shaped
workload (T=2048 tokens, H=4096, I=1536, E=64 experts, top-8), synthetic
inputs already resident in HBM, timed as K replays of one moe_forward (the
library's one-call layer) recorded into a CUDA graph, between two CUDA
events (direct calls if capture is refused).  The metric is useful
bf16 TFLOP/s (6*T*k*H*I FLOPs per step) with microseconds per layer beside
it; a second pass through the four step calls, with events between them,
gives the per-step breakdown and the up call's roofline, and an end-to-end
loop calls moe_forward on inputs copied in from host memory (and its output
copied back) every step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the slow, plain C implementation the
tests check against) on a bounded sample of the same workload.  Under
torchrun every rank runs an independent replica (the layer does not shard
across GPUs here); rank 0 prints the aggregate.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer µs and bf16 TFLOP/s on 1 GB300; % of tensor peak / HBM roofline"
UNIT = "TFLOP/s"
WORKLOAD = 2
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def kernel_source_hash() -> str:
    """Hash of the GEMM kernel's code (comments and blank lines left out, so
    that an edit of comments alone keeps the recorded counters valid)."""
    h = hashlib.sha256()
    for n in ("moe_gemm.cu", "moe_device.cuh"):
        with open(os.path.join(ROOT, "combine_moe_route_04_gb300", "csrc", n), encoding="utf-8") as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode("utf-8") + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, watts = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            try:
                watts.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w": statistics.median(watts) if watts else None}


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def layer_flops(cfg) -> float:
    return 6.0 * cfg.T * cfg.k * cfg.H * cfg.I


def max_over_ranks(values, device=None):
    """Each value's maximum over the ranks of the default process group (the
    slowest replica sets the step time); the values unchanged on one rank."""
    import torch
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def aggregate_tflops(world: int, flops_per_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs its own replica of the layer, so
    N ranks do N layers' work in the slowest rank's step time."""
    return world * flops_per_step / (ms_per_step * 1e-3) / 1e12


def layer_bytes(cfg, touched: int, r_pad: int) -> dict:
    """Algorithmic bytes of each step of one layer: what the method must move
    (useful rows only; every touched expert's weights once)."""
    T, H, I, E, k = cfg.shape
    R = T * k
    return {"route": T * E * 4 + 12 * T * k + 4 * r_pad,
            "up": touched * 2 * H * I * 2 + T * H * 2 + R * I * 2,
            "down": touched * I * H * 2 + R * I * 2 + R * H * 2,
            "combine": R * H * 2 + 8 * T * k + T * H * 2}


def layer_roofline(cfg, touched: int, r_pad: int, ms_step: float, pk: dict, pk_src: str) -> dict:
    """The layer's roofline: the slower of its useful FLOPs at the measured
    sustained bf16 rate and its algorithmic bytes at the measured copy
    bandwidth; frac = that floor / the measured time per layer."""
    b = layer_bytes(cfg, touched, r_pad)
    total_b = float(sum(b.values()))
    flops = layer_flops(cfg)
    t_hbm = total_b / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops_sustained"] * 1e12)
    t = ms_step * 1e-3
    if t_hbm >= t_tc:
        bound, achieved, peak, unit = "hbm", total_b / t / 1e9, pk["hbm_gbs"], "GB/s"
        src = "%s hbm_gbs" % pk_src
    else:
        bound, achieved, peak, unit = "tensor", flops / t / 1e12, pk["bf16_tflops_sustained"], "TFLOP/s"
        src = "%s bf16_tflops_sustained" % pk_src
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": max(t_hbm, t_tc) / t,
            "peak_source": src, "floor_us": max(t_hbm, t_tc) * 1e6, "hbm_floor_us": t_hbm * 1e6,
            "tensor_floor_us": t_tc * 1e6, "algorithmic_bytes": total_b, "bytes_by_step": b,
            "useful_flops": flops, "us_per_layer": ms_step * 1e3}


def cpu_oracle_sample(cfg, inp, seconds=15.0, max_tokens=256):
    """Times the oracle on the host cores on a bounded sample of the workload:
    routing for all tokens, then tokens' outputs one by one until ~`seconds`.
    Returns (TFLOP/s, description, cores)."""
    import numpy as np
    import oracle
    oracle.build_oracle()
    cores = oracle.num_threads()
    t0 = time.perf_counter()
    r = oracle.route(inp["logits"], cfg.k)
    t_route = time.perf_counter() - t0
    toks_done = 0
    t_tok = 0.0
    batch = max(1, min(16, cores))
    while t_tok < seconds and toks_done < max_tokens:
        toks = np.arange(toks_done, toks_done + batch, dtype=np.int32) % cfg.T
        t1 = time.perf_counter()
        oracle.tokens_out(toks, r.topk_ids, r.topk_w, inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"])
        t_tok += time.perf_counter() - t1
        toks_done += batch
    per_tok = t_tok / toks_done
    est_layer_s = t_route + per_tok * cfg.T
    tflops = layer_flops(cfg) / est_layer_s / 1e12
    desc = ("oracle route over all %d tokens (%.2f s) + %d tokens' outputs (%.1f s, %.3f s/token), "
            "scaled to the %d-token layer" % (cfg.T, t_route, toks_done, t_tok, per_tok, cfg.T))
    return tflops, desc, cores, est_layer_s


def reference_step(cfg, inp, pool, cores, step):
    """One bounded sample of the oracle on the host cores: routing over all
    tokens, then one (token, slot) row of the expert MLP per core, in parallel
    (the oracle's row functions).  Returns the layer time this implies (s)."""
    import numpy as np
    import oracle
    t0 = time.perf_counter()
    r = oracle.route(inp["logits"], cfg.k)
    t_route = time.perf_counter() - t0
    rows = [((step * cores + i) * 7919 % cfg.T, (step * cores + i) % cfg.k) for i in range(cores)]

    def one(tj):
        t, j = tj
        e = int(r.topk_ids[t, j])
        hrow = oracle.expert_up_row(inp["x"][t], inp["w_gate"][e], inp["w_up"][e])
        return oracle.expert_down_row(hrow, inp["w_down"][e])

    t1 = time.perf_counter()
    list(pool.map(one, rows))
    t_rows = time.perf_counter() - t1
    return t_route + t_rows * (cfg.T * cfg.k) / len(rows)


def run_reference(args, world, rank):
    """The oracle timed as it stands on the host cores, on the same workload
    and metric; each of the W + K steps is one bounded sample (a few tens of
    ms), so the run stays within minutes for the default K."""
    if rank != 0:
        return 0
    from concurrent.futures import ThreadPoolExecutor
    import moe_inputs
    import oracle
    oracle.build_oracle()
    cfg = moe_inputs.config(args.workload)
    inp = moe_inputs.make_inputs(cfg)
    cores = os.cpu_count() or 1
    est = []
    with ThreadPoolExecutor(max_workers=cores) as pool:
        for i in range(args.warmup + args.steps):
            v = reference_step(cfg, inp, pool, cores, i)
            if i >= args.warmup:
                est.append(v)
    layer_s = statistics.median(est)
    value = layer_flops(cfg) / layer_s / 1e12
    desc = ("per step: oracle routing over all %d tokens + %d (token, slot) rows of the expert MLP, one "
            "per host core, scaled to the layer's %d rows; median of %d steps"
            % (cfg.T, cores, cfg.T * cfg.k, args.steps))
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": layer_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": "%s (T=%d,H=%d,I=%d,E=%d,k=%d)" % ((cfg.name,) + cfg.shape)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc, "extrapolated": True},
            "extrapolated": True,
            "extrapolation": ("ms_per_step is an estimate of one whole layer on the host cores, scaled "
                              "from each step's sample; the run itself takes a few tens of ms per step"),
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local):
    workload = args.workload
    import numpy as np
    import torch

    import combine_moe_route_04_gb300 as moe
    import moe_inputs
    from combine_moe_route_04_gb300 import _build

    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local)
    if rank == 0:
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    moe.load()

    cfg = moe_inputs.config(workload)
    inp = moe_inputs.make_inputs(cfg)
    T, H, I, E, k = cfg.shape
    s = moe.shape(T, H, I, E, k)
    stream = torch.cuda.Stream(device=dev)

    def up_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    # Timed iterations must not find their inputs in L2.  Where one layer's
    # resident bytes (weights, X, logits, workspace, out) exceed twice the L2
    # size that holds by itself; below it, iteration i uses buffer set
    # i % n_sets, copies of the same values, so that the sets together span
    # at least twice the L2 size and each one is evicted before its reuse.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2**20)
    set_bytes = (3 * E * H * I * 2 + T * H * 2 + T * E * 4 + T * H * 2 + int(moe.workspace_size(s)))
    n_sets = 1 if set_bytes >= 2 * l2_bytes else min(64, -(-2 * l2_bytes // set_bytes))
    host = {n: up_bf16(inp[n]) for n in ("x", "w_gate", "w_up", "w_down")}
    host["logits"] = torch.from_numpy(inp["logits"]).to(dev)
    sets = []
    for j in range(n_sets):
        ws_j = moe.alloc_workspace(s, dev)
        sets.append({"logits": host["logits"] if j == 0 else host["logits"].clone(),
                     "x": host["x"] if j == 0 else host["x"].clone(),
                     "wg": host["w_gate"] if j == 0 else host["w_gate"].clone(),
                     "wu": host["w_up"] if j == 0 else host["w_up"].clone(),
                     "wd": host["w_down"] if j == 0 else host["w_down"].clone(),
                     "out": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
                     "ws": ws_j, "v": moe.workspace_views(s, ws_j)})
    del host
    logits, x, out, ws, v = (sets[0][n] for n in ("logits", "x", "out", "ws", "v"))
    mb, mr = moe.capacity(s)
    sh = stream.cuda_stream
    lib = moe.load()
    import ctypes
    sp = ctypes.byref(s)

    def step_by_step(ev=None, b=sets[0]):
        # the layer's five steps through the C ABI, with events between them
        bv, bws = b["v"], b["ws"].data_ptr()
        if ev is not None:
            ev[0].record(stream)
        rc = lib.moe_route(sp, b["logits"].data_ptr(), bv.topk_ids, bv.topk_w, bv.counts, bv.off_pad,
                           bv.block_expert, bv.num_blocks, bv.gather_idx, bv.scatter_idx, bws, sh)
        if ev is not None:
            ev[1].record(stream)
        rc |= lib.moe_grouped_gemm_up(sp, b["x"].data_ptr(), bv.scatter_idx, bv.counts, bv.off_pad,
                                      b["wg"].data_ptr(), b["wu"].data_ptr(), bv.h, bws, sh)
        if ev is not None:
            ev[2].record(stream)
        rc |= lib.moe_grouped_gemm_down(sp, bv.h, bv.counts, bv.off_pad, b["wd"].data_ptr(), bv.Y, bws, sh)
        if ev is not None:
            ev[3].record(stream)
        rc |= lib.moe_combine(sp, bv.Y, bv.scatter_idx, bv.topk_w, b["out"].data_ptr(), bws, sh)
        if ev is not None:
            ev[4].record(stream)
        if rc:
            raise RuntimeError("moe step failed: %d" % rc)

    def forward(b=sets[0]):
        rc = lib.moe_forward(sp, b["logits"].data_ptr(), b["x"].data_ptr(), b["wg"].data_ptr(),
                             b["wu"].data_ptr(), b["wd"].data_ptr(), b["out"].data_ptr(), b["ws"].data_ptr(), sh)
        if rc:
            raise RuntimeError("moe_forward failed: %d" % rc)

    def all_status_clean():
        return all(moe.last_device_status(b["ws"], sh) == 0 for b in sets)

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup, n_sets)):
            forward(sets[i % n_sets])
    torch.cuda.synchronize(dev)
    if not all_status_clean():
        raise RuntimeError("device status after warm-up")
    for b in sets[1:]:
        if not torch.equal(b["out"], out):
            raise RuntimeError("buffer sets disagree after warm-up")

    # The timed loop replays CUDA graphs of recorded moe_forward calls (the
    # same five kernels and dependent-launch edges, without the per-call host
    # work).  One graph holds a run of G consecutive forwards (G = n_sets when
    # the buffer sets rotate, else 10), as a model's layers sit back to back
    # in one graph: forward j+1's routing is a dependent launch of forward j's
    # combine, and the gap between two graph replays is paid once per G
    # layers.  Steps past the last whole run replay one-forward graphs, which
    # are also timed by themselves (graph_of_one_us).  If capture is refused
    # the loop calls moe_forward directly.
    G = n_sets if n_sets > 1 else 10
    launch = "cuda_graph"
    singles = [torch.cuda.CUDAGraph() for _ in sets]
    chain = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.stream(stream):
            for g, b in zip(singles, sets):
                with torch.cuda.graph(g, stream=stream):
                    forward(b)
            with torch.cuda.graph(chain, stream=stream):
                for j in range(G):
                    forward(sets[j % n_sets])
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            for g in singles:
                g.replay()
            chain.replay()
        torch.cuda.synchronize(dev)
        if not all_status_clean():
            raise RuntimeError("device status after a graph replay")
        for b in sets[1:]:
            if not torch.equal(b["out"], out):
                raise RuntimeError("buffer sets disagree after the graph replays")
    except Exception as exc:  # noqa: BLE001 -- any capture failure falls back to direct calls
        launch = "direct calls (graph capture failed: %s)" % str(exc).splitlines()[0][:120]
        singles = chain = None
        torch.cuda.synchronize(dev)

    def run_steps(n, chained=True):
        # n consecutive layers, layer i on buffer set i mod n_sets
        if singles is None:
            for i in range(n):
                forward(sets[i % n_sets])
            return
        q = n // G if chained else 0
        for _ in range(q):
            chain.replay()
        for i in range(q * G, n):
            singles[i % n_sets].replay()

    # ---------------- timed region: K layers as graph replays (above), events
    # on the launching stream around all K
    K = args.steps
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        run_steps(K)
        t_end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if rank == 0 else None
    total_ms = t_start.elapsed_time(t_end)
    if not all_status_clean():
        raise RuntimeError("device status after timed region")

    # ---------------- the same K layers, one graph replay per layer
    o0 = torch.cuda.Event(enable_timing=True)
    o1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        o0.record(stream)
        run_steps(K, chained=False)
        o1.record(stream)
    torch.cuda.synchronize(dev)
    one_ms = o0.elapsed_time(o1) / K
    if not all_status_clean():
        raise RuntimeError("device status after the one-forward graphs")

    # ---------------- breakdown: the same K layers as the four C-ABI steps
    # with an event between each (the events also cut the launch overlap
    # between the steps, so these sum to a little more than the layer)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    with torch.cuda.stream(stream):
        for i in range(K):
            step_by_step(evs[i], sets[i % n_sets])
    torch.cuda.synchronize(dev)
    parts = {"route": [], "up": [], "down": [], "combine": []}
    for e in evs:
        parts["route"].append(e[0].elapsed_time(e[1]))
        parts["up"].append(e[1].elapsed_time(e[2]))
        parts["down"].append(e[2].elapsed_time(e[3]))
        parts["combine"].append(e[3].elapsed_time(e[4]))
    if not all_status_clean():
        raise RuntimeError("device status after the breakdown")
    steps_ms = sum(e[0].elapsed_time(e[4]) for e in evs) / K

    # ---------------- the dominant kernel alone: the gate/up GEMM on the rows
    # the last step gathered (moe_grouped_gemm_up_rows), K launches between
    # events on the launching stream
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g0.record(stream)
        for i in range(K):
            b = sets[i % n_sets]
            bv = b["v"]
            if lib.moe_grouped_gemm_up_rows(sp, bv.Xp, bv.counts, bv.off_pad, b["wg"].data_ptr(),
                                            b["wu"].data_ptr(), bv.h, b["ws"].data_ptr(), sh):
                raise RuntimeError("moe_grouped_gemm_up_rows failed")
        g1.record(stream)
    torch.cuda.synchronize(dev)
    gemm_ms = g0.elapsed_time(g1) / K
    if not all_status_clean():
        raise RuntimeError("device status after the GEMM timing")

    # ---------------- end to end: host buffers, copies inside the timed region
    # Every step copies its inputs (logits, X) from pinned host memory and its
    # output back.  The copies run on a second stream, double-buffered, so
    # step i+1's inputs and step i-1's output move while step i computes.
    logits_h = torch.from_numpy(inp["logits"]).pin_memory()
    x_h = torch.from_numpy(np.ascontiguousarray(inp["x"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    out_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    logits_d = [torch.empty_like(logits) for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    out_d = [torch.empty_like(out) for _ in range(2)]
    cs_in = torch.cuda.Stream(device=dev)    # host -> device copies
    cs_out = torch.cuda.Stream(device=dev)   # device -> host copies (the link is full duplex)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of slot b copied in
    ev_done = [torch.cuda.Event() for _ in range(2)]   # forward of slot b finished
    ev_out = [torch.cuda.Event() for _ in range(2)]    # output of slot b copied out
    Ke = max(10, K)   # as many steps as the kernel-only loop: comparable time under the power cap
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_clocks = ClockSampler(local)
    if rank == 0:
        e2e_clocks.start()
    torch.cuda.synchronize(dev)
    e0.record(cs_in)
    cs_out.wait_event(e0)
    stream.wait_event(e0)
    for i in range(Ke):
        b = i & 1
        with torch.cuda.stream(cs_in):
            if i >= 2:
                cs_in.wait_event(ev_done[b])    # step i-2 no longer reads these inputs
            logits_d[b].copy_(logits_h, non_blocking=True)
            x_d[b].copy_(x_h, non_blocking=True)
            ev_in[b].record(cs_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])        # step i-2's output has been copied out
        w = sets[i % n_sets]
        moe.moe_forward_raw(s, logits_d[b].data_ptr(), x_d[b].data_ptr(), w["wg"].data_ptr(), w["wu"].data_ptr(),
                            w["wd"].data_ptr(), out_d[b].data_ptr(), w["ws"].data_ptr(), sh)
        ev_done[b].record(stream)
        with torch.cuda.stream(cs_out):
            cs_out.wait_event(ev_done[b])
            out_h[b].copy_(out_d[b], non_blocking=True)
            ev_out[b].record(cs_out)
    cs_in.wait_event(ev_out[(Ke - 1) & 1])
    cs_in.wait_event(ev_out[Ke & 1])
    e1.record(cs_in)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / Ke
    e2e_clk = e2e_clocks.stop() if rank == 0 else None
    if not torch.equal(out_h[(Ke - 1) & 1], out_d[(Ke - 1) & 1].cpu()):
        raise RuntimeError("end-to-end output copy mismatch")
    h2d = logits_h.numel() * 4 + x_h.numel() * 2
    d2h = out_h[0].numel() * 2

    # ---------------- aggregate over ranks (max time)
    ms_step, e2e_ms = max_over_ranks([total_ms / K, e2e_ms], dev)
    if rank != 0:
        return 0

    flops = layer_flops(cfg)
    value = aggregate_tflops(world, flops, ms_step)
    e2e_value = aggregate_tflops(world, flops, e2e_ms)
    pk, pk_src = peaks()
    up_ms = statistics.mean(parts["up"])
    up_flops = 4.0 * T * k * H * I
    traffic_call = recorded_traffic("grouped_gemm_up") if workload == WORKLOAD else None
    traffic = recorded_traffic("grouped_gemm_window_kernel_up") if workload == WORKLOAD else None
    cpu_v, cpu_desc, cpu_cores, _ = cpu_oracle_sample(cfg, inp, seconds=15.0, max_tokens=cfg.T)
    counts = ws[v.counts - ws.data_ptr():v.counts - ws.data_ptr() + 4 * E].view(torch.int32).cpu().numpy()
    touched = int((counts > 0).sum())
    def roofline_of(alg_bytes, ms):
        # the bound is the larger floor: bytes at the measured copy bandwidth
        # vs FLOPs at the measured sustained bf16 rate
        tflops = up_flops / (ms * 1e-3) / 1e12
        gbs = alg_bytes / (ms * 1e-3) / 1e9
        extra = {"algorithmic_bytes_per_launch": alg_bytes, "algorithmic_flops_per_launch": up_flops,
                 "us_per_launch": ms * 1e3, "hbm_frac": gbs / pk["hbm_gbs"],
                 "tensor_frac_sustained": tflops / pk["bf16_tflops_sustained"],
                 "tensor_frac_burst": tflops / pk["bf16_tflops"]}
        if alg_bytes / pk["hbm_gbs"] / 1e9 >= up_flops / pk["bf16_tflops_sustained"] / 1e12:
            return dict(extra, bound="hbm", achieved=gbs, peak=pk["hbm_gbs"], unit="GB/s",
                        frac=gbs / pk["hbm_gbs"], peak_source="%s hbm_gbs" % pk_src)
        return dict(extra, bound="tensor", achieved=tflops, peak=pk["bf16_tflops_sustained"], unit="TFLOP/s",
                    frac=tflops / pk["bf16_tflops_sustained"], peak_source="%s bf16_tflops_sustained" % pk_src)

    # Algorithmic bytes of the gate/up step (each touched expert's W_gate and
    # W_up once, each token row of X once, h written once): the figure the
    # kernel's roofline fraction is quoted on.  The kernel timed alone reads
    # the gathered rows Xp (T*k rows) instead of X; that figure is reported
    # beside it as frac_with_xp.
    up_bytes = touched * 2 * H * I * 2 + T * H * 2 + T * k * I * 2
    gemm_bytes_xp = touched * 2 * H * I * 2 + T * k * H * 2 + T * k * I * 2
    roof = roofline_of(up_bytes, gemm_ms)
    roof_xp = roofline_of(gemm_bytes_xp, gemm_ms)
    roof_call = roofline_of(up_bytes, up_ms)
    if n_sets == 1:
        l2_note = ("inputs larger than L2: %.2f GB resident per layer (%.2f GB of expert weights), L2 %.0f MB; "
                   "no flush" % (set_bytes / 1e9, 3 * E * H * I * 2 / 1e9, l2_bytes / 1e6))
    else:
        l2_note = ("inputs larger than L2 by rotation: %d buffer sets of %.1f MB (weights, X, logits, workspace, "
                   "out), step i on set i mod %d, %.0f MB in all against L2 %.0f MB; no flush"
                   % (n_sets, set_bytes / 1e6, n_sets, n_sets * set_bytes / 1e6, l2_bytes / 1e6))
    nb = int(ws[v.num_blocks - ws.data_ptr():v.num_blocks - ws.data_ptr() + 4].view(torch.int32).item())
    layer_roof = layer_roofline(cfg, touched, nb * 128, ms_step, pk, pk_src)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "us_per_layer": ms_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "%s (T=%d,H=%d,I=%d,E=%d,k=%d)" % ((cfg.name,) + cfg.shape),
                   "T": T, "H": H, "I": I, "E": E, "k": k,
                   "l2": l2_note,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "launch": launch if singles is None else
                   "cuda_graph: %d forwards per graph, %d replays + %d one-forward replays"
                   % (G, K // G, K % G)},
        "per_kernel_us": {n: statistics.mean(vv) * 1e3 for n, vv in parts.items()},
        "step_by_step_us": steps_ms * 1e3,
        "graph_of_one_us": one_ms * 1e3,
        "roofline": dict(roof, kernel="grouped_gemm_window_kernel<up> (token-window CTA-pair tcgen05 grouped "
                                      "GEMM, timed through moe_grouped_gemm_up_rows)",
                         bytes_model="touched experts' W_gate and W_up once + X once (T*H*2) + h once",
                         traffic=traffic,
                         frac_with_xp=roof_xp["frac"],
                         bytes_with_xp=gemm_bytes_xp,
                         up_call=dict(roof_call, kernel="moe_grouped_gemm_up call (row gather + the GEMM)",
                                      traffic=traffic_call)),
        "layer_roofline": layer_roof,
        "cpu_baseline": {"value": cpu_v, "unit": UNIT, "cores": cpu_cores, "kind": "oracle",
                         "sample": cpu_desc},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "clocks": e2e_clk},
        "gpu_launches": moe.FORWARD_KERNELS * K,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_profile(args, local):
    """Warm-up forwards plus one forward of the chosen workload (for ncu)."""
    import numpy as np
    import torch

    import combine_moe_route_04_gb300 as moe
    import moe_inputs
    from combine_moe_route_04_gb300 import _build

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    cfg = moe_inputs.config(args.workload)
    if args.shape:
        T, H, I, E, k = (int(v) for v in args.shape.split(","))
        cfg = moe_inputs.MoEConfig("shape_%d_%d_%d_%d_%d" % (T, H, I, E, k), T, H, I, E, k, seed=7)
    inp = moe_inputs.make_inputs(cfg)
    s = moe.shape(*cfg.shape)

    def up_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    logits = torch.from_numpy(inp["logits"]).to(dev)
    x, wg, wu, wd = (up_bf16(inp[n]) for n in ("x", "w_gate", "w_up", "w_down"))
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    ws = moe.alloc_workspace(s, dev)
    for _ in range(args.warmup + 1):
        moe.moe_forward(s, logits, x, wg, wu, wd, out, ws)
    torch.cuda.synchronize(dev)
    rc = moe.last_device_status(ws)
    print(json.dumps({"profile_run": cfg.name, "forwards": args.warmup + 1, "device_status": rc}))
    return 0 if rc == 0 else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--profile", action="store_true",
                    help="run --warmup forwards, then one more forward, and exit (no timing): "
                         "the command line for ncu captures")
    ap.add_argument("--workload", type=int, default=WORKLOAD,
                    help="which workload (1-5) to time (default: the pages-shaped layer)")
    ap.add_argument("--shape", type=str, default=None,
                    help="with --profile: T,H,I,E,k of a synthetic shape instead of a workload")
    args = ap.parse_args()
    world, rank, local = dist_init()
    if args.profile:
        return run_profile(args, local)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
