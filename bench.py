#!/usr/bin/env python3
"""Benchmark of the Mamba2 mixer core on GB300.

Workload: one Nemotron-H mixer at the real shape (H=128, P=80, N=128, G=8,
K=4; bf16 activations, fp32 state), batch 1, a T=300-frame timeline (24 s at
12.5 frames/s), chunk 128. One bench step is one pass of the whole hot path
for one layer: the full-history chunked scan over the 300 frames (conv +
SiLU, dt, SSD scan) followed by one cached single-frame step (frame 301) from
the scan's final state. Steps cycle through 27 independently seeded layers
(the Mamba layers of the 56-layer pattern), so the working set (~570 MB) is
larger than L2 and no step reuses another's data from cache.

value   = tokens per second = 301 frames x steps / device time (CUDA events).
e2e     = the same metric through the C ABI with host buffers: pinned host ->
          device copies of each step's inputs and device -> host copies of its
          outputs inside the timed region.
roofline: the dominant kernel (the fused SSD scan kernel, mamba2_scan_chunks),
          algorithmic bytes per launch / its CUDA-event duration, against the
          measured HBM copy bandwidth; a tensor-core figure is reported beside it.
cpu_baseline / --impl reference: the fp64 oracle on the host cores.

Multi-GPU (torchrun): every rank runs the same workload on its own GPU with
no data exchange (independent replicas, weak scaling); only the timing is
reduced (max over ranks).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from seeded_inputs import MAMBA_LAYERS, REAL_SHAPE, device_mixer_inputs, mixer_inputs  # noqa: E402

T_FRAMES = 300
CHUNK = 128
N_LAYERS = len(MAMBA_LAYERS)
METRIC = "Mamba2 scan tokens/s and per-frame step µs; % of HBM / bf16 MMA roofline"
WORKLOAD = ("Nemotron-H Mamba2 mixer, real shape H=128 P=80 N=128 G=8 K=4, batch 1, T=300 chunked scan "
            "(chunk 128) + 1 cached step, bf16 activations / fp32 state, 27 layers cycled")

# Algorithmic work per unit:
#   scan bytes per token: x|B|C in 24,576 + dt 256 + y out 20,480 = 45,312 B
#   plus the final fp32 state (H*P*N*4 = 5,242,880 B) and conv tail (3*12288*2) per sequence.
#   scan MMA flops per token at chunk Q, counting the causal (lower-triangular)
#   half of the two Q x Q products: C.B^T Q*N*G + M.x Q*P*H + chunk state
#   2*N*P*H + C.h 2*N*P*H = 6,684,672 at Q = 128 (5,963,776 at Q = 64).
#   step bytes per session: 2 x 5,242,880 state + 2 x 73,728 conv tail + 24,832 in + 20,480 out.
# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one SSD-kernel
# launch of this workload, from an ncu capture of the kernel. It describes one
# version of the kernel source; for any other version the traffic is reported
# as unknown (null).
SSD_TRAFFIC = {"bytes": 8868096, "m2_scan_cu_sha1": "f2e8ceba94155ffc9651c1b51785356cc27d0f6a"}
SCAN_BYTES_PER_TOKEN = 45312
STATE_BYTES = 128 * 80 * 128 * 4
TAIL_BYTES = 3 * 12288 * 2


def scan_flops_per_token(q):
    """Algorithmic MMA flops per token of the chunked scan at chunk length q
    (causal halves of the two q x q products; the chunk state and C.h in full)."""
    H, P, N, G = 128, 80, 128, 8
    return q * N * G + q * P * H + 4 * N * P * H


SCAN_FLOPS_PER_TOKEN = scan_flops_per_token(CHUNK)
STEP_BYTES_PER_SESSION = 2 * STATE_BYTES + 2 * TAIL_BYTES + 24832 + 20480


def ssd_traffic_for_current_source():
    import hashlib
    src = os.path.join(ROOT, "full_duplex_speech_gb300", "csrc", "m2_scan.cu")
    try:
        sha = hashlib.sha1(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    return SSD_TRAFFIC["bytes"] if sha == SSD_TRAFFIC["m2_scan_cu_sha1"] else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return dict(hbm=j["hbm_gbs"], bf16=j["bf16_tflops"], bf16_sust=j.get("bf16_tflops_sustained"),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, source="fallback")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for ts, r in rows if t0 - 0.1 <= ts <= t1 + 0.1] or [r for _, r in rows[-3:]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(tokens_per_rank: float, ms_local: float, world: int, device=None):
    """Whole-job throughput: tokens of all ranks over the slowest rank's time
    (independent replicas, weak scaling). Returns (tokens/s, max ms)."""
    ms = reduce_max(ms_local, world, device)
    return world * tokens_per_rank / (ms * 1e-3), ms


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a float over all ranks (the only cross-rank operation)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- oracle leg
def oracle_tokens_per_s(budget_s: float, nthreads: int, heads_cap=None):
    """The fp64 oracle (as it stands) on one layer of the workload: the
    T=301-frame recurrence (300 prefill frames + 1 cached frame; a cached step
    is one more iteration of the same loop) for a sample of heads, timed
    until `budget_s` seconds of work; tokens/s scaled to all 128 heads."""
    import oracle
    d = REAL_SHAPE
    inp = mixer_inputs(1000, d, 1, T_FRAMES + 1, "bf16")
    hs = 16 if heads_cap is None else heads_cap
    t0 = time.perf_counter()
    oracle.mixer_scan(d, inp, heads=(0, hs), nthreads=nthreads)
    one = time.perf_counter() - t0
    reps, elapsed = 1, one
    while elapsed < budget_s:
        t0 = time.perf_counter()
        oracle.mixer_scan(d, inp, heads=(0, hs), nthreads=nthreads)
        elapsed += time.perf_counter() - t0
        reps += 1
    per_rep = elapsed / reps
    # hs heads took per_rep seconds: all 128 heads take per_rep * 128 / hs
    value = (T_FRAMES + 1) / (per_rep * d.H / hs)
    return value, dict(heads=hs, reps=reps, seconds=elapsed)


def run_reference(args, world, rank):
    """--impl reference: the oracle timed on the host cores, rank 0 only."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    nthreads = os.cpu_count() or 1
    # each step is a bounded sample: sized so that warmup + steps take ~2 minutes
    budget_total = 120.0
    d = REAL_SHAPE
    inp = mixer_inputs(1000, d, 1, T_FRAMES + 1, "bf16")
    t0 = time.perf_counter()
    oracle.mixer_scan(d, inp, heads=(0, 8), nthreads=nthreads)
    per_head = (time.perf_counter() - t0) / 8
    per_step = budget_total / max(1, args.steps + args.warmup)
    hs = int(max(1, min(d.H, per_step / max(per_head, 1e-9))))
    hs = max(1, min(d.H, (hs // nthreads) * nthreads or hs))
    for _ in range(args.warmup):
        oracle.mixer_scan(d, inp, heads=(0, hs), nthreads=nthreads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.mixer_scan(d, inp, heads=(0, hs), nthreads=nthreads)
        times.append(time.perf_counter() - t0)
    ms = 1000.0 * sum(times) / len(times) * d.H / hs  # scaled to all 128 heads
    value = (T_FRAMES + 1) / (ms / 1000.0)
    sample = (f"per step: oracle fp64 recurrence over 301 frames for {hs} of 128 heads of one layer, "
              f"scaled by 128/{hs}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; distributions of the tiny/real mixer configs)",
            "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": T_FRAMES + 1},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- GPU leg
class Layer:
    """Device buffers of one layer: inputs for 301 frames, outputs, scratch."""

    def __init__(self, m2, seed, torch, dev):
        d = REAL_SHAPE
        self.inp = mixer_inputs(seed, d, 1, T_FRAMES + 1, "bf16")

        def dt(a):
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
            return torch.from_numpy(a).to(dev)

        # one step's inputs (the 300 prefill frames and the cached frame of x,
        # B, C, dt_raw) packed into one device buffer, and its outputs (y, y1)
        # into another, so that the end-to-end run copies each with one call
        parts = {}
        for k in ("x", "B", "C", "dt_raw"):
            v = np.ascontiguousarray(self.inp[k])
            parts["s" + k] = np.ascontiguousarray(v[:, :T_FRAMES])
            parts["f" + k] = np.ascontiguousarray(v[:, T_FRAMES])
        offs, total = {}, 0
        for k, v in parts.items():
            offs[k] = total
            total += (v.nbytes + 255) // 256 * 256
        host = np.zeros(total, dtype=np.uint8)
        for k, v in parts.items():
            host[offs[k]:offs[k] + v.nbytes] = v.view(np.uint8).reshape(-1)
        self.in_bytes = sum(v.nbytes for v in parts.values())
        self.dev_in = torch.from_numpy(host).to(dev)
        self.host_in = torch.from_numpy(host).pin_memory()

        def view(buf, off, a):
            return buf[off:off + a.nbytes].view(torch.bfloat16).view(a.shape)

        self.seq = {k: view(self.dev_in, offs["s" + k], parts["s" + k]) for k in ("x", "B", "C", "dt_raw")}
        self.frame = {k: view(self.dev_in, offs["f" + k], parts["f" + k]) for k in ("x", "B", "C", "dt_raw")}
        self.p = {k: dt(self.inp[k]) for k in ("A_log", "D", "dt_bias", "conv_w", "conv_b")}
        self.dims = m2.dims(1, T_FRAMES, d.H, d.P, d.N, d.G, d.K, "bf16")
        ny, ny1 = T_FRAMES * d.H * d.P, d.H * d.P
        self.dev_out = torch.empty(ny + ny1, dtype=torch.bfloat16, device=dev)
        self.host_out = torch.empty(ny + ny1, dtype=torch.bfloat16).pin_memory()
        self.out_bytes = (ny + ny1) * 2
        self.y = self.dev_out[:ny].view(1, T_FRAMES, d.H, d.P)
        self.y1 = self.dev_out[ny:].view(1, d.H, d.P)
        self.fs = torch.empty((1, d.H, d.P, d.N), dtype=torch.float32, device=dev)
        self.fc = torch.empty((1, d.K - 1, d.CH), dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(m2.mamba2_scan_workspace_bytes(self.dims, CHUNK), dtype=torch.uint8, device=dev)
        self.wss = torch.empty(m2.mamba2_step_workspace_bytes(self.dims, 1), dtype=torch.uint8, device=dev)

    def scan_args(self):
        s, p = self.seq, self.p
        return (self.dims, s["x"], s["B"], s["C"], s["dt_raw"], p["A_log"], p["D"], p["dt_bias"], p["conv_w"],
                p["conv_b"], CHUNK, None, None, self.y, self.fs, self.fc, self.ws)

    def step_args(self):
        f, p = self.frame, self.p
        return (self.dims, 1, f["x"], f["B"], f["C"], f["dt_raw"], p["A_log"], p["D"], p["dt_bias"],
                p["conv_w"], p["conv_b"], self.fs, self.fc, self.y1, self.wss)


def enqueue_step(m2, L, stream, ev=None):
    """One bench step on `stream`: the scan, then one cached step. Without
    events it is the public calls (mamba2_conv_scan, mamba2_step). With
    ev = (a, b, c) the scan is issued as its two halves with events around
    the SSD kernel (mamba2_scan_chunks) and around the step call."""
    if not ev:
        m2.mamba2_conv_scan(*L.scan_args(), stream=stream)
        m2.mamba2_step(*L.step_args(), stream=stream)
        return
    m2.mamba2_scan_prepare_bc(*L.scan_args(), stream=stream)
    ev[0].record(stream)
    m2.mamba2_scan_chunks(*L.scan_args(), stream=stream)
    ev[1].record(stream)
    m2.mamba2_step(*L.step_args(), stream=stream)
    ev[2].record(stream)


def _time_step_graph(m2, torch, stream, arg_list, reps):
    """Average microseconds of one pass over `arg_list` (mamba2_step argument
    tuples), captured as one CUDA graph and replayed `reps` times."""
    with torch.cuda.stream(stream):
        for a in arg_list:
            m2.mamba2_step(*a, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for a in arg_list:
            m2.mamba2_step(*a, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def _time_graph(torch, stream, fn, reps):
    """Average microseconds of one fn() (which enqueues on `stream`),
    captured as one CUDA graph and replayed `reps` times."""
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def _sessions_step_args(m2, torch, dev, L, S):
    """mamba2_step arguments for S sessions of layer L's weights, with random
    states (the timing does not depend on their values)."""
    d = REAL_SHAPE
    g = torch.Generator(device=dev).manual_seed(64)
    fr = {k: torch.randn((S,) + tuple(v.shape[1:]), generator=g, device=dev).to(v.dtype)
          for k, v in L.frame.items()}
    ssm = torch.randn((S, d.H, d.P, d.N), generator=g, device=dev) * 0.01
    conv = torch.randn((S, d.K - 1, d.CH), generator=g, device=dev).to(torch.bfloat16)
    y = torch.empty((S, d.H, d.P), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(m2.mamba2_step_workspace_bytes(L.dims, S), dtype=torch.uint8, device=dev)
    p = L.p
    return (L.dims, S, fr["x"], fr["B"], fr["C"], fr["dt_raw"], p["A_log"], p["D"], p["dt_bias"], p["conv_w"],
            p["conv_b"], ssm, conv, y, ws)


def lm_position_bytes(cfg, S, cached):
    """Algorithmic bytes of one cached position: every weight read once
    (4-bit fields with their bf16 scales and biases; bf16 attention
    projections), each Mamba block's fp32 state and conv tail read and
    written, each attention block's cached keys and values read and the new
    ones written, the residual stream read and written per block."""
    d = cfg.mixer
    HP, GN = d.H * d.P, d.G * d.N
    W = 2 * HP + 2 * GN + d.H
    q4 = lambda o, i: o * i // 2 + 2 * o * (i // 64) * 2  # noqa: E731
    m = q4(W, cfg.hidden) + q4(cfg.hidden, HP) + S * (2 * HP * d.N * 4 + 2 * 3 * d.CH * 2)
    kv = cfg.n_kv_heads * cfg.head_dim * 2
    a = ((cfg.n_heads + 2 * cfg.n_kv_heads) * cfg.head_dim * cfg.hidden + cfg.hidden * cfg.n_heads * cfg.head_dim) * 2
    a += S * (2 * kv * cached + 2 * kv)
    nm, na = cfg.kinds.count("M"), cfg.kinds.count("*")
    return nm * m + na * a + len(cfg.kinds) * S * cfg.hidden * 2 * 2


def lm_position_leg(m2, torch, dev, stream, peaks):
    from seeded_inputs import REAL_LM, device_lm_weights
    cfg, S, cached, max_len = REAL_LM, 1, 750, 1024
    d = cfg.mixer
    wdev = device_lm_weights(7, cfg, dev)
    layers = []
    for i, kind in enumerate(cfg.kinds):
        L = dict(wdev[i])
        if kind == "M":
            L["ssm_state"] = torch.zeros((S, d.H, d.P, d.N), device=dev)
            L["conv_state"] = torch.zeros((S, d.K - 1, d.CH), dtype=torch.bfloat16, device=dev)
        else:
            shape = (S, cfg.n_kv_heads, max_len, cfg.head_dim)
            L["k_cache"] = torch.randn(shape, device=dev).to(torch.bfloat16)
            L["v_cache"] = torch.randn(shape, device=dev).to(torch.bfloat16)
        layers.append(L)
    model = m2.lm_model(cfg.kinds, layers, cfg.hidden, m2.dims(0, 0, d.H, d.P, d.N, d.G, d.K, "bf16"), cfg.n_heads,
                        cfg.n_kv_heads, cfg.head_dim, max_len, cfg.eps)
    ws = torch.empty(m2.mamba2_lm_workspace_bytes(model, S, 1, 1), dtype=torch.uint8, device=dev)
    lens = torch.full((S,), cached, dtype=torch.int32, device=dev)
    h = torch.randn((S, cfg.hidden), device=dev).to(torch.bfloat16)
    torch.cuda.synchronize()

    def one():
        m2.mamba2_lm_step(model, S, h, lens, ws, stream=stream)

    us = _time_graph(torch, stream, one, reps=20)
    nbytes = lm_position_bytes(cfg, S, cached)
    out = {"sessions": S, "blocks": cfg.kinds, "cached_positions": cached, "us_per_position": us,
           "bytes_per_position": nbytes, "achieved_gbs": nbytes / (us * 1e-6) / 1e9,
           "frac_hbm": nbytes / (us * 1e-6) / 1e9 / peaks["hbm"],
           # 'M': in_proj, conv, state update, out_proj; '*': q|k|v, attention, out projection
           "kernels_per_position": 4 * cfg.kinds.count("M") + 3 * cfg.kinds.count("*")}

    # the full-history recompute of 300 positions through the same blocks
    # (mamba2_lm_prefill from empty caches: chunked scans, the projections as
    # GEMMs, attention position by position); each replay first restores the
    # residual stream the call updates in place (a 2.7 MB copy, included)
    T, chunk = 300, 128
    pws = torch.empty(m2.mamba2_lm_workspace_bytes(model, S, T, chunk), dtype=torch.uint8, device=dev)
    plens = torch.zeros((S,), dtype=torch.int32, device=dev)
    h0 = torch.randn((S * T, cfg.hidden), device=dev).to(torch.bfloat16)
    hp = torch.empty_like(h0)
    torch.cuda.synchronize()

    def prefill():
        hp.copy_(h0)
        m2.mamba2_lm_prefill(model, S, T, hp, plens, chunk, pws, stream=stream)

    with torch.cuda.stream(stream):
        p_us = _time_graph(torch, stream, prefill, reps=3)
    out["prefill_T300"] = {"positions": T, "chunk": chunk, "us_per_prefill": p_us,
                           "positions_per_s": S * T / (p_us * 1e-6)}
    del wdev, layers, model, ws, pws
    torch.cuda.synchronize()
    return out


def run_gpu(args, world, rank, local):
    import torch
    from full_duplex_speech_gb300 import build as m2build
    m2build.build()
    import full_duplex_speech_gb300 as m2
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    m2.load()
    peaks = load_peaks()
    layers = [Layer(m2, 1000 + i, torch, dev) for i in range(N_LAYERS)]
    stream = torch.cuda.Stream(device=dev)
    K, W = args.steps, args.warmup
    torch.cuda.synchronize()

    # warm-up (eager), then capture the timed sequence in CUDA graphs
    with torch.cuda.stream(stream):
        for i in range(W):
            enqueue_step(m2, layers[i % N_LAYERS], stream)
    torch.cuda.synchronize()

    try:
        mk = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
        mk()
        graph_events = True
    except TypeError:
        graph_events = False

    sweep = min(K, N_LAYERS)
    g_full = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_full, stream=stream):
        for i in range(sweep):
            enqueue_step(m2, layers[i], stream)
    # a second graph of one sweep with events around the SSD kernel and the step
    # call, replayed right after the timed region for per-kernel durations
    evs = [[torch.cuda.Event(enable_timing=True, external=True) if graph_events else None for _ in range(3)]
           for _ in range(N_LAYERS)]
    g_ev = None
    if graph_events:
        g_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_ev, stream=stream):
            for i in range(N_LAYERS):
                enqueue_step(m2, layers[i], stream, evs[i])
    rem = K % sweep
    g_rem = None
    if rem:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=stream):
            for i in range(rem):
                enqueue_step(m2, layers[i], stream)
    with torch.cuda.stream(stream):  # CUDAGraph.replay() launches on the current stream
        g_full.replay()  # one untimed replay after capture
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    torch.cuda.nvtx.range_push("bench_timed")
    with torch.cuda.stream(stream):
        # ~1 ms of GPU spin ahead of the first event, so that the host has
        # submitted the graph replays by the time the GPU reaches it: the
        # timed region then holds the K steps' device time only, not the
        # host's submission latency (which a short --steps run would feel)
        torch.cuda._sleep(2_000_000)
        e0.record(stream)
        for _ in range(K // sweep):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if g_ev is not None:
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_ev.replay()
        torch.cuda.synchronize()
    barrier(world)
    time.sleep(0.2)
    clocks.stop()
    ms_local = e0.elapsed_time(e1)
    value, ms_total = aggregate(K * (T_FRAMES + 1), ms_local, world, dev)
    ms_per_step = ms_total / K

    # per-kernel durations: from the events inside the last full sweep of the timed region
    if graph_events:
        ssd_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(N_LAYERS)]
        step_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(N_LAYERS)]
        timing_src = ("CUDA events in a graph of one 27-layer sweep (scan issued as its two halves), "
                      "replayed right after the timed region")
    else:
        ssd_ms, step_ms = [], []
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(N_LAYERS)]
        with torch.cuda.stream(stream):
            torch.cuda._sleep(50_000_000)  # keep the GPU busy while the host enqueues ahead
            for i in range(N_LAYERS):
                enqueue_step(m2, layers[i], stream, ev[i])
        torch.cuda.synchronize()
        ssd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(N_LAYERS)]
        step_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(N_LAYERS)]
        timing_src = "CUDA events on the launch stream (eager, host ahead of the GPU)"
    ssd_avg = sum(ssd_ms) / len(ssd_ms)
    step_avg = sum(step_ms) / len(step_ms)

    ssd_bytes = SCAN_BYTES_PER_TOKEN * T_FRAMES + STATE_BYTES + TAIL_BYTES
    ssd_gbs = ssd_bytes / (ssd_avg * 1e-3) / 1e9
    ssd_flops = SCAN_FLOPS_PER_TOKEN * T_FRAMES
    ssd_tfs = ssd_flops / (ssd_avg * 1e-3) / 1e12
    step_gbs = STEP_BYTES_PER_SESSION / (step_avg * 1e-3) / 1e9

    # cached decode: one frame through all 27 layers (batch 1), and one layer
    # call for 64 sessions; graphs of consecutive step calls, no events between
    # them, so the launches keep their programmatic dependencies
    torch.cuda.nvtx.range_push("step_frame")
    frame_us = _time_step_graph(m2, torch, stream, [(L.step_args()) for L in layers], reps=50)
    torch.cuda.nvtx.range_pop()
    step_frame = {"us_per_frame_27_layers": frame_us, "us_per_layer": frame_us / N_LAYERS,
                  "achieved_gbs": N_LAYERS * STEP_BYTES_PER_SESSION / (frame_us * 1e-6) / 1e9}
    step_frame["frac_hbm"] = step_frame["achieved_gbs"] / peaks["hbm"]
    s64 = _sessions_step_args(m2, torch, dev, layers[0], 64)
    torch.cuda.synchronize()  # its tensors were made on torch's stream, not `stream`
    torch.cuda.nvtx.range_push("step64")
    s64_us = _time_step_graph(m2, torch, stream, [s64], reps=50)
    torch.cuda.nvtx.range_pop()
    step64 = {"sessions": 64, "us_per_call": s64_us,
              "achieved_gbs": 64 * STEP_BYTES_PER_SESSION / (s64_us * 1e-6) / 1e9}
    step64["frac_hbm"] = step64["achieved_gbs"] / peaks["hbm"]
    del s64
    torch.cuda.synchronize()

    # the whole scan (both kernels) of the real-scan workload at chunk 64 and
    # 128, 27 layers cycled in a graph; tensor figures from each chunk's
    # algorithmic flops
    chunk_sweep = {}
    torch.cuda.nvtx.range_push("chunk_sweep")
    for q in (64, 128):
        qws = [torch.empty(m2.mamba2_scan_workspace_bytes(L.dims, q), dtype=torch.uint8, device=dev)
               for L in layers]
        torch.cuda.synchronize()

        def q_scans():
            for L, w in zip(layers, qws):
                a = list(L.scan_args())
                a[10], a[16] = q, w
                m2.mamba2_conv_scan(*a, stream=stream)

        q_us = _time_graph(torch, stream, q_scans, reps=20) / N_LAYERS
        q_tfs = scan_flops_per_token(q) * T_FRAMES / (q_us * 1e-6) / 1e12
        chunk_sweep[str(q)] = {"us_per_scan": q_us, "tokens_per_s": T_FRAMES / (q_us * 1e-6),
                               "algorithmic_tflops": q_tfs, "frac_bf16": q_tfs / peaks["bf16"],
                               "note": "whole scan (B/C prologue + SSD kernel); flops of the SSD contractions"}
        del qws
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()

    # the gated output norm over the T=300 rows of a scan's y (8 buffer sets
    # cycled, 147 MB, larger than L2)
    d = REAL_SHAPE
    gn = torch.Generator(device=dev).manual_seed(77)
    norm_sets = [(torch.randn((T_FRAMES, d.H * d.P), generator=gn, device=dev).to(torch.bfloat16),
                  torch.randn((T_FRAMES, d.H * d.P), generator=gn, device=dev).to(torch.bfloat16),
                  1 + 0.1 * torch.randn(d.H * d.P, generator=gn, device=dev),
                  torch.empty((T_FRAMES, d.H * d.P), dtype=torch.bfloat16, device=dev)) for _ in range(8)]
    torch.cuda.synchronize()

    def norm_pass():
        for yv, zv, wv, ov in norm_sets:
            m2.mamba2_gated_norm(layers[0].dims, T_FRAMES, yv, zv, wv, 1e-5, ov, stream=stream)

    torch.cuda.nvtx.range_push("gated_norm")
    norm_us = _time_graph(torch, stream, norm_pass, reps=50) / len(norm_sets)
    torch.cuda.nvtx.range_pop()
    norm_bytes = T_FRAMES * d.H * d.P * 6 + d.H * d.P * 4
    gated_norm = {"rows": T_FRAMES, "us_per_call": norm_us, "bytes_per_call": norm_bytes,
                  "achieved_gbs": norm_bytes / (norm_us * 1e-6) / 1e9}
    gated_norm["frac_hbm"] = gated_norm["achieved_gbs"] / peaks["hbm"]
    del norm_sets
    torch.cuda.synchronize()

    # 4-bit group-64 quantized mixer projections (in_proj 4480 -> 22656,
    # out_proj 10240 -> 4480) for 1 and 4 rows of x (one cached frame of 1 or 4
    # sessions), and for 300 rows (a prefill of 300 positions: the tensor-core
    # GEMM), 4 random weight sets per shape (> L2) cycled in a graph
    qlinear = {}
    torch.cuda.nvtx.range_push("qlinear")
    for name, n_in, n_out in (("in_proj", 4480, 22656), ("out_proj", 10240, 4480)):
        wsets = []
        for _ in range(4):
            wsets.append((torch.randint(-2**31, 2**31 - 1, (n_out, n_in // 8), dtype=torch.int32, device=dev),
                          (torch.rand(n_out, n_in // 64, device=dev) * 0.01).bfloat16(),
                          (torch.rand(n_out, n_in // 64, device=dev) * -0.05).bfloat16()))
        wbytes = n_out * n_in // 2 + 2 * n_out * (n_in // 64) * 2
        for rows in (1, 4, 300):
            qx = torch.randn(rows, n_in, device=dev).bfloat16()
            qy = torch.empty(rows, n_out, dtype=torch.bfloat16, device=dev)
            torch.cuda.synchronize()

            def q_pass():
                for wq, sc, bi in wsets:
                    m2.mamba2_qlinear(rows, n_in, n_out, qx, wq, sc, bi, qy, stream=stream)

            q_us = _time_graph(torch, stream, q_pass, reps=20) / len(wsets)
            qb = wbytes + rows * (n_in + n_out) * 2
            qlinear[f"{name}_rows{rows}"] = {"in": n_in, "out": n_out, "rows": rows, "us_per_call": q_us,
                                             "bytes_per_call": qb, "achieved_gbs": qb / (q_us * 1e-6) / 1e9,
                                             "frac_hbm": qb / (q_us * 1e-6) / 1e9 / peaks["hbm"]}
            if rows >= 40:  # the GEMM: its tensor fraction (2 flops per weight and row)
                tfs = 2.0 * rows * n_in * n_out / (q_us * 1e-6) / 1e12
                qlinear[f"{name}_rows{rows}"].update({"tflops": tfs, "frac_bf16": tfs / peaks["bf16"]})
        del wsets
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()

    # cached decode of the attention layers (40 query heads, 8 kv heads,
    # head_dim 128): one session with 750 and 7500 frames cached (60 s and the
    # 600 s session limit), 64 sessions with 750; sets of KV caches cycled in a
    # graph so that together they exceed L2. Algorithmic bytes per call: every
    # cached key and value read once, the new ones read and written to the
    # cache, q read and out written.
    attn = {}
    torch.cuda.nvtx.range_push("attn_decode")
    AHQ, AHKV, AD = 40, 8, 128
    for name, a_s, a_len, nsets in (("b1_len750", 1, 750, 48), ("b1_len7500", 1, 7500, 8),
                                    ("s64_len750", 64, 750, 2)):
        a_tmax = a_len + 1
        ga = torch.Generator(device=dev).manual_seed(91)
        asets = []
        for _ in range(nsets):
            asets.append(dict(
                kc=torch.randn((a_s, AHKV, a_tmax, AD), generator=ga, device=dev).bfloat16(),
                vc=torch.randn((a_s, AHKV, a_tmax, AD), generator=ga, device=dev).bfloat16(),
                q=torch.randn((a_s, AHQ, AD), generator=ga, device=dev).bfloat16(),
                kn=torch.randn((a_s, AHKV, AD), generator=ga, device=dev).bfloat16(),
                vn=torch.randn((a_s, AHKV, AD), generator=ga, device=dev).bfloat16(),
                out=torch.empty((a_s, AHQ, AD), dtype=torch.bfloat16, device=dev)))
        a_lens = torch.full((a_s,), a_len, dtype=torch.int32, device=dev)
        a_ws = torch.empty(m2.mamba2_attn_decode_workspace_bytes(a_s, AHQ, AHKV, AD, a_tmax), dtype=torch.uint8,
                           device=dev)
        torch.cuda.synchronize()

        def a_pass():
            for z in asets:
                m2.mamba2_attn_decode(a_s, AHQ, AHKV, AD, a_tmax, "bf16", a_lens, z["q"], z["kn"], z["vn"], z["kc"],
                                      z["vc"], AD ** -0.5, z["out"], a_ws, stream=stream)

        a_us = _time_graph(torch, stream, a_pass, reps=20) / nsets
        a_bytes = a_s * AHKV * AD * 2 * (2 * a_len + 4) + a_s * AHQ * AD * 2 * 2
        attn[name] = {"sessions": a_s, "cached_positions": a_len, "us_per_call": a_us, "bytes_per_call": a_bytes,
                      "achieved_gbs": a_bytes / (a_us * 1e-6) / 1e9,
                      "frac_hbm": a_bytes / (a_us * 1e-6) / 1e9 / peaks["hbm"]}
        del asets, a_ws
        torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()

    # long prefill: one layer at batch 4, T=4096 (the parity tests run all 27
    # layers of it); the whole scan and its SSD kernel alone, CUDA events
    PB, PT = 4, 4096
    pf = device_mixer_inputs(4242, d, PB, PT, dev)
    pdims = m2.dims(PB, PT, d.H, d.P, d.N, d.G, d.K, "bf16")
    py = torch.empty((PB, PT, d.H, d.P), dtype=torch.bfloat16, device=dev)
    pfs = torch.empty((PB, d.H, d.P, d.N), device=dev)
    pfc = torch.empty((PB, d.K - 1, d.CH), dtype=torch.bfloat16, device=dev)
    pws = torch.empty(m2.mamba2_scan_workspace_bytes(pdims, CHUNK), dtype=torch.uint8, device=dev)
    pargs = (pdims, pf["x"], pf["B"], pf["C"], pf["dt_raw"], pf["A_log"], pf["D"], pf["dt_bias"], pf["conv_w"],
             pf["conv_b"], CHUNK, None, None, py, pfs, pfc, pws)
    torch.cuda.synchronize()
    pev = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    torch.cuda.nvtx.range_push("prefill")
    with torch.cuda.stream(stream):
        for _ in range(2):
            m2.mamba2_conv_scan(*pargs, stream=stream)
        pev[0].record(stream)
        for _ in range(5):
            m2.mamba2_conv_scan(*pargs, stream=stream)
        pev[1].record(stream)
        for k in range(3):
            m2.mamba2_scan_prepare_bc(*pargs, stream=stream)
            pev[2 + 2 * k].record(stream)
            m2.mamba2_scan_chunks(*pargs, stream=stream)
            pev[3 + 2 * k].record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    pf_ms = pev[0].elapsed_time(pev[1]) / 5
    pf_ssd_ms = sum(pev[2 + 2 * k].elapsed_time(pev[3 + 2 * k]) for k in range(3)) / 3
    pf_bytes = SCAN_BYTES_PER_TOKEN * PB * PT + PB * (STATE_BYTES + TAIL_BYTES)
    pf_flops = SCAN_FLOPS_PER_TOKEN * PB * PT
    prefill = {"batch": PB, "T": PT, "chunk": CHUNK, "ms_per_layer": pf_ms, "tokens_per_s": PB * PT / (pf_ms * 1e-3),
               "ssd_ms": pf_ssd_ms,
               "ssd_frac_hbm": pf_bytes / (pf_ssd_ms * 1e-3) / 1e9 / peaks["hbm"],
               "ssd_frac_bf16": pf_flops / (pf_ssd_ms * 1e-3) / 1e12 / peaks["bf16"]}
    del pf, py, pfs, pfc, pws
    torch.cuda.synchronize()

    # one cached position of the hybrid model (27 Mamba + 4 attention blocks
    # of Nemotron-H at full size, synthetic weights, one session with 750
    # positions in its KV caches): mamba2_lm_step replayed from a CUDA graph;
    # the weights (2.7 GB) exceed L2, so every replay streams them again
    lm = lm_position_leg(m2, torch, dev, stream, peaks)

    # End to end through the C ABI with host buffers: every step copies its
    # inputs in from pinned host memory (one copy) and its results out (one
    # copy), around the public calls (mamba2_conv_scan, mamba2_step). Three
    # streams pipeline the copies of one step under the compute of the next,
    # and one 27-step window is captured as a CUDA graph and replayed.
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)

    def e2e_window():
        fork = torch.cuda.Event()
        fork.record(stream)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        for L in layers:
            with torch.cuda.stream(s_in):
                L.dev_in.copy_(L.host_in, non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(s_in)
            stream.wait_event(landed)
            enqueue_step(m2, L, stream)
            done = torch.cuda.Event()
            done.record(stream)
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                L.host_out.copy_(L.dev_out, non_blocking=True)
        for st_ in (s_in, s_out):
            join = torch.cuda.Event()
            join.record(st_)
            stream.wait_event(join)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e2e_window()
    torch.cuda.synchronize()
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=stream):
        e2e_window()
    reps = max(2, min(8, K // N_LAYERS))
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ge.replay()
        a0.record(stream)
        for _ in range(reps):
            ge.replay()
        a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(a0.elapsed_time(a1), world, dev) / (reps * N_LAYERS)
    e2e = {"value": world * (T_FRAMES + 1) / (e2e_ms * 1e-3), "unit": "tokens/s",
           "h2d_bytes_per_step": layers[0].in_bytes, "d2h_bytes_per_step": layers[0].out_bytes,
           "ms_per_step": e2e_ms, "steps": reps * N_LAYERS,
           "how": "per step one copy of the inputs from pinned host memory and one copy of y, y1 back to it, "
                  "on two copy streams pipelined under the compute stream; 27-step windows replayed as a CUDA "
                  "graph"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nthreads = os.cpu_count() or 1
        v, info = oracle_tokens_per_s(args.cpu_seconds, nthreads)
        v1, info1 = oracle_tokens_per_s(args.cpu_seconds / 2, 1, heads_cap=4)
        cpu = {"value": v, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
               "sample": (f"fp64 oracle, one layer: 301-frame recurrence (300 prefill + 1 cached) for "
                          f"{info['heads']} of 128 heads, {info['reps']} reps in {info['seconds']:.1f} s, "
                          f"scaled by 128/{info['heads']}"),
               "single_thread": {"value": v1, "unit": "tokens/s", "cores": 1,
                                 "sample": (f"the same recurrence on one thread for {info1['heads']} heads, "
                                            f"{info1['reps']} reps in {info1['seconds']:.1f} s, scaled by "
                                            f"128/{info1['heads']}")}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded; no checkpoint or dataset)",
            "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": T_FRAMES + 1,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2: 27 layer buffer sets (~570 MB) cycled"},
            "roofline": {"bound": "hbm", "kernel": "scan_ssd_kernel (mamba2_scan_chunks)",
                         "achieved": ssd_gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": ssd_gbs / peaks["hbm"],
                         "traffic": args.ssd_traffic if args.ssd_traffic is not None else ssd_traffic_for_current_source(),
                         "algorithmic_bytes_per_launch": ssd_bytes, "avg_launch_ms": ssd_avg,
                         "byte_counts": ("achieved = algorithmic_bytes_per_launch / avg_launch_ms; traffic = "
                                         "measured DRAM bytes per launch (ncu), lower than the algorithmic "
                                         "bytes because y and the final state are still in L2 when the "
                                         "kernel ends"),
                         "tensor_fraction": "roofline_tensor (the scan's own target is a bf16 tensor fraction)",
                         "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)",
                         "timing": timing_src},
            "roofline_tensor": {"kernel": "scan_ssd_kernel", "achieved": ssd_tfs, "peak": peaks["bf16"],
                                "unit": "TFLOP/s", "frac": ssd_tfs / peaks["bf16"],
                                "algorithmic_flops_per_launch": ssd_flops,
                                "flops": "causal halves of the two chunk x chunk products, chunk 128"},
            "scan_chunk_sweep_T300": chunk_sweep,
            "step": {"us_per_layer_call_in_bench_step": step_avg * 1e3, "achieved_gbs": step_gbs,
                     "frac_hbm": step_gbs / peaks["hbm"], "bytes_per_call": STEP_BYTES_PER_SESSION,
                     "sessions": 1},
            "step_frame_b1": step_frame,
            "step_64_sessions": step64,
            "gated_norm_T300": gated_norm,
            "qlinear_4bit_g64": qlinear,
            "attn_decode": attn,
            "prefill_b4_T4096": prefill,
            "lm_position_b1": lm,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": 4 * K,
            "clocks": clocks.summary(t_wall0, t_wall1),
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5400)
    ap.add_argument("--warmup", type=int, default=27)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ssd-traffic", type=float, default=None,
                    help="ncu dram bytes per SSD launch, when a capture of the current kernel exists")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
