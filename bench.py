#!/usr/bin/env python3
"""Benchmark of the GDN speculative-decode verify step on GB300.

One step = one pass of the whole path over one verify window of the serving
workload: gdn_verify_step (conv + SiLU, q|k L2 norm, raw gates, chunked gated
delta rule writing the final and K-1 intermediate states) followed by
gdn_rollback to synthetic accept lengths U{1..K}.  Workload: B=32 sequences,
K=16 window tokens, 16 q/k heads broadcast to 32 v heads, dk=dv=128 fp32 state,
conv width 4 over 8192 channels, bf16 activations and outputs.

Prints one JSON line.  `value` is verified window tokens per second per GDN
layer, summed over ranks (each rank runs its own batch: weak scaling), timed on
the device with CUDA events; `e2e` is the same metric with each step's inputs
copied from pinned host memory and its output copied back inside the timed
region; `roofline` is the verify kernel's algorithmic bytes over its measured
launch time against the measured HBM copy bandwidth; `cpu_baseline` is the CPU
oracle on the host cores over a bounded sample.

    python bench.py [--steps K] [--warmup W] [--impl gdn|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified tokens/s per GDN layer (K=16,B=32) and HBM GB/s as % of GB300 peak"
UNIT = "tokens/s"
WORKLOAD = "serve16"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "gdn_verify_kernel_serve16.md")
LAUNCHES_PER_STEP = 3   # q/k prologue, state stream, rollback


# ------------------------------------------------------------------ algorithmic bytes
def verify_bytes(d, out_bytes: int = 2) -> int:
    """Bytes the verify step must move at minimum for one launch over B sequences.

    Per sequence: state read (S), K states written (K-1 intermediates + final),
    conv history read and K conv snapshots written, x (bf16), a and b (bf16),
    outputs.  Per launch: conv taps, A_log and dt_bias.
    """
    S = d.Hv * d.dv * d.dk * 4
    ccv = (d.W - 1) * d.C * 4
    per_seq = S + d.K * S + ccv + d.K * ccv + d.K * d.C * 2 + d.K * 2 * d.Hv * 2 + d.K * d.Hv * d.dv * out_bytes
    per_launch = d.W * d.C * 4 + 2 * d.Hv * 4
    return d.B * per_seq + per_launch


PREFILL_LENS = [8192] * 8  # prompts of the prefill measurement


def prefill_mma_flops(n_chunks: int, Hk: int, Hv: int, dk: int, dv: int) -> int:
    """bf16 tensor-core FLOPs one prefill call issues, three MMAs (hi.hi, hi.lo, lo.hi) per
    product.  State kernel, per (chunk, v-head, 64 state rows): S [k^|q^]^T (2 x 64 x 64 x dk),
    u = r W^T and o = u MQ^T (64 x 64 x 64 each) and the state update (64 x dk x 64).  Chunk
    kernel, per (chunk, q/k head): the Gram products [k^; q^] k^T (128 x 64 x dk)."""
    state = 3 * (2 * 64 * 64 * dk + 2 * 64 * 64 * 64 + 64 * dk * 64) * Hv * (dv // 64)
    gram = 3 * (128 * 64 * dk) * Hk
    return 2 * (state + gram) * n_chunks


def measured_peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def run_prefill(args, world, dev, barrier, max_over_ranks):
    """Prefill of PREFILL_LENS prompts at the serving layer shape through gdn_prefill, inputs
    resident; tokens/s over `steps` calls after `warmup`."""
    import torch

    from speculative_decode_verify_gdn_gb300 import gdn
    from speculative_decode_verify_gdn_gb300.synth import WORKLOADS, Dims, Gen, make_layer, make_prompts

    w = WORKLOADS[WORKLOAD]
    lens = PREFILL_LENS
    d = Dims(B=len(lens), K=1, Hk=w.dims.Hk, Hv=w.dims.Hv, dk=w.dims.dk, dv=w.dims.dv)
    g = Gen(w.seed + 99)
    lay = make_layer(g, d, w.dists)
    pr = make_prompts(g, d, lens, w.dists)
    N = int(pr.cu[-1])
    dims = gdn.make_dims(d.B, 1, d.Hk, d.Hv, d.dk, d.dv, d.W, 1.0, 1e-6, 0)

    def bf(b):
        return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(dev).view(torch.bfloat16)

    def f32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)

    cu = torch.from_numpy(pr.cu).to(dev)
    x, a, b = bf(pr.x), bf(pr.a), bf(pr.b)
    S, CS = f32(lay.state), f32(lay.conv_state)
    Al, dt, cw = f32(lay.A_log), f32(lay.dt_bias), f32(lay.conv_w)
    out = torch.empty((N, d.Hv, d.dv), dtype=torch.bfloat16, device=dev)
    ws = gdn.alloc_prefill_workspace(dims, N, dev)
    stream = torch.cuda.current_stream()

    def call():
        gdn.gdn_prefill(dims, cu, x, a, b, Al, dt, cw, CS, CS, S, S, out, ws, stream)

    n = max(3, min(args.steps, 20))
    for _ in range(args.warmup):
        call()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        call()
    e1.record(stream)
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / n
    if gdn.gdn_device_status(clear=True):
        raise RuntimeError("device status flags after the prefill calls")
    chunks = sum((L + 63) // 64 for L in lens)
    tf = prefill_mma_flops(chunks, d.Hk, d.Hv, d.dk, d.dv) / (ms * 1e-3) / 1e12
    peak, kind = measured_peak_tflops()
    res = {"value": world * N / (ms * 1e-3), "unit": "tokens/s", "ms_per_call": ms, "calls": n,
           "gpu_launches": 3 * n,
           "workload": f"{len(lens)} prompts x {lens[0]} tokens, Hk={d.Hk} Hv={d.Hv} dk={d.dk} dv={d.dv}, "
                       "bf16 inputs and outputs, f32 state, in place",
           "tensor": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                      "peak_source": f"{kind} (MEASURED_PEAKS.json bf16_tflops)",
                      "what": "bf16 MMA FLOPs of the state and chunk kernels over the whole call "
                              "(all three kernels)"},
           "what": "gdn_prefill per call: cu_seqlens check, per-chunk q/k kernel, tensor-core state pass"}
    del ws, out, x
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ peaks, clocks, profile
def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        # samples under load: within 30% of the busiest clock seen (idle edges excluded)
        top = max(sm) if sm else 0
        loaded = [s for s in sm if s >= 0.7 * top] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def profile_traffic(kernel_digest: str):
    """DRAM bytes per verify launch from the committed ncu summary, if taken on these kernels."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    m_d = re.search(r"kernel_digest:\s*([0-9a-f]+)", text)
    m_t = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not m_d or not m_t or m_d.group(1) != kernel_digest:
        return None
    return int(m_t.group(1))


# ------------------------------------------------------------------ CPU oracle (baseline / reference arm)
def _oracle_worker(args):
    """Runs in a spawned process: oracle rounds of one sequence for `seconds` (or `rounds`)."""
    seed, n_tok, seconds, rounds = args
    sys.path.insert(0, ROOT)
    from oracle import gdn_oracle as O
    from speculative_decode_verify_gdn_gb300.synth import WORKLOADS, Dims, Gen, bf16_bits_to_f32, make_layer, make_round
    w = WORKLOADS[WORKLOAD]
    d = Dims(B=1, K=n_tok, Hk=w.dims.Hk, Hv=w.dims.Hv, dk=w.dims.dk, dv=w.dims.dv, W=w.dims.W)
    g = Gen(seed)
    lay = make_layer(g, d, w.dists)
    rnds = [make_round(g, d, w.dists) for _ in range(4)]
    S, H = lay.state.astype(np.float64), lay.conv_state.astype(np.float64)
    done, t0 = 0, time.perf_counter()
    while True:
        r = rnds[done % 4]
        res = O.verify_step(d, bf16_bits_to_f32(r.x), bf16_bits_to_f32(r.a), bf16_bits_to_f32(r.b), lay.A_log,
                            lay.dt_bias, lay.conv_w, H, S)
        S, H = O.rollback(r.accept_len, S, res["states"], H, res["conv_inter"])
        done += 1
        el = time.perf_counter() - t0
        if (rounds is not None and done >= rounds) or (rounds is None and el >= seconds):
            return done, el


def oracle_pool_size() -> int:
    return max(1, min(os.cpu_count() or 1, 16))


def cpu_oracle_throughput(seconds: float = 12.0, n_tok: int = 16):
    """Tokens/s of the oracle on the host cores: one process per core, each on its own sequence."""
    import multiprocessing as mp
    procs = oracle_pool_size()
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs) as pool:
        pool.map(_oracle_worker, [(7 + i, n_tok, 0.0, 1) for i in range(procs)])   # import + warm
        t0 = time.perf_counter()
        res = pool.map(_oracle_worker, [(7 + i, n_tok, seconds, None) for i in range(procs)])
        wall = time.perf_counter() - t0
    rounds = sum(r[0] for r in res)
    return rounds * n_tok / wall, procs, rounds, wall


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of each rank's `x` (the slowest rank sets the job's time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms / 1e3)


# ------------------------------------------------------------------ device arm
def run_gdn(args):
    import torch
    import torch.distributed as dist

    from speculative_decode_verify_gdn_gb300 import gdn
    from speculative_decode_verify_gdn_gb300.build import build_library, kernel_source_digest
    from speculative_decode_verify_gdn_gb300.runtime import GdnLayerState
    from speculative_decode_verify_gdn_gb300.synth import (WORKLOADS, Gen, make_layer, make_output_gate, make_round,
                                                            make_tree)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    # the oracle pool starts (spawn) before the first CUDA call
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tps, procs, rounds, wall = cpu_oracle_throughput(args.cpu_seconds)
        cpu = {"value": tps, "unit": UNIT, "cores": procs, "kind": "oracle",
               "sample": f"{procs} processes x {rounds // max(procs, 1)}+ rounds of one sequence "
                         f"(K=16 window + rollback, 32 v-heads, 128x128 state) in {wall:.1f}s, fp64 numpy"}

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build_library()
    gdn.load_library()

    w = WORKLOADS[WORKLOAD]
    d = w.dims
    g = Gen(w.seed + 1000 * rank)
    lay = make_layer(g, d, w.dists)
    st = GdnLayerState.create(d, lay, device=f"cuda:{local}", out_f32=False)
    n_in = 8  # distinct windows cycled through the steps, resident in HBM
    rnds = [make_round(g, d, w.dists) for _ in range(n_in)]
    dev = st.x.device
    xs = [torch.from_numpy(r.x.view(np.int16)).to(dev).view(torch.bfloat16) for r in rnds]
    as_ = [torch.from_numpy(r.a.view(np.int16)).to(dev).view(torch.bfloat16) for r in rnds]
    bs = [torch.from_numpy(r.b.view(np.int16)).to(dev).view(torch.bfloat16) for r in rnds]
    accs = [torch.from_numpy(r.accept_len).to(dev) for r in rnds]
    stream = torch.cuda.current_stream()
    dims = st.dims
    S0, CS, CI, SI, OUT, WS = st.states[0], st.conv_states[0], st.conv_inter, st.state_inter, st.out, st.workspace

    def step(i, ev=None):
        j = i % n_in
        if ev is not None:
            ev[0].record(stream)
        gdn.gdn_verify_step(dims, xs[j], as_[j], bs[j], st.A_log, st.dt_bias, st.conv_w, CS, CS, CI, S0, S0, SI,
                            OUT, WS, stream)
        if ev is not None:
            ev[1].record(stream)
        gdn.gdn_rollback(dims, accs[j], None, S0, SI, None, CS, CI, stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup):
        step(i)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local) as clocks:
        t_start.record(stream)
        for i in range(args.steps):
            step(args.warmup + i, evs[i])
        t_end.record(stream)
        barrier()
    ms = t_start.elapsed_time(t_end)
    verify_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    flags = gdn.gdn_device_status(clear=True)
    if flags:
        raise RuntimeError(f"device status flags {flags} after the timed steps")
    ms = max_over_ranks(ms, world, dev)
    value = job_throughput(d.B * d.K * args.steps, world, ms)

    # the same steps with each window's rollback applied on the next verify's read
    # (gdn_verify_resume): no rollback copy, one verify call per step
    def resume_step(i):
        j, jp = i % n_in, (i - 1) % n_in
        gdn.gdn_verify_resume(dims, accs[jp], xs[j], as_[j], bs[j], st.A_log, st.dt_bias, st.conv_w, CS, CI, None,
                              CS, CI, S0, SI, None, S0, SI, OUT, WS, stream)

    for i in range(args.warmup):
        resume_step(i + 1)
    barrier()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for i in range(args.steps):
        resume_step(args.warmup + 1 + i)
    r1.record(stream)
    barrier()
    rms = max_over_ranks(r0.elapsed_time(r1), world, dev)
    resume = {"value": job_throughput(d.B * d.K * args.steps, world, rms), "unit": UNIT,
              "ms_per_step": rms / args.steps, "gpu_launches": 2 * args.steps,
              "what": "gdn_verify_resume per step: the previous window's rollback applied on read, no copy"}
    if gdn.gdn_device_status(clear=True):
        raise RuntimeError("device status flags after the resume steps")

    # token-tree verify (gdn_verify_tree) on the same shapes: one seeded tree per sequence in
    # which each node continues the previous one with probability 1/2, else branches
    parent = torch.from_numpy(make_tree(Gen(w.seed + 77), d.B, d.K, 0.5)).to(dev)

    def tree_step(i):
        j = i % n_in
        gdn.gdn_verify_tree(dims, parent, xs[j], as_[j], bs[j], st.A_log, st.dt_bias, st.conv_w, CS, CS, CI, S0, S0,
                            SI, OUT, WS, stream)

    for i in range(args.warmup):
        tree_step(i)
    barrier()
    r0.record(stream)
    n_tree = max(3, args.steps // 5)
    for i in range(n_tree):
        tree_step(i)
    r1.record(stream)
    barrier()
    tms = max_over_ranks(r0.elapsed_time(r1), world, dev)
    tree = {"value": job_throughput(d.B * d.K * n_tree, world, tms), "unit": "tree nodes/s",
            "ms_per_step": tms / n_tree, "steps": n_tree, "gpu_launches": 2 * n_tree,
            "hbm_frac": verify_bytes(d, out_bytes=2) / (tms / n_tree * 1e-3) / 1e9 / measured_peak_gbs()[0],
            "what": "gdn_verify_tree per step, B=32 trees of 16 nodes (chain continuation 1/2)"}
    if gdn.gdn_device_status(clear=True):
        raise RuntimeError("device status flags after the tree steps")

    # verify with the gated RMS output norm fused into the epilogue (gdn_verify_gated): z gate
    # [B, K, Hv, dv] bf16 and the norm weight [dv] resident like the other inputs
    zb, nw = make_output_gate(Gen(w.seed + 88), d)
    zg = torch.from_numpy(zb.view(np.int16)).to(dev).view(torch.bfloat16)
    nwg = torch.from_numpy(nw).to(dev)

    def gated_step(i):
        j = i % n_in
        gdn.gdn_verify_gated(dims, xs[j], as_[j], bs[j], st.A_log, st.dt_bias, st.conv_w, CS, CS, CI, S0, S0, SI,
                             zg, nwg, 1e-6, OUT, WS, stream)

    for i in range(args.warmup):
        gated_step(i)
    barrier()
    r0.record(stream)
    n_gated = max(3, args.steps // 5)
    for i in range(n_gated):
        gated_step(i)
    r1.record(stream)
    barrier()
    gms = max_over_ranks(r0.elapsed_time(r1), world, dev)
    gbytes = verify_bytes(d, out_bytes=2) + zg.numel() * 2 + nwg.numel() * 4
    gated = {"value": job_throughput(d.B * d.K * n_gated, world, gms), "unit": UNIT,
             "ms_per_step": gms / n_gated, "steps": n_gated, "gpu_launches": 2 * n_gated,
             "hbm_frac": gbytes / (gms / n_gated * 1e-3) / 1e9 / measured_peak_gbs()[0],
             "what": "gdn_verify_gated per step: verify with the gated RMS output norm fused (no rollback)"}
    if gdn.gdn_device_status(clear=True):
        raise RuntimeError("device status flags after the gated steps")

    prefill = run_prefill(args, world, dev, barrier, max_over_ranks)

    # e2e: every step's inputs come from pinned host memory and its output goes back, inside the
    # timed region, as a serving loop would run it: double-buffered device inputs and outputs,
    # host-to-device copies on one stream, device-to-host on another, so that step i + 1's
    # inputs and step i - 1's output move while step i computes (events order every reuse)
    e2e = None
    if not args.no_e2e:
        hx = [torch.from_numpy(r.x.view(np.int16)).view(torch.bfloat16).pin_memory() for r in rnds]
        ha = [torch.from_numpy(r.a.view(np.int16)).view(torch.bfloat16).pin_memory() for r in rnds]
        hb = [torch.from_numpy(r.b.view(np.int16)).view(torch.bfloat16).pin_memory() for r in rnds]
        hacc = [torch.from_numpy(r.accept_len).pin_memory() for r in rnds]
        hout = [torch.empty(OUT.shape, dtype=OUT.dtype).pin_memory() for _ in range(2)]
        X2 = [st.x, torch.empty_like(st.x)]
        A2 = [st.a, torch.empty_like(st.a)]
        B2 = [st.b, torch.empty_like(st.b)]
        ACC2 = [st.accept_len, torch.empty_like(st.accept_len)]
        OUT2 = [OUT, torch.empty_like(OUT)]
        h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        for q in range(2):
            comp_done[q].record(stream)
            d2h_done[q].record(stream)

        def e2e_step(i):
            j, q = i % n_in, i % 2
            with torch.cuda.stream(h2d_s):
                h2d_s.wait_event(comp_done[q])  # step i - 2 is done with these buffers
                X2[q].copy_(hx[j], non_blocking=True)
                A2[q].copy_(ha[j], non_blocking=True)
                B2[q].copy_(hb[j], non_blocking=True)
                ACC2[q].copy_(hacc[j], non_blocking=True)
                h2d_done[q].record(h2d_s)
            stream.wait_event(h2d_done[q])
            stream.wait_event(d2h_done[q])  # step i - 2's output has left OUT2[q]
            gdn.gdn_verify_step(dims, X2[q], A2[q], B2[q], st.A_log, st.dt_bias, st.conv_w, CS, CS, CI, S0, S0, SI,
                                OUT2[q], WS, stream)
            gdn.gdn_rollback(dims, ACC2[q], None, S0, SI, None, CS, CI, stream)
            comp_done[q].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(comp_done[q])
                hout[q].copy_(OUT2[q], non_blocking=True)
                d2h_done[q].record(d2h_s)

        n_e2e = max(3, min(args.steps, args.e2e_steps))
        for i in range(args.warmup):
            e2e_step(i)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_s.wait_event(e0)  # the first step's copies start inside the timed region
        for i in range(n_e2e):
            e2e_step(i)
        for q in range(2):
            stream.wait_event(d2h_done[q])  # ... and the last outputs have arrived before it ends
        e1.record(stream)
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1), world, dev)
        bi = sum(t.numel() * t.element_size() for t in (hx[0], ha[0], hb[0], hacc[0]))
        bo = hout[0].numel() * hout[0].element_size()
        e2e = {"value": job_throughput(d.B * d.K * n_e2e, world, ems), "unit": UNIT, "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "steps": n_e2e,
               "what": "gdn_verify_step + gdn_rollback per step through the C ABI, inputs copied from pinned host "
                       "memory and the output copied back every step, copies on their own streams overlapping "
                       "the neighbouring steps' kernels (double-buffered)"}

    peak, peak_kind = measured_peak_gbs()
    vbytes = verify_bytes(d, out_bytes=2)
    achieved = vbytes / (verify_ms / 1e3) / 1e9
    digest = kernel_source_digest()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "GDN verify window: B=32 sequences, K=16 tokens, Hk=16 q/k heads broadcast to "
                               "Hv=32 v heads, dk=dv=128 fp32 state, conv W=4 over C=8192, bf16 activations "
                               "and outputs, accept lengths U{1..16}, verify + rollback per step",
                   "global_batch": world * d.B, "seq_len": d.K, "parallelism": f"replicas x{world} (no exchange)",
                   "l2": "no flush: each step moves 1.2 GB (> 129 MB L2)", "per_step": "gdn_verify_step + gdn_rollback"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profile_traffic(digest),
                     "kernel": "gdn_verify_step (gdn_qk_prologue_kernel + gdn_state_stream_kernel, overlapped)",
                     "algorithmic_bytes_per_launch": vbytes, "launch_ms": verify_ms,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "kernel_digest": digest},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks.summary(),
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "zero_copy_rollback": resume,
        "tree_verify": tree,
        "gated_verify": gated,
        "prefill": prefill,
    }
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ reference arm (the CPU oracle)
def run_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import multiprocessing as mp
    procs = oracle_pool_size()
    # calibrate: one full K=16 window of one sequence per step, shrunk if the run would be long
    t_cal = _oracle_worker((3, 16, 0.0, 1))[1]
    budget = 150.0
    n_tok = 16
    while n_tok > 1 and (args.steps + args.warmup) * t_cal * n_tok / 16 / procs > budget:
        n_tok //= 2
    ctx = mp.get_context("spawn")
    per = [(args.steps + i) // procs for i in range(procs)]
    with ctx.Pool(procs) as pool:
        pool.map(_oracle_worker, [(11 + i, n_tok, 0.0, max(1, args.warmup // procs)) for i in range(procs)])
        t0 = time.perf_counter()
        res = pool.map(_oracle_worker, [(11 + i, n_tok, 0.0, max(1, per[i])) for i in range(procs)])
        wall = time.perf_counter() - t0
    steps = sum(r[0] for r in res)
    value = steps * n_tok / wall
    sample = (f"{steps} steps, each one sequence x {n_tok}-token window (+ rollback) of the B=32 K=16 workload, "
              f"fp64 numpy oracle over {procs} processes")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3 / max(steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "GDN verify window: B=32 sequences, K=16 tokens, Hk=16 q/k heads broadcast to "
                               "Hv=32 v heads, dk=dv=128 fp32 state, conv W=4 over C=8192, bf16 activations "
                               "and outputs, accept lengths U{1..16}, verify + rollback per step",
                   "global_batch": 32, "seq_len": 16, "parallelism": "host cores"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": procs, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_prefill_only(args):
    import torch

    from speculative_decode_verify_gdn_gb300 import gdn
    from speculative_decode_verify_gdn_gb300.build import build_library

    torch.cuda.set_device(0)
    build_library()
    gdn.load_library()
    dev = torch.device("cuda", 0)
    res = run_prefill(args, 1, dev, torch.cuda.synchronize, lambda v, world, dev: v)
    print(json.dumps({"prefill": res}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--e2e-steps", type=int, default=1000)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", choices=["prefill"], default=None,
                    help="run one side measurement alone (for profiling) and print its JSON object")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.only == "prefill":
        run_prefill_only(args)
    else:
        run_gdn(args)


if __name__ == "__main__":
    main()
