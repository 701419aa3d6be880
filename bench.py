#!/usr/bin/env python3
"""Benchmark of the GDN speculative-decode verify step on GB300.

One step = one pass of the whole path over one verify window of the serving
workload: the previous window's rollback to its accept lengths (a5, applied on
read) and this window's conv + SiLU, q|k L2 norm, raw gates and chunked gated
delta rule writing the final and K-1 intermediate states (a1..a4), all in one
gdn_verify_resume call.  Workload: B=32 sequences, K=16 window tokens, 16 q/k
heads broadcast to 32 v heads, dk=dv=128 fp32 state, conv width 4 over 8192
channels, bf16 activations and outputs, accept lengths U{1..16}.

Prints one JSON line.  `value` is verified window tokens per second per GDN
layer, summed over ranks (each rank runs its own batch: weak scaling), timed on
the device with CUDA events; `e2e` is the same metric with each step's inputs
copied from pinned host memory and its output copied back inside the timed
region; `roofline` is the verify call's algorithmic bytes over its measured
launch time against the measured HBM copy bandwidth; `cpu_baseline` is the CPU
oracle on the host cores over a bounded sample.  Further objects time the
copying rollback, the token-tree and gated-norm variants, the prompt prefill
and the other verify workloads of the study (plain decode, one-sequence
DFlash-width rounds, batched DSpark width, the 48-layer stack), each beside the
oracle on one host thread and on all of them.

    python bench.py [--steps K] [--warmup W] [--impl gdn|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
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
TRAFFIC_SIDECAR = os.path.join(ROOT, "profiles", "verify_traffic.json")
LAUNCHES_PER_STEP = 2   # verify, q|k history (the rollback is applied on read)
N_WINDOWS = 8           # distinct windows resident in HBM, cycled through the steps
SIDE_MIN_STEPS = 200    # floor of timed work of every side measurement ...
SIDE_MIN_SECONDS = 0.25  # ... in steps and in seconds, whichever is more


def headline_config(world: int) -> dict:
    return {"workload": "GDN verify window: B=32 sequences, K=16 tokens, Hk=16 q/k heads broadcast to Hv=32 v heads, "
                        "dk=dv=128 fp32 state, conv W=4 over C=8192, bf16 activations and outputs, accept lengths "
                        "U{1..16}; per step the previous window's rollback applied on read + verify "
                        "(gdn_verify_resume)",
            "global_batch": world * 32, "seq_len": 16, "parallelism": f"replicas x{world} (no exchange)",
            "l2": "no flush: each step moves 1.2 GB (> 129 MB L2)", "per_step": "gdn_verify_resume"}


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


# ------------------------------------------------------------------ peaks, clocks, profile
def measured_peak_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


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


def profile_traffic(digest: str):
    """DRAM bytes per verify call from the committed ncu sidecar, if it was taken on the
    verify kernels as they are now (same digest of their sources), else None."""
    try:
        with open(TRAFFIC_SIDECAR) as f:
            side = json.load(f)
    except (OSError, ValueError):
        return None
    if side.get("kernel_digest") != digest:
        return None
    return int(side["traffic_bytes_per_launch"])


# ------------------------------------------------------------------ CPU oracle (baselines and reference arm)
def host_cores() -> int:
    """Cores this process may run on (the affinity mask), which is what the oracle pool uses."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_worker(args):
    """Runs in a spawned process: the oracle on one sequence of workload `name` (its layer
    shape with B=1), window after window with the rollback to the window's accept length, for
    `seconds` (or `rounds` windows).  Returns (windows, seconds)."""
    name, seed, seconds, rounds = args
    sys.path.insert(0, ROOT)
    from dataclasses import replace

    from oracle import gdn_oracle as O
    from speculative_decode_verify_gdn_gb300.synth import WORKLOADS, Gen, bf16_bits_to_f32, make_layer, make_round
    w = WORKLOADS[name]
    d = replace(w.dims, B=1)
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


class OraclePool:
    """A pool of spawned processes, one per host core, each single-threaded, running the oracle.
    Created before the first CUDA call (a pool forked after it would hang)."""

    def __init__(self):
        import multiprocessing as mp
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.procs = host_cores()
        self.pool = mp.get_context("spawn").Pool(self.procs)
        self.pool.map(_oracle_worker, [("tiny", 1, 0.0, 1)] * self.procs)   # imports done, warm

    def close(self):
        self.pool.close()
        self.pool.join()

    def rate(self, name: str, seconds: float, procs: int, seed0: int = 7):
        """Window tokens per second of the oracle on `procs` processes (each its own sequence)."""
        from speculative_decode_verify_gdn_gb300.synth import WORKLOADS
        K = WORKLOADS[name].dims.K
        t0 = time.perf_counter()
        res = self.pool.map(_oracle_worker, [(name, seed0 + i, seconds, None) for i in range(procs)], chunksize=1)
        wall = time.perf_counter() - t0
        windows = sum(r[0] for r in res)
        return {"value": windows * K / wall, "unit": "tokens/s per layer", "cores": procs, "kind": "oracle",
                "sample": f"{procs} process(es) x {windows // procs}+ windows of one sequence ({name} layer shape, "
                          f"B=1, K={K}, rollback per window) in {wall:.1f} s, fp64 numpy, one thread each"}

    def both(self, name: str, seconds: float):
        return {"single_thread": self.rate(name, seconds, 1), "all_cores": self.rate(name, seconds, self.procs)}


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


# ------------------------------------------------------------------ device-side helpers
class Ctx:
    """What every device measurement shares: ranks, stream, barrier, status checks."""

    def __init__(self, world, rank, local):
        import torch
        self.world, self.rank, self.local = world, rank, local
        self.dev = torch.device("cuda", local)
        self.stream = torch.cuda.current_stream()

    def barrier(self):
        import torch
        import torch.distributed as dist
        if self.world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_ms(self, ms):
        return max_over_ranks(ms, self.world, self.dev)

    def check(self, what):
        from speculative_decode_verify_gdn_gb300 import gdn
        flags = gdn.gdn_device_status(clear=True)
        if flags:
            raise RuntimeError(f"device status flags {flags} after {what}")

    def timed(self, fn, n, warmup=3, first=0):
        """Mean ms per call of fn(i) over n calls (CUDA events on the stream, after `warmup`
        untimed calls, a barrier on both sides), max over ranks."""
        import torch
        for i in range(warmup):
            fn(first + i)
        self.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for i in range(n):
            fn(first + warmup + i)
        e1.record(self.stream)
        self.barrier()
        return self.max_ms(e0.elapsed_time(e1)) / n

    def side_steps(self, fn, first=0):
        """Calls of fn that make at least SIDE_MIN_STEPS and SIDE_MIN_SECONDS of timed work."""
        probe = self.timed(fn, 10, warmup=3, first=first)
        return max(SIDE_MIN_STEPS, math.ceil(SIDE_MIN_SECONDS * 1e3 / max(probe, 1e-6)))


def _bf(bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def _f32(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


class Windows:
    """N_WINDOWS verify windows of one workload resident on the device (x, a, b, accept lengths)."""

    def __init__(self, g, d, dists, dev, n=N_WINDOWS):
        import torch
        from speculative_decode_verify_gdn_gb300.synth import make_round
        self.rnds = [make_round(g, d, dists) for _ in range(n)]
        self.x = [_bf(r.x, dev) for r in self.rnds]
        self.a = [_bf(r.a, dev) for r in self.rnds]
        self.b = [_bf(r.b, dev) for r in self.rnds]
        self.acc = [torch.from_numpy(r.accept_len).to(dev) for r in self.rnds]
        self.n = n


class Layer:
    """Device buffers of one layer carried in place from window to window."""

    def __init__(self, g, d, dists, dev, out_f32=False):
        import torch
        from speculative_decode_verify_gdn_gb300 import gdn
        from speculative_decode_verify_gdn_gb300.synth import make_layer
        lay = make_layer(g, d, dists)
        self.d = d
        self.dims = gdn.make_dims(d.B, d.K, d.Hk, d.Hv, d.dk, d.dv, d.W, 1.0, 1e-6, int(out_f32))
        self.A_log, self.dt_bias, self.conv_w = _f32(lay.A_log, dev), _f32(lay.dt_bias, dev), _f32(lay.conv_w, dev)
        self.S, self.CS = _f32(lay.state, dev), _f32(lay.conv_state, dev)
        self.SI = (torch.empty((d.B, d.K - 1, d.Hv, d.dv, d.dk), dtype=torch.float32, device=dev)
                   if d.K > 1 else None)
        self.CI = torch.empty((d.B, d.K, d.W - 1, d.C), dtype=torch.float32, device=dev)
        self.out = torch.empty((d.B, d.K, d.Hv, d.dv), dtype=torch.float32 if out_f32 else torch.bfloat16,
                               device=dev)
        self.ws = gdn.alloc_workspace(self.dims, dev)

    def resume(self, win, j, jp, stream, x=None, a=None, b=None, acc=None, out=None):
        """Window j after the rollback of window jp's accept lengths, applied on read."""
        from speculative_decode_verify_gdn_gb300 import gdn
        gdn.gdn_verify_resume(self.dims, win.acc[jp] if acc is None else acc, win.x[j] if x is None else x,
                              win.a[j] if a is None else a, win.b[j] if b is None else b, self.A_log, self.dt_bias,
                              self.conv_w, self.CS, self.CI if self.d.K > 1 else None, None, self.CS, self.CI,
                              self.S, self.SI, None, self.S, self.SI, self.out if out is None else out, self.ws,
                              stream)

    def verify(self, win, j, stream):
        from speculative_decode_verify_gdn_gb300 import gdn
        gdn.gdn_verify_step(self.dims, win.x[j], win.a[j], win.b[j], self.A_log, self.dt_bias, self.conv_w, self.CS,
                            self.CS, self.CI if self.d.K > 1 else None, self.S, self.S, self.SI, self.out, self.ws,
                            stream)

    def rollback(self, win, j, stream):
        from speculative_decode_verify_gdn_gb300 import gdn
        gdn.gdn_rollback(self.dims, win.acc[j], None, self.S, self.SI, None, self.CS, self.CI, stream)


def _hbm(bytes_, ms):
    peak, _ = measured_peak_gbs()
    gbs = bytes_ / (ms * 1e-3) / 1e9
    return gbs, gbs / peak


def run_prefill(args, ctx):
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
    dev = ctx.dev
    dims = gdn.make_dims(d.B, 1, d.Hk, d.Hv, d.dk, d.dv, d.W, 1.0, 1e-6, 0)
    cu = torch.from_numpy(pr.cu).to(dev)
    x, a, b = _bf(pr.x, dev), _bf(pr.a, dev), _bf(pr.b, dev)
    del pr
    S, CS = _f32(lay.state, dev), _f32(lay.conv_state, dev)
    Al, dt, cw = _f32(lay.A_log, dev), _f32(lay.dt_bias, dev), _f32(lay.conv_w, dev)
    out = torch.empty((N, d.Hv, d.dv), dtype=torch.bfloat16, device=dev)
    ws = gdn.alloc_prefill_workspace(dims, N, dev)

    def call(i):
        gdn.gdn_prefill(dims, cu, x, a, b, Al, dt, cw, CS, CS, S, S, out, ws, ctx.stream)

    n = max(3, min(args.steps, 20))
    ms = ctx.timed(call, n, warmup=args.warmup)
    ctx.check("the prefill calls")
    chunks = sum((L + 63) // 64 for L in lens)
    tf = prefill_mma_flops(chunks, d.Hk, d.Hv, d.dk, d.dv) / (ms * 1e-3) / 1e12
    peak, kind = measured_peak_tflops()
    res = {"value": ctx.world * N / (ms * 1e-3), "unit": "tokens/s", "ms_per_call": ms, "calls": n,
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


# ------------------------------------------------------------------ the other verify workloads
def _oracle_obj(cpu, name):
    return None if cpu is None else cpu.get(name)


def run_decode(args, ctx, cpu):
    """Plain decode, K=1, B=1 at the 16/32-head, 128-dim layer: 1000 successive steps with the
    state carried in place, launched one by one and replayed from a CUDA graph."""
    import torch

    from speculative_decode_verify_gdn_gb300.synth import WORKLOADS, Gen
    w = WORKLOADS["decode"]
    d = w.dims
    g = Gen(w.seed + 1000 * ctx.rank)
    lay = Layer(g, d, w.dists, ctx.dev)
    win = Windows(g, d, w.dists, ctx.dev)
    steps = w.rounds

    def step(i):
        lay.verify(win, i % win.n, None)

    eager = ctx.timed(step, steps, warmup=args.warmup)
    ctx.check("the decode steps")
    graph = {"error": None}
    try:
        gs = torch.cuda.Stream(device=ctx.dev)
        gs.wait_stream(ctx.stream)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=gs, capture_error_mode="thread_local"):
            for i in range(win.n):
                lay.verify(win, i, None)
        ctx.stream.wait_stream(gs)
        reps = steps // win.n
        gms = ctx.timed(lambda i: cg.replay(), reps, warmup=3) / win.n
        ctx.check("the decode graph replays")
        graph = {"us_per_step": gms * 1e3, "steps": reps * win.n, "steps_per_graph": win.n}
    except Exception as exc:  # the eager figure stands alone
        graph = {"error": f"{type(exc).__name__}: {exc}"[:300]}
    best = min(eager, graph["us_per_step"] / 1e3) if graph.get("us_per_step") else eager
    vb = verify_bytes(d)
    gbs, frac = _hbm(vb, best)
    return {"workload": w.description + ", 1000 carried steps", "value": ctx.world * d.B * d.K / (best * 1e-3),
            "unit": "tokens/s per layer", "us_per_step_eager": eager * 1e3, "graph": graph, "steps": steps,
            "launches_per_step": 2, "bound": "launch (the step moves 4.5 MB: 0.67 us at the measured HBM peak)",
            "algorithmic_bytes_per_step": vb, "hbm_gbs": gbs, "hbm_frac": frac,
            "step": "gdn_verify_step in place (K=1: no rollback)", "oracle": _oracle_obj(cpu, "decode")}


def run_rounds(args, ctx, cpu, name, rounds, layers=1, what=""):
    """Verify rounds of workload `name` with the rollback of each window applied on the next
    window's read (gdn_verify_resume), `layers` distinct layers per round; tokens/s per layer."""
    import torch

    from speculative_decode_verify_gdn_gb300.synth import WORKLOADS, Gen
    w = WORKLOADS[name]
    d = w.dims
    g = Gen(w.seed + 1000 * ctx.rank)
    lays = [Layer(g, d, w.dists, ctx.dev) for _ in range(layers)]
    win = Windows(g, d, w.dists, ctx.dev)

    def rnd(i):
        for li, lay in enumerate(lays):
            lay.resume(win, (i + li) % win.n, (i + li - 1) % win.n, ctx.stream)

    ms = ctx.timed(rnd, rounds, warmup=min(args.warmup, 3), first=1)
    ctx.check(f"the {name} rounds")
    # one layer: also the rounds replayed from a CUDA graph of one cycle of the windows (the
    # launches through the Python binding can take longer than a one-sequence round on the GPU)
    graph = None
    if layers == 1:
        try:
            gs = torch.cuda.Stream(device=ctx.dev)
            gs.wait_stream(ctx.stream)
            cg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(cg, stream=gs, capture_error_mode="thread_local"):
                for i in range(1, win.n + 1):
                    lays[0].resume(win, i % win.n, (i - 1) % win.n, gs)
            ctx.stream.wait_stream(gs)
            reps = max(1, rounds // win.n)
            gms = ctx.timed(lambda i: cg.replay(), reps, warmup=3) / win.n
            ctx.check(f"the {name} graph replays")
            graph = {"ms_per_round": gms, "rounds": reps * win.n, "rounds_per_graph": win.n}
        except Exception as exc:  # the eager figure stands alone
            graph = {"error": f"{type(exc).__name__}: {exc}"[:300]}
    best = min(ms, graph["ms_per_round"]) if graph and graph.get("ms_per_round") else ms
    per_layer = best / layers
    vb = verify_bytes(d)
    gbs, frac = _hbm(vb, per_layer)
    res = {"workload": w.description + (f", {layers} layers with distinct weights and states" if layers > 1 else ""),
           "value": ctx.world * d.B * d.K / (per_layer * 1e-3), "unit": "tokens/s per layer",
           "ms_per_round": best, "ms_per_round_eager": ms, "rounds": rounds, "layers": layers,
           "gpu_launches_per_round": 2 * layers,
           "algorithmic_bytes_per_layer_round": vb, "hbm_gbs": gbs, "hbm_frac": frac,
           "step": what or "gdn_verify_resume per layer and round (rollback of the previous window on read)",
           "oracle": _oracle_obj(cpu, name)}
    if graph is not None:
        res["graph"] = graph
    if layers > 1 and res["oracle"]:
        o = res["oracle"]["all_cores"]["value"]
        res["oracle_round_ms_extrapolated"] = d.B * d.K * layers / o * 1e3
    del lays, win
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ device arm
def run_gdn(args):
    import torch
    import torch.distributed as dist

    from speculative_decode_verify_gdn_gb300 import gdn
    from speculative_decode_verify_gdn_gb300.build import build_library, verify_kernel_digest
    from speculative_decode_verify_gdn_gb300.synth import WORKLOADS, Gen, make_output_gate, make_tree

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    # the oracle pool starts (spawn) before the first CUDA call
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        pool = OraclePool()
        cpu = {WORKLOAD: {"single_thread": pool.rate(WORKLOAD, args.cpu_seconds / 3, 1),
                          "all_cores": pool.rate(WORKLOAD, args.cpu_seconds, pool.procs)}}
        if not args.headline_only:
            for name in ("decode", "dflash", "dspark"):
                cpu[name] = pool.both(name, args.cpu_seconds / 4)
            cpu["stack48"] = cpu[WORKLOAD]   # one layer of the stack is the serving layer at B=8
        pool.close()

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build_library()
    gdn.load_library()
    ctx = Ctx(world, rank, local)

    w = WORKLOADS[WORKLOAD]
    d = w.dims
    g = Gen(w.seed + 1000 * rank)
    lay = Layer(g, d, w.dists, ctx.dev)
    win = Windows(g, d, w.dists, ctx.dev)
    stream = ctx.stream

    peak, peak_kind = measured_peak_gbs()
    vbytes = verify_bytes(d, out_bytes=2)
    extra = {}
    with ClockSampler(local) as clocks:
        # the copying rollback first (gdn_verify_step then gdn_rollback per step): it also brings the
        # idle GPU up to its working clocks before the headline steps, which follow without a gap
        def copy_step(i):
            j = i % win.n
            lay.verify(win, j, stream)
            lay.rollback(win, j, stream)

        n = ctx.side_steps(copy_step)
        cms = ctx.timed(copy_step, n, warmup=3)
        ctx.check("the copy-rollback steps")
        extra["copy_rollback"] = {"value": job_throughput(d.B * d.K, world, cms), "unit": UNIT, "ms_per_step": cms,
                                  "steps": n, "gpu_launches": 3 * n, "hbm_frac": _hbm(vbytes, cms)[1],
                                  "what": "gdn_verify_step + gdn_rollback (a copy of the accepted intermediate) "
                                          "per step"}

        # the headline: K steps of gdn_verify_resume, each window after the previous window's
        # rollback applied on read
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.warmup):
            lay.resume(win, (i + 1) % win.n, i % win.n, stream)
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ctx.barrier()
        t_start.record(stream)
        for k in range(args.steps):
            i = args.warmup + 1 + k
            evs[k][0].record(stream)
            lay.resume(win, i % win.n, (i - 1) % win.n, stream)
            evs[k][1].record(stream)
        t_end.record(stream)
        ctx.barrier()
    ms = ctx.max_ms(t_start.elapsed_time(t_end))
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    ctx.check("the timed steps")
    value = job_throughput(d.B * d.K * args.steps, world, ms)
    achieved = vbytes / (call_ms / 1e3) / 1e9
    digest = verify_kernel_digest()

    with ClockSampler(local) as clocks_side:
        # e2e: every step's inputs come from pinned host memory and its output goes back,
        # inside the timed region, as a serving loop would run it: double-buffered device inputs
        # and outputs, host-to-device copies on one stream, device-to-host on another, so that
        # step i + 1's inputs and step i - 1's output move while step i computes (events order
        # every reuse)
        e2e = None
        if not args.no_e2e:
            e2e = run_e2e(args, ctx, lay, win)

        if not args.headline_only:
            # token-tree verify on the same shapes: one seeded tree per sequence in which each node
            # continues the previous one with probability 1/2, else branches
            parent = torch.from_numpy(make_tree(Gen(w.seed + 77), d.B, d.K, 0.5)).to(ctx.dev)

            def tree_step(i):
                j = i % win.n
                gdn.gdn_verify_tree(lay.dims, parent, win.x[j], win.a[j], win.b[j], lay.A_log, lay.dt_bias,
                                    lay.conv_w, lay.CS, lay.CS, lay.CI, lay.S, lay.S, lay.SI, lay.out, lay.ws, stream)

            n = ctx.side_steps(tree_step)
            tms = ctx.timed(tree_step, n, warmup=3)
            ctx.check("the tree steps")
            extra["tree_verify"] = {"value": job_throughput(d.B * d.K, world, tms), "unit": "tree nodes/s",
                                    "ms_per_step": tms, "steps": n, "gpu_launches": 2 * n,
                                    "hbm_frac": _hbm(vbytes, tms)[1],
                                    "what": "gdn_verify_tree per step, B=32 trees of 16 nodes (chain continuation "
                                            "1/2)"}

            # verify with the gated RMS output norm fused into the epilogue: z gate [B, K, Hv, dv]
            # bf16 and the norm weight [dv] resident like the other inputs
            zb, nw = make_output_gate(Gen(w.seed + 88), d)
            zg, nwg = _bf(zb, ctx.dev), _f32(nw, ctx.dev)

            def gated_step(i):
                j = i % win.n
                gdn.gdn_verify_gated(lay.dims, win.x[j], win.a[j], win.b[j], lay.A_log, lay.dt_bias, lay.conv_w,
                                     lay.CS, lay.CS, lay.CI, lay.S, lay.S, lay.SI, zg, nwg, 1e-6, lay.out, lay.ws,
                                     stream)

            n = ctx.side_steps(gated_step)
            gms = ctx.timed(gated_step, n, warmup=3)
            ctx.check("the gated steps")
            gbytes = vbytes + zg.numel() * 2 + nwg.numel() * 4
            extra["gated_verify"] = {"value": job_throughput(d.B * d.K, world, gms), "unit": UNIT,
                                     "ms_per_step": gms, "steps": n, "gpu_launches": 2 * n,
                                     "hbm_frac": _hbm(gbytes, gms)[1],
                                     "what": "gdn_verify_gated per step: verify with the gated RMS output norm "
                                             "fused (no rollback)"}
            del lay, win, zg
            torch.cuda.empty_cache()

            extra["workloads"] = {
                "decode": run_decode(args, ctx, cpu),
                "dflash": run_rounds(args, ctx, cpu, "dflash", WORKLOADS["dflash"].rounds),
                "dspark": run_rounds(args, ctx, cpu, "dspark", max(SIDE_MIN_STEPS, WORKLOADS["dspark"].rounds)),
                "stack48": run_rounds(args, ctx, cpu, "stack48", WORKLOADS["stack48"].rounds,
                                      layers=WORKLOADS["stack48"].layers),
            }
            extra["prefill"] = run_prefill(args, ctx)

    cpu_line = None
    if cpu is not None:
        c = cpu[WORKLOAD]
        cpu_line = dict(c["all_cores"], unit=UNIT, single_thread=c["single_thread"], host_cpu_count=os.cpu_count())
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": headline_config(world),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profile_traffic(digest),
                     "kernel": "gdn_verify_resume (gdn_verify_kernel + gdn_qk_history_kernel, the second "
                               "started by programmatic dependent launch inside the first)",
                     "algorithmic_bytes_per_launch": vbytes, "launch_ms": call_ms,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "kernel_digest": digest},
        "cpu_baseline": cpu_line,
        "e2e": e2e,
        "clocks": clocks.summary(),
        "clocks_side_measurements": clocks_side.summary(),
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
    }
    line.update(extra)
    if cpu is not None and not args.headline_only:
        line["cpu_oracle_by_workload"] = cpu
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, ctx, lay, win):
    """The headline step through the C ABI with its inputs (x, a, b, the previous window's
    accept lengths) copied from pinned host memory and its output copied back every step."""
    import torch
    stream = ctx.stream
    hx = [t.cpu().pin_memory() for t in win.x]
    ha = [t.cpu().pin_memory() for t in win.a]
    hb = [t.cpu().pin_memory() for t in win.b]
    hacc = [t.cpu().pin_memory() for t in win.acc]
    hout = [torch.empty(lay.out.shape, dtype=lay.out.dtype).pin_memory() for _ in range(2)]
    X2 = [torch.empty_like(win.x[0]) for _ in range(2)]
    A2 = [torch.empty_like(win.a[0]) for _ in range(2)]
    B2 = [torch.empty_like(win.b[0]) for _ in range(2)]
    ACC2 = [torch.empty_like(win.acc[0]) for _ in range(2)]
    OUT2 = [lay.out, torch.empty_like(lay.out)]
    h2d_s, d2h_s = torch.cuda.Stream(device=ctx.dev), torch.cuda.Stream(device=ctx.dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for q in range(2):
        comp_done[q].record(stream)
        d2h_done[q].record(stream)

    def e2e_step(i):
        j, jp, q = i % win.n, (i - 1) % win.n, i % 2
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(comp_done[q])  # step i - 2 is done with these buffers
            X2[q].copy_(hx[j], non_blocking=True)
            A2[q].copy_(ha[j], non_blocking=True)
            B2[q].copy_(hb[j], non_blocking=True)
            ACC2[q].copy_(hacc[jp], non_blocking=True)
            h2d_done[q].record(h2d_s)
        stream.wait_event(h2d_done[q])
        stream.wait_event(d2h_done[q])  # step i - 2's output has left OUT2[q]
        lay.resume(win, j, jp, stream, x=X2[q], a=A2[q], b=B2[q], acc=ACC2[q], out=OUT2[q])
        comp_done[q].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(comp_done[q])
            hout[q].copy_(OUT2[q], non_blocking=True)
            d2h_done[q].record(d2h_s)

    n = max(args.steps, ctx.side_steps(e2e_step, first=1))
    for i in range(3):
        e2e_step(1 + i)
    ctx.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_s.wait_event(e0)  # the first step's copies start inside the timed region
    for i in range(n):
        e2e_step(4 + i)
    for q in range(2):
        stream.wait_event(d2h_done[q])  # ... and the last outputs have arrived before it ends
    e1.record(stream)
    ctx.barrier()
    ems = ctx.max_ms(e0.elapsed_time(e1))
    ctx.check("the e2e steps")
    d = lay.d
    bi = sum(t.numel() * t.element_size() for t in (hx[0], ha[0], hb[0], hacc[0]))
    bo = hout[0].numel() * hout[0].element_size()
    return {"value": job_throughput(d.B * d.K * n, ctx.world, ems), "unit": UNIT, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "steps": n,
            "what": "gdn_verify_resume per step through the C ABI, x, a, b and the previous window's accept lengths "
                    "copied from pinned host memory and the output copied back every step, copies on their own "
                    "streams overlapping the neighbouring steps' kernels (double-buffered)"}


# ------------------------------------------------------------------ reference arm (the CPU oracle)
def run_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    pool = OraclePool()
    # a step is the serving step's work: B = 32 sequences' K=16 windows (+ rollback), spread over the
    # processes; shrunk (and said so) if the run would take more than about 150 s
    t_cal = _oracle_worker((WORKLOAD, 3, 0.0, 1))[1]
    procs = pool.procs
    total = args.steps * 32
    while total > procs and total * t_cal / procs > 150.0:
        total //= 2
    per = [(total + i) // procs for i in range(procs)]
    pool.pool.map(_oracle_worker, [(WORKLOAD, 11 + i, 0.0, max(1, args.warmup * 32 // procs)) for i in range(procs)])
    t0 = time.perf_counter()
    res = pool.pool.map(_oracle_worker, [(WORKLOAD, 11 + i, 0.0, max(1, per[i])) for i in range(procs)], chunksize=1)
    wall = time.perf_counter() - t0
    pool.close()
    windows = sum(r[0] for r in res)
    value = windows * 16 / wall
    sample = (f"{windows} windows of one sequence each ({windows / 32:.1f} steps of the B=32 K=16 workload, 16 tokens "
              f"+ rollback per window), fp64 numpy oracle over {procs} single-threaded processes")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3 / max(windows / 32, 1e-9),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(world),
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": procs, "kind": "oracle", "sample": sample,
                         "host_cpu_count": os.cpu_count()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_only(args):
    """One measurement alone (for profiling under ncu): `verify` = the headline steps without
    the baselines, e2e or side measurements; `prefill` = the prefill calls."""
    import torch

    from speculative_decode_verify_gdn_gb300 import gdn
    from speculative_decode_verify_gdn_gb300.build import build_library
    from speculative_decode_verify_gdn_gb300.synth import WORKLOADS, Gen

    torch.cuda.set_device(0)
    build_library()
    gdn.load_library()
    ctx = Ctx(1, 0, 0)
    if args.only == "prefill":
        print(json.dumps({"prefill": run_prefill(args, ctx)}), flush=True)
        return
    w = WORKLOADS[WORKLOAD]
    lay = Layer(Gen(w.seed), w.dims, w.dists, ctx.dev)
    win = Windows(Gen(w.seed + 1), w.dims, w.dists, ctx.dev)
    if args.only == "verify":
        ms = ctx.timed(lambda i: lay.resume(win, i % win.n, (i - 1) % win.n, ctx.stream), args.steps,
                       warmup=args.warmup, first=1)
    else:
        from speculative_decode_verify_gdn_gb300.synth import make_tree
        parent = torch.from_numpy(make_tree(Gen(w.seed + 77), w.dims.B, w.dims.K, 0.5)).to(ctx.dev)

        def tree_step(i):
            j = i % win.n
            gdn.gdn_verify_tree(lay.dims, parent, win.x[j], win.a[j], win.b[j], lay.A_log, lay.dt_bias, lay.conv_w,
                                lay.CS, lay.CS, lay.CI, lay.S, lay.S, lay.SI, lay.out, lay.ws, ctx.stream)
        ms = ctx.timed(tree_step, args.steps, warmup=args.warmup)
    ctx.check(args.only)
    print(json.dumps({args.only: {"ms_per_step": ms, "steps": args.steps}}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="time the headline, its e2e and the copying rollback only")
    ap.add_argument("--only", choices=["prefill", "verify", "tree"], default=None,
                    help="run one measurement alone (for profiling) and print its JSON object")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_gdn(args)


if __name__ == "__main__":
    main()
