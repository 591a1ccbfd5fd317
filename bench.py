#!/usr/bin/env python
"""Throughput of the MoK layer (forward + backward) on GB300.

One step = one pass of the whole hot path over one batch: build the schedule
from the batch's routing, the forward (gate/up + SwiGLU, down + router scale +
scatter, shared expert, combine) and the backward (dgrad, SwiGLU backward,
router-weight grad, grouped wgrad, shared expert, fixed-order reductions).
In MXFP8 workloads the step also prequantises the weights (they change every
optimiser step).

`python bench.py [--gpus N --steps K --warmup W] [--workload NAME]` prints one
JSON line.  Under torchrun each rank runs its own batch of the workload (data
parallel, no collective on the data path: weak scaling); the time is the max
over ranks.  `--impl reference` times the CPU oracle instead (rank 0 only).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "large_T65536"
METRIC = "MoE layer fwd+bwd tokens/s (TFLOP/s and % of GB300 dense tensor peak alongside)"
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2


# ----------------------------------------------------------------- helpers
def layer_flops(c):
    """Algorithmic FLOP of one fwd+bwd (padding rows excluded): forward
    6*H*I per routed row + 6*H*I_s per token; backward twice the forward."""
    fwd = 6.0 * c["T"] * c["k"] * c["H"] * c["I"] + 6.0 * c["T"] * c["H"] * c["I_s"]
    return fwd, 3.0 * fwd


def stage_flops(c):
    """Algorithmic FLOP of each GEMM stage (same names as the C ABI stages)."""
    T, k, H, I, Is = c["T"], c["k"], c["H"], c["I"], c["I_s"]
    R = T * k
    return {
        "fwd_gateup": 4.0 * R * H * I, "fwd_down": 2.0 * R * I * H,
        "fwd_shared_gateup": 4.0 * T * H * Is, "fwd_shared_down": 2.0 * T * Is * H,
        "bwd_down": 2.0 * R * H * I, "bwd_wgrad_down": 2.0 * R * H * I,
        "bwd_wgrad_gateup": 4.0 * R * H * I, "bwd_dgrad_gateup": 4.0 * R * H * I,
        "bwd_shared_down": 2.0 * T * H * Is, "bwd_shared_wgrad_down": 2.0 * T * H * Is,
        "bwd_shared_wgrad_gateup": 4.0 * T * H * Is, "bwd_shared_dgrad": 4.0 * T * H * Is,
    }


FWD_GEMM_STAGES = ("fwd_gateup", "fwd_down", "fwd_shared_gateup", "fwd_shared_down")
LONG_STEP_MS = 20.0   # steps longer than this run the tensor cores under the power cap


def dist_env():
    """(rank, world size, local rank) of this process as torchrun sets them."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value, world, device):
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if world <= 1:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(T, world, steps, total_ms):
    """Whole-job throughput: every rank processes its own T tokens per step
    (weak scaling); total_ms is the slowest rank's time for all steps."""
    return T * max(world, 1) * steps / (total_ms / 1e3)


def launches_per_step(c, windows=1, ring=False):
    """Kernels of this library launched by one step (mirrors the C ABI's sequence
    with the default permuted dispatch).  With a macrobatch ring (forward and
    backward alike) the routed experts run in `windows` windows, each with its
    own dispatch and routed GEMMs, and each call builds a schedule view per
    window when there is more than one."""
    mode = c["mode"]
    mx = mode in ("mxfp8", "mxfp8_full")
    full = mode == "mxfp8_full"
    shared = c["I_s"] > 0
    W = windows
    n = 3                                   # schedule: count, scan, scatter
    n += 1 if -(-c["T"] * c["k"] // 1024) > 64 else 0   # and per-expert chunk offsets (large schedules)
    n += 2 * W if W > 1 else 0              # window views, forward and backward
    n += 1 + 2 * W + 1                      # status hand-over, routed gate/up + down, combine
    if shared:
        n += 2
    if mx:
        n += 3 + (3 if shared else 0)       # weight prequantisation (every step)
        n += 1                              # weight scales into the tensor-core layout (one launch)
    n += W                                  # x into schedule order (MXFP8: quantised, token order too)
    if mx:
        n += W                              # and its scales into the tensor-core layout
    if full:                                # (the prequantisation above writes both weight copies)
        n += 1                              # transposed weights' scales into the tensor-core layout
        n += 2 * W + (2 if shared else 0)   # x transposed; dy rows + transposed (schedule, token order)
        n += 4 * W + (4 if shared else 0)   # GEMMs (the SwiGLU backward writes its MXFP8 outputs)
        n += 2                              # combine dx, reduce d_w
        return n
    # dy rows into schedule order; x's rows too when the forward's copy does
    # not span the schedule (a ring)
    n += W * (2 if ring else 1)
    n += 4 * W + 2                          # routed dgrad/wgrad x4, combine dx, reduce d_w
    if shared:
        n += 4
    return n


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash(kernel="gemm_kernel"):
    """Hash of the sources a GEMM kernel is built from: the bf16 engine
    (gemm_kernel) from gemm.cuh and ptx.cuh, the block-scaled one
    (gemm_mx_kernel) from those and gemm_mx.cuh."""
    names = ["gemm.cuh", "ptx.cuh"] + (["gemm_mx.cuh"] if kernel.startswith("gemm_mx_kernel") else [])
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "mixture_experts_layer_mok_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, stage):
    """DRAM bytes per launch of the stage's kernel from a committed ncu summary,
    valid only while the GEMM kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
        ent = rec[workload][stage]
        if ent["kernel_source"] == kernel_source_hash(ent["kernel"]):
            return ent["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = str(gpu_index)
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", self.gpu], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons, pw = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------- oracle timing
class OracleSample:
    """The CPU oracle (float64 NumPy) timed on units of the workload that
    together make up a whole layer, each with the amortisation it has in a
    whole-layer run:

    - a routed unit is forward + backward of one expert over the rows routed
      to it (a k = 1 layer over those rows with their router weights; at most
      ``max_rows`` of them).  In the MXFP8 modes the oracle quantises the
      expert's weights inside the call, once per unit, as a whole-layer call
      does once per expert;
    - a shared unit is the shared expert alone over as many tokens.

    A token costs k routed rows and one shared row, so tokens/s =
    1 / (k * s_routed + s_shared), with s_* the measured seconds per row of
    each kind.  Units run one shared to k routed (experts in turn).  Each
    unit's inputs are cut out and widened to float64 before its timed call."""

    def __init__(self, inp, mode, max_rows):
        import oracle

        self.inp = inp
        self.k = inp.top_experts.shape[1]
        self.E = inp.w_gate.shape[0]
        self.shared = inp.ws_gate is not None
        self.max_rows = max_rows
        self.fwd = oracle.layer_forward_mxfp8 if mode in ("mxfp8", "mxfp8_full") else oracle.layer_forward
        self.bwd = {"mxfp8": oracle.layer_backward_mxfp8,
                    "mxfp8_full": oracle.layer_backward_mxfp8_full}.get(mode, oracle.layer_backward)
        te = inp.top_experts
        self.cnt = torch_bincount(te, self.E)
        self.next_e = 0
        self.n = 0                       # units run so far (decides the next unit's kind)
        self.reset()

    def reset(self):
        """Forget the units timed so far (the unit cycle goes on)."""
        self.time = {"routed": 0.0, "shared": 0.0}
        self.rows = {"routed": 0, "shared": 0}
        self.units = {"routed": 0, "shared": 0}

    @staticmethod
    def _np(t):
        return None if t is None else t.detach().to("cpu").double().numpy()

    def _routed_unit(self):
        while self.cnt[self.next_e] == 0:
            self.next_e = (self.next_e + 1) % self.E
        e = self.next_e
        self.next_e = (e + 1) % self.E
        inp = self.inp
        t_e, j_e = (v[:self.max_rows] for v in (inp.top_experts == e).nonzero(as_tuple=True))
        n = int(t_e.numel())
        args = (self._np(inp.x[t_e]), self._np(inp.router_w[t_e, j_e].reshape(-1, 1)),
                __import__("numpy").zeros((n, 1), dtype="int64"), self._np(inp.w_gate[e:e + 1]),
                self._np(inp.w_up[e:e + 1]), self._np(inp.w_down[e:e + 1]), None, None, None)
        return "routed", n, args, self._np(inp.dy[t_e])

    def _shared_unit(self):
        import numpy as np

        inp = self.inp
        n = min(self.max_rows, inp.x.shape[0])
        e0 = np.zeros((0,) + tuple(inp.w_gate.shape[1:]))
        d0 = np.zeros((0,) + tuple(inp.w_down.shape[1:]))
        args = (self._np(inp.x[:n]), np.zeros((n, 0)), np.zeros((n, 0), dtype=np.int64), e0, e0, d0,
                self._np(inp.ws_gate), self._np(inp.ws_up), self._np(inp.ws_down))
        return "shared", n, args, self._np(inp.dy[:n])

    def run_unit(self):
        """One unit (the next in the 1 shared : k routed cycle, shared first);
        returns its seconds."""
        shared = self.shared and self.n % (self.k + 1) == 0
        kind, n, a, dy = self._shared_unit() if shared else self._routed_unit()
        t0 = time.perf_counter()
        self.fwd(*a)
        self.bwd(*a[:6], dy, *a[6:])
        el = time.perf_counter() - t0
        self.n += 1
        self.time[kind] += el
        self.rows[kind] += n
        self.units[kind] += 1
        return el

    def tokens_per_s(self):
        s_r = self.time["routed"] / max(self.rows["routed"], 1)
        s_s = self.time["shared"] / self.rows["shared"] if self.rows["shared"] else 0.0
        return 1.0 / (self.k * s_r + s_s)

    def describe(self):
        d = (f"{self.units['routed']} routed units (one expert each over at most {self.max_rows} of the rows "
             f"routed to it; {self.rows['routed']} rows in {self.time['routed']:.1f} s)")
        if self.shared:
            d += (f" and {self.units['shared']} shared units (the shared expert over {self.max_rows} tokens; "
                  f"{self.rows['shared']} rows in {self.time['shared']:.1f} s)")
        return d + ", float64 NumPy; tokens/s = 1 / (k * s_routed_row + s_shared_row)"


def torch_bincount(te, E):
    import torch

    return torch.bincount(te.reshape(-1).to("cpu"), minlength=E).tolist()


# Rows per oracle unit: at most this many of an expert's rows (the T=4096
# layers route about 512 rows to an expert, the large layer about 2048).
CPU_UNIT_ROWS = 1024


def cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count()


# ----------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mok", "reference"], default="mok")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--stages", action="store_true", help="print per-stage times to stderr")
    ap.add_argument("--capacity", type=float, default=None, help="override the workload's capacity multiplier")
    ap.add_argument("--minibatch", type=int, default=None, help="override the workload's minibatch size")
    ap.add_argument("--dispatch", choices=["auto", "permute", "fused"], default="auto",
                    help="how the bf16 GEMMs receive token rows (same results)")
    ap.add_argument("--debug-flags", type=int, default=0,
                    help="MOK_DEBUG_* flags that change kernel choices only (e.g. 4: single CTAs, 8: MXFP8 CTA pairs)")
    ap.add_argument("--macrobatch", type=int, default=0,
                    help="rows of the token ring, forward and backward (0: one pass; same results)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.debug_flags & 1:
        ap.error("--debug-flags 1 withholds a GEMM signal (a timeout test), not a kernel choice")

    rank, world, local = dist_env()

    from mixture_experts_layer_mok_gb300 import inputs as gen

    c = dict(gen.WORKLOADS[args.workload])
    if args.capacity is not None:
        c["capacity"] = args.capacity
    if args.minibatch is not None:
        c["minibatch"] = args.minibatch
    fwd_flop, step_flop = layer_flops(c)
    config = {"workload": args.workload, "T": c["T"], "H": c["H"], "I": c["I"], "E": c["E"], "k": c["k"],
              "I_s": c["I_s"], "routing": "zipf s=%.1f" % c["skew"] if c["skew"] else "softmax top-k",
              "minibatch": c["minibatch"], "capacity_multiplier": c["capacity"],
              "fwd_precision": "bf16" if c["mode"] == "bf16" else "mxfp8",
              "bwd_precision": "mxfp8" if c["mode"] == "mxfp8_full" else "bf16", "global_batch_tokens": c["T"] * max(world, 1),
              "parallelism": f"dp{world} (independent batches, no collective)",
              "l2": "flushed between steps (512 MiB write, outside the timed spans)"}
    if args.dispatch != "auto" or args.debug_flags:
        config.update(dispatch=args.dispatch, debug_flags=args.debug_flags)
    if args.macrobatch:
        config.update(macrobatch_size=args.macrobatch)

    if args.impl == "reference":
        return run_reference(args, c, config, rank, world)

    import torch

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import mixture_experts_layer_mok_gb300 as mok
    from mixture_experts_layer_mok_gb300 import _lib

    _lib.load()  # fails loudly when the library is not built
    big = c["E"] * c["I"] * c["H"] > 3e8      # draw large layers on the GPU (seeded all the same)
    inp = gen.make_workload(args.workload, seed=rank, device=dev if big else "cpu")
    g = inp.to(dev)
    w = mok.Weights(g.w_gate, g.w_up, g.w_down, g.ws_gate, g.ws_up, g.ws_down)
    mode = c["mode"]
    E, T, k, H, I, Is = c["E"], c["T"], c["k"], c["H"], c["I"], c["I_s"]
    lib = _lib.load()
    m = mok.MODES[mode]
    ctx_bytes = lib.mok_ctx_bytes_ring(T, k, E, H, I, Is, m, args.macrobatch)
    ws_bytes = lib.mok_bwd_workspace_bytes_ring(T, k, E, H, I, Is, m, args.macrobatch)
    config.update(ctx_ws_gib=round((ctx_bytes + ws_bytes) / 2**30, 2))
    ctx_buf = torch.empty(ctx_bytes, dtype=torch.uint8, device=dev)
    ws_buf = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    grads = {"dx": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
             "d_router_w": torch.empty((T, k), dtype=torch.float32, device=dev),
             "d_w_gate": torch.empty_like(g.w_gate), "d_w_up": torch.empty_like(g.w_up),
             "d_w_down": torch.empty_like(g.w_down)}
    if Is:
        grads.update(d_ws_gate=torch.empty_like(g.ws_gate), d_ws_up=torch.empty_like(g.ws_up),
                     d_ws_down=torch.empty_like(g.ws_down))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def run_step(x, rw, top, dy, events=None, prep_events=None, y_out=None, g_out=None):
        if prep_events:
            prep_events[0].record()
        wq = mok.quantize_weights(w, backward=(mode == "mxfp8_full")) if mode != "bf16" else w
        sched = mok.schedule(top, E, c["capacity"])
        if prep_events:
            prep_events[1].record()
        _, ctx = mok.forward(x, rw, sched, wq, mode=mode, minibatch=c["minibatch"],
                             out=y if y_out is None else y_out, ctx_buf=ctx_buf, events=events,
                             dispatch=args.dispatch, debug=args.debug_flags, macrobatch=args.macrobatch)
        mok.backward(dy, x, rw, sched, ctx, wq, minibatch=c["minibatch"], grads=grads if g_out is None else g_out,
                     ws_buf=ws_buf, events=events, dispatch=args.dispatch, debug=args.debug_flags,
                     macrobatch=args.macrobatch)
        return ctx

    for _ in range(args.warmup):
        ctx = run_step(g.x, g.router_w, g.top_experts, g.dy)
    torch.cuda.synchronize()
    if ctx.status() != 0:
        raise RuntimeError(f"device status {ctx.status()} after warm-up")
    # a ring smaller than the schedule's worst case runs the routed experts in
    # windows (one, when the actual rows fit)
    max_rows = (T * k + 127 * E) // 128 * 128
    ring_on = 0 < -(-args.macrobatch // 128) * 128 < max_rows
    n_windows = 1
    if ring_on:
        cnt = mok.schedule(g.top_experts, E, c["capacity"]).arrays()["cnt"].cpu().tolist()
        n_windows = len(mok.macrobatch_plan(cnt, args.macrobatch))
        config.update(macrobatch_windows=n_windows)

    nst = _lib.MOK_NUM_STAGES
    K = args.steps
    names = _lib.STAGE_NAMES
    sf = stage_flops(c)
    # ---- stage profile, outside the timed region: every stage's events.  Each
    # event record costs the device a few microseconds, so the timed steps
    # below record only the dominant stage's pair.
    prof_steps = 5
    ev_prof = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nst)] for _ in range(prof_steps)]
    ev_prep = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(prof_steps)]
    for i in range(prof_steps):
        flush.zero_()
        run_step(g.x, g.router_w, g.top_experts, g.dy, events=ev_prof[i], prep_events=ev_prep[i])
    torch.cuda.synchronize()
    st_ms = {names[s]: sum(ev_prof[i][2 * s].elapsed_time(ev_prof[i][2 * s + 1]) for i in range(prof_steps)) /
             prof_steps for s in range(nst)}
    # the caller's part of a step: weight prequantisation (MXFP8 modes) and the schedule build
    st_ms["step_prep"] = sum(e[0].elapsed_time(e[1]) for e in ev_prep) / prof_steps
    gemm_stages = {n: v for n, v in st_ms.items() if n in sf and sf[n] > 0}
    dom = max(gemm_stages, key=gemm_stages.get)
    di = names.index(dom)

    ev_start = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_end = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_dom = []
    for _ in range(K):
        evs = [None] * (2 * nst)
        evs[2 * di] = torch.cuda.Event(enable_timing=True)
        evs[2 * di + 1] = torch.cuda.Event(enable_timing=True)
        ev_dom.append(evs)
    sampler = ClockSampler(dev.index) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()                       # evict L2 between steps (outside the timed spans)
        ev_start[i].record(stream)
        run_step(g.x, g.router_w, g.top_experts, g.dy, events=ev_dom[i])
        ev_end[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler else None
    if world > 1:
        torch.distributed.barrier()
    step_ms = [ev_start[i].elapsed_time(ev_end[i]) for i in range(K)]
    total_ms = sum(step_ms)
    if ctx.status() != 0:
        raise RuntimeError(f"device status {ctx.status()} in the timed region")
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / K
    tokens_per_s = job_tokens_per_s(T, world, K, total_ms)
    tflops = step_flop * max(world, 1) * K / (total_ms / 1e3) / 1e12

    # the dominant GEMM's launches inside the timed region, on their stream
    dom_ms = sum(ev_dom[i][2 * di].elapsed_time(ev_dom[i][2 * di + 1]) for i in range(K)) / K
    peaks = load_peaks()
    achieved = sf[dom] / (dom_ms / 1e3) / 1e12
    gemm_ms = sum(gemm_stages.values())
    gemm_tflops = sum(sf[n] for n in gemm_stages) / (gemm_ms / 1e3) / 1e12
    if args.stages and rank == 0:
        for n in names + ["step_prep"]:
            extra = f"  {sf[n] / (st_ms[n] / 1e3) / 1e12:8.1f} TFLOP/s" if n in gemm_stages else ""
            print(f"  {n:26s} {st_ms[n]:8.4f} ms{extra}", file=sys.stderr)

    # ---- end to end through the public API with host buffers.  Like a training
    # loop with a prefetching loader: each step's inputs come from pinned host
    # memory and its results go back to it, on a copy stream that overlaps the
    # neighbouring steps' compute (inputs and outputs double-buffered on the
    # device).  The timed region runs from the first input copy to the last
    # result copy.  No L2 flush: every step streams its 0.8 GB or more of
    # weights through the 129 MB L2.
    e2e = None
    if not args.no_e2e:
        hx = inp.x.cpu().pin_memory()
        hrw = inp.router_w.cpu().pin_memory()
        htop = inp.top_experts.cpu().pin_memory()
        hdy = inp.dy.cpu().pin_memory()
        oy = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
        odx = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
        odw = torch.empty((T, k), dtype=torch.float32).pin_memory()
        hosts_in = (hx, hrw, htop, hdy)
        ins = [tuple(torch.empty_like(t) for t in (g.x, g.router_w, g.top_experts, g.dy)) for _ in range(2)]
        # y, dx and d_router_w go back to the host: two copies each; the weight
        # gradients stay on the device and are shared by the two slots
        outs = [(torch.empty_like(y), {n: (torch.empty_like(v) if n in ("dx", "d_router_w") else v)
                                       for n, v in grads.items()}) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in hosts_in)
        d2h = sum(t.numel() * t.element_size() for t in (oy, odx, odw))
        copy = torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)

        def put(slot):                      # host -> device inputs of one step, on the copy stream
            with torch.cuda.stream(copy):
                for d, hsrc in zip(ins[slot], hosts_in):
                    d.copy_(hsrc, non_blocking=True)
                ev_in[slot].record(copy)

        def pipeline(n, timed):
            torch.cuda.synchronize()
            if timed:
                e_start.record(copy)
            for slot in range(min(n, 2)):
                put(slot)
            for i in range(n):
                slot = i % 2
                stream.wait_event(ev_in[slot])
                if i >= 2:
                    stream.wait_event(ev_out[slot])   # step i-2's results have left this slot
                run_step(*ins[slot], y_out=outs[slot][0], g_out=outs[slot][1])
                ev_done[slot].record(stream)
                with torch.cuda.stream(copy):
                    copy.wait_event(ev_done[slot])
                    oy.copy_(outs[slot][0], non_blocking=True)
                    odx.copy_(outs[slot][1]["dx"], non_blocking=True)
                    odw.copy_(outs[slot][1]["d_router_w"], non_blocking=True)
                    ev_out[slot].record(copy)
                if i + 2 < n:
                    put(slot)                       # step i+2's inputs (step i is done with the slot)
            if timed:
                e_end.record(copy)
            torch.cuda.synchronize()

        Ke = max(3, min(K, 50))
        pipeline(3, False)
        pipeline(Ke, True)
        e_ms = e_start.elapsed_time(e_end)
        e_ms = max_over_ranks(e_ms, world, dev)
        e2e = {"value": round(job_tokens_per_s(T, world, Ke, e_ms), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
               "what": "pinned host x, router weights, top-k ids, dy -> device; schedule + fwd + bwd through "
                       "the binding; y, dx, d_router_w -> host; copies on a second stream overlap the "
                       "neighbouring steps' compute (double-buffered), all inside the timed region"}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sample = OracleSample(inp, mode, CPU_UNIT_ROWS)
        need = 1 + (1 if sample.shared else 0)        # at least one unit of each kind
        el = 0.0
        while el < 10.0 or sample.n < need:
            el += sample.run_unit()
        cpu = {"value": round(sample.tokens_per_s(), 3), "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{args.workload} layer: " + sample.describe()}
        del sample

    # a kernel timed inside a long step runs at the sustained (power-capped)
    # rate; one inside a short step at the burst rate
    long_step = ms_per_step > LONG_STEP_MS and peaks.get("bf16_tflops_sustained")
    peak_key = "bf16_tflops_sustained" if long_step else "bf16_tflops"
    kind = "sustained" if long_step else "burst"
    base_src = (f"{peaks['source']} bf16 {kind} (MEASURED_PEAKS.json)" if peaks["source"] == "measured"
                else f"fallback bf16 {kind}")
    if (mode == "mxfp8" and dom in FWD_GEMM_STAGES) or mode == "mxfp8_full":
        # block-scaled E4M3 GEMM: the bf16 figure times the nominal dense fp8:bf16 ratio (4.5 / 2.25)
        dom_peak, dom_src = 2.0 * peaks[peak_key], base_src + " x 2 (nominal dense fp8:bf16 ratio)"
    else:
        dom_peak, dom_src = peaks[peak_key], base_src
    line = {
        "metric": METRIC,
        "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": max(world, 1), "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "mxfp8": "mxfp8-fwd/bf16-bwd"}.get(mode, "mxfp8-fwd/mxfp8-bwd"),
        "data": "synthetic (seeded; weights N(0,0.02), x and dy N(0,1), softmax top-k routing)",
        "config": config,
        "tflops": round(tflops, 1),
        "tc_peak_frac": round(tflops / peaks[peak_key], 4),
        "gemm_tflops": round(gemm_tflops, 1),
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1),
                     "peak": dom_peak, "unit": "TFLOP/s", "frac": round(achieved / dom_peak, 4),
                     "peak_source": dom_src,
                     "traffic": recorded_traffic(args.workload, dom),
                     "algorithmic_flop_per_launch": sf[dom], "ms_per_launch": round(dom_ms, 4),
                     "timed": "CUDA events around this stage in every timed step" + (
                         "; with the ring they span the stage's first to last window, other stages"
                         " included, so achieved is a lower bound" if n_windows > 1 else "")},
        "stage_ms": {n: round(v, 4) for n, v in st_ms.items()},
        "stage_ms_from": "5 untimed steps recording every stage's events (the timed steps record the dominant stage's only)",
        "gpu_launches": launches_per_step(c, n_windows, ring_on) * K,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "wall_s": round(wall, 3),
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args, c, config, rank, world):
    """The CPU oracle as the reference arm: each step is one oracle unit of the
    same workload (see OracleSample) on the host cores; tokens/s follows from
    the per-row times of the units run in the timed steps."""
    if rank != 0:
        return
    from mixture_experts_layer_mok_gb300 import inputs as gen

    dev = "cpu"
    if c["E"] * c["I"] * c["H"] > 3e8:   # the same seeded draw as the measured arm (on the GPU), cut up on the host
        import torch

        if torch.cuda.is_available():
            dev = torch.device("cuda", 0)
    inp = gen.make_workload(args.workload, seed=0, device=dev)
    sample = OracleSample(inp, c["mode"], CPU_UNIT_ROWS)
    for _ in range(args.warmup):
        sample.run_unit()
    warm = (dict(sample.time), dict(sample.rows), dict(sample.units))
    sample.reset()
    el_total = 0.0
    for _ in range(args.steps):
        el_total += sample.run_unit()
    if sample.rows["routed"] == 0 or (sample.shared and sample.rows["shared"] == 0):
        # too few timed steps for both kinds: take the missing kind from the warm-up units
        for kind in sample.time:
            if sample.rows[kind] == 0:
                sample.time[kind], sample.rows[kind], sample.units[kind] = (w[kind] for w in warm)
    value = sample.tokens_per_s()
    desc = f"{args.workload} layer, each timed step one oracle unit: " + sample.describe()
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3),
            "unit": "tokens/s", "n_gpus": world, "device": "host cores only (rank 0; the oracle does no GPU work)",
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * el_total / args.steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)", "config": config,
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
