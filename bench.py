#!/usr/bin/env python
"""Benchmark of the MoE layer (token dispatch + expert compute) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dsv3|l4mav|small|tiny|profile]

One step = one pass of the whole layer over one batch of T tokens whose
inputs (x, the router weight and logit offset, the expert weights) are
already in HBM: router logits (x @ Wr + offset) -> route -> counts +
overflow check -> capped path, or the chunked dropless fallback when a shard
overflows -> (per pass) permute + dedup -> GEMM1 + SwiGLU -> GEMM2 ->
combine.  The default workload is the DeepSeek-V3-shaped layer (T=8192,
H=7168, E=256, k=8, F=2048, 8 shards, Zipf s=1.2 routing,
ragged_buffer_factor 2.0), on which the grouped GEMM target is stated.

The timed step is moe_router_logits followed by one launch of the traced
layer graph (moe_layer_graph_create_traced): the branch is a conditional
node on the device, so no step waits on the host.  CUDA events on the launch
stream bracket every step (and the router); the graph writes a device
timestamp at every stage boundary, from which the per-stage times of the
roofline come, in the same timed launches.  L2 is flushed (a 256 MiB write)
between steps, outside the events.  The same layer through the stepwise
entry points (host flag read, CUDA events between stages) is checked bit
for bit against moe_layer and the graph, and reported under ``stepwise``;
``untraced_graph`` is the graph without the stamps; ``warm_l2`` the traced
launches without the flush.  ``e2e`` is the same metric through the C ABI
with pinned host buffers: x and the logit offset copied in, the router and
the layer graph, y copied out, every step, the copies overlapping the
neighbouring steps on two copy streams (``e2e.serial``: through moe_layer,
copies in line).  ``cpu_baseline`` is the float64 oracle timed on a bounded
token sample of the same workload on the host cores.  The default run then
times every other workload of the benchmark briefly (``configs``: tiny,
small, the DeepSeek-V3 layer as one uncapped pass under uniform and Zipf
routing, Llama4-Maverick, and the routing/permute/dedup sweep at 1K-64K
tokens under three routings), each with its own clock record.

``--backward`` times the layer's backward pass instead (its own JSON line):
route -> check -> per pass: permute, GEMM1 keeping g and u, GEMM2, combine
backward, down-projection dgrad with the SwiGLU backward, gate/up dgrad,
permute backward -> route backward -> the two weight-gradient GEMMs over
the rows of every pass (one launch each), the permute tables again a pass
ahead on the side stream.  Its ``e2e`` goes through moe_layer_backward with
x, logits and dy copied in and dx and dlogits copied out every step, the
copies overlapping the neighbouring steps (``e2e.serial``: in line); the
weight gradients stay in HBM.  With torchrun (N > 1) every rank runs an
independent replica on its own tokens (weak scaling, no collective on the
data path); the reported time is the max over ranks.
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

# BLAS threads for the oracle: every core this process may use.
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") \
    else (os.cpu_count() or 1)
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from synth import (WORKLOADS, make_logit_offset, make_router_weight,  # noqa: E402
                   make_weights, make_x)
from synth.workloads import make_dy  # noqa: E402

METRIC = "MoE layer tokens/sec at 1 GB300; permute GB/s and GMM TFLOP/s vs roofline"
METRIC_BWD = "MoE layer backward tokens/sec at 1 GB300 (forward recomputed per pass)"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}

# bench-only workload for profiling captures: the DeepSeek-V3 layer shape with
# 32 experts and 1024 tokens (2.8 GB of weights: larger than L2, a few GB in
# total on the device)
PROFILE_WL = WORKLOADS["dsv3"].with_(name="profile_dsv3_e32", T=1024, E=32)
# the backward's kernel captures: DeepSeek-V3 layer shape with 8 experts,
# 256 tokens (256 rows per expert, as at full size) in 4 fallback chunks, so
# the weight gradients sum 4 row segments; ~2 GB on the device
PROFILE_BWD_WL = WORKLOADS["dsv3"].with_(name="profile_bwd_dsv3_e8", T=256,
                                         E=8, n_chunks=4)

# oracle sample sizes (tokens) for the CPU baseline and the reference arm
CPU_SAMPLE = {"dsv3": 32, "l4mav": 32, "small": 1024, "tiny": 256,
              "profile_dsv3_e32": 32}
REF_SAMPLE = {"dsv3": 8, "l4mav": 8, "small": 256, "tiny": 256,
              "profile_dsv3_e32": 8}
BWD_CPU_SAMPLE = {"dsv3": 8, "l4mav": 8, "small": 256, "tiny": 256,
                  "profile_dsv3_e32": 8}


def workload_by_name(name, sweep_T=65536, routing=None):
    if name == "profile":
        return PROFILE_WL
    if name == "profile_bwd":
        return PROFILE_BWD_WL
    if name == "sweep":
        from synth import sweep_workload
        return sweep_workload(sweep_T, routing or "zipf")
    return WORKLOADS[name]


# ------------------------------------------------------------------ peaks --
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_digest(kernel):
    """First 16 hex digits of the sha256 of the code a GEMM kernel is built
    from (the shared tensor-core header + its own file), comments and blank
    lines left out, so that an edit of a comment keeps a profile valid."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "mixture_experts_token_gb300", "csrc")
    own = "wgrad_tc.cu" if kernel.endswith("_wgrad") else "gmm_tc.cu"
    h = hashlib.sha256()
    for name in ("tc_common.cuh", own):
        with open(os.path.join(csrc, name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        lines = [re.sub(r"\s*//.*$", "", ln).rstrip() for ln in
                 src.splitlines()]
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    try:
        digest = kernel_source_digest(kernel)
        path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
        want = None
        for line in open(path):
            if line.startswith("traffic_bytes_per_launch:"):
                parts = line.split()
                if len(parts) >= 4 and parts[3] == digest:
                    want = float(parts[1])
        return want
    except OSError:
        return None


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.device = device

    def _id(self):
        try:
            u = str(torch.cuda.get_device_properties(self.device).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return str(self.device)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self._id()}",
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ ranks ------
def max_over_ranks(value: float, device) -> float:
    """Max of a per-rank float over all ranks (the slowest rank's time);
    the value itself with one process."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or \
            dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_workload(wl, rank: int):
    """Each rank runs an independent replica on its own tokens and weights:
    the same shapes, a seed shifted by the rank (weak scaling)."""
    return wl.with_(seed=wl.seed + rank)


def whole_job_tokens_per_s(world: int, T: int, ms_per_step: float) -> float:
    return world * T / (ms_per_step / 1e3)


# ------------------------------------------------------------ the layer ---
class Layer:
    """Inputs in HBM and every buffer of the stepwise calls."""

    def __init__(self, wl, device, seed_offset=0, mode="fallback"):
        import mixture_experts_token_gb300 as moe
        self.moe = moe
        self.mode = mode
        self.wl = replica_workload(wl, seed_offset)
        w = self.wl
        self.cfg = moe.make_config(w.T, w.H, w.E, w.k, w.F, w.S, w.factor,
                                   w.n_chunks, w.dtype, w.renorm,
                                   w.redundant_slots)
        self.x = make_x(w, device)
        # router: logits = x @ Wr + offset, computed by the library in each
        # step (here once more so that the logits exist before any step)
        self.wr = make_router_weight(w, device)
        self.offset_np = make_logit_offset(w)
        self.offset = None if self.offset_np is None else \
            torch.from_numpy(self.offset_np).to(device)
        self.logits = torch.empty((w.T, w.E), dtype=torch.float32,
                                  device=device)
        moe.moe_router_logits(self.cfg, self.x, self.wr, self.offset,
                              self.logits)
        self.dispatch_only = w.F == 0   # the routing/permute sweep
        self.W = make_weights(w, device) if not self.dispatch_only else None
        self.b = moe.alloc_step_buffers(self.cfg, device)
        self.b["y"].zero_()
        self.ws = moe.layer_workspace(self.cfg, moe.MOE_WS_LAYER, device)
        self.chunk = moe.moe_chunk_tokens(self.cfg)
        # Two sets of a pass's permute tables: the tables of pass i+1 are
        # computed on the side stream while pass i runs its expert FFN.
        # Set 0 is the step buffers themselves.
        keys = ("sorted_token", "group_offsets", "uniq_offsets",
                "uniq_tokens", "expand_idx", "n_dropped", "permute_ws")
        self.tabs = [{k: self.b[k] for k in keys},
                     {k: torch.empty_like(self.b[k]) for k in keys}]
        self.side = torch.cuda.Stream(device=device)
        self.pass_events = []   # (tables ready, pass done) per pass, reused
        self.routed = torch.cuda.Event()   # the step's routing is done
        self._subs = {}

    def sub(self, t0, t1, capped):
        """Pass over tokens [t0, t1): the config the library uses (built
        once per pass shape)."""
        if capped:
            return self.cfg
        key = t1 - t0
        if key not in self._subs:
            self._subs[key] = self.cfg.with_(T=key, ragged_buffer_factor=-1.0,
                                             n_chunks=0, redundant_slots=0)
        return self._subs[key]

    def step(self, ev=None, hold_cycles=0):
        """One layer step through the entry points; ev(name) marks stages.
        hold_cycles > 0 puts a GPU sleep of that many cycles (its own stage,
        "hold") before the first pass, so that the host has queued the
        pass's launches before the GPU reaches them.  Returns the list of
        passes (t0, t1, capped)."""
        moe, b, c, W = self.moe, self.b, self.cfg, self.W
        mark = ev or (lambda name: None)
        mark("router")
        moe.moe_router_logits(c, self.x, self.wr, self.offset, self.logits,
                              b["status"])
        mark("route")
        moe.moe_route(c, self.logits, b["topk_idx"], b["topk_w"], b["status"])
        self.routed.record()   # the side stream's tables start after it
        if self.mode != "fallback":
            passes = [(0, c.T, self.mode == "capped")]
            return self._passes(passes, mark, hold_cycles)
        mark("check")
        moe.moe_check_overflow(c, b["topk_idx"], b["expert_counts"],
                               b["expert_offsets"], b["shard_counts"],
                               b["overflow_flag"], b["required_factor"],
                               b["capacity"])
        planned = c.redundant_slots > 0
        if planned:
            mark("plan")
            moe.moe_plan_duplication(c, b["expert_counts"], b["divert"],
                                     b["slot_of"], b["group_expert"],
                                     b["shard_after"], b["flag_after"])
        mark("flag")
        flag = int((b["flag_after"] if planned else b["overflow_flag"]).item())
        if not flag:
            passes = [(0, c.T, True)]
        else:
            passes = [(t0, min(c.T, t0 + self.chunk), False)
                      for t0 in range(0, c.T, self.chunk)]
        return self._passes(passes, mark, hold_cycles)

    def _tables(self, pas, i, stream, ready, side_times=None, after=None):
        """Permute tables of pass i over tokens pas = (t0, t1, capped) into
        table set i % 2, on `stream` (after event `after`, if given);
        records `ready`.  Side-stream work is timed into side_times."""
        moe, b = self.moe, self.b
        t0, t1, capped = pas
        sc = self.sub(t0, t1, capped)
        tb = self.tabs[i % 2]
        plan = {}
        if capped and sc.redundant_slots > 0:
            plan = dict(divert=b["divert"], slot_of=b["slot_of"])
        timed = side_times is not None and stream is self.side
        if after is not None:
            stream.wait_event(after)
        if timed:
            ev0 = torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
        moe.moe_permute_tables(
            sc, b["topk_idx"][t0:t1], capped, b["row_of"][t0:t1],
            tb["sorted_token"], tb["group_offsets"], tb["uniq_offsets"],
            tb["n_dropped"], tb["permute_ws"], stream=stream, **plan)
        if ready is not None:
            ready.record(stream)
        if timed:
            ev1 = torch.cuda.Event(enable_timing=True)
            ev1.record(stream)
            side_times.append((ev0, ev1))

    def _passes(self, passes, mark, hold_cycles=0):
        """The passes, each: permute tables -> row scatter -> GEMM1 ->
        GEMM2 -> combine.  The first pass's tables run on the main stream;
        those of pass i+1 are queued on the side stream after pass i's
        work, so they run during pass i's FFN.  They reuse the table set of
        pass i-1 and wait for that pass's combine."""
        moe, b, W = self.moe, self.b, self.W
        if hold_cycles:
            mark("hold")
            torch.cuda._sleep(hold_cycles)
        main, side = torch.cuda.current_stream(), self.side
        while len(self.pass_events) < len(passes):
            self.pass_events.append((torch.cuda.Event(), torch.cuda.Event()))
        ready = [e[0] for e in self.pass_events]
        done = [e[1] for e in self.pass_events]
        side_times = getattr(mark, "side", None)

        def tables(i, stream):
            # the side stream's first table work waits for the routing;
            # a reused table set, for the combine of the pass that read it
            after = self.routed if i == 1 else \
                (done[i - 2] if i >= 2 else None)
            self._tables(passes[i], i, stream,
                         ready[i] if stream is side else None, side_times,
                         after)

        for i, (t0, t1, capped) in enumerate(passes):
            sc = self.sub(t0, t1, capped)
            tb = self.tabs[i % 2]
            row_of = b["row_of"][t0:t1]
            groups = {}
            if capped and sc.redundant_slots > 0:
                groups = dict(n_groups=sc.E + sc.S * sc.redundant_slots,
                              group_expert=b["group_expert"])
            mark("permute")
            if i == 0:
                tables(0, main)
            else:
                main.wait_event(ready[i])
            moe.moe_permute_scatter(sc, self.x[t0:t1], row_of,
                                    tb["uniq_offsets"], b["x_sorted"],
                                    tb["uniq_tokens"], tb["expand_idx"],
                                    tb["permute_ws"])
            if self.dispatch_only:
                # no expert FFN: the combine reads the permuted rows back
                mark("combine")
                moe.moe_combine(sc, b["x_sorted"], row_of,
                                b["topk_w"][t0:t1], b["y"][t0:t1])
                done[i].record(main)
                if i + 1 < len(passes):
                    tables(i + 1, side)
                continue
            mark("gmm_gate_up")
            moe.moe_gmm_gate_up(sc, b["x_sorted"], tb["group_offsets"], W[0],
                                W[1], b["h"], b["status"], **groups)
            mark("gmm_down")
            moe.moe_gmm_down(sc, b["h"], tb["group_offsets"], W[2],
                             b["y_sorted"], b["status"], **groups)
            mark("combine")
            moe.moe_combine(sc, b["y_sorted"], row_of, b["topk_w"][t0:t1],
                            b["y"][t0:t1])
            done[i].record(main)
            if i + 1 < len(passes):
                tables(i + 1, side)
        mark(None)
        return passes

    def api_layer(self, x, logits, y):
        mode = {"fallback": self.moe.MOE_MODE_FALLBACK_LAYER,
                "capped": self.moe.MOE_MODE_CAPPED,
                "dropless": self.moe.MOE_MODE_DROPLESS}[self.mode]
        W = self.W if self.W is not None else (None, None, None)
        return self.moe.moe_layer(self.cfg, x, logits, *W, y, mode,
                                  self.ws, self.b["status"])


class StageTimer:
    """CUDA events on the current stream between consecutive stage marks;
    `side` collects (start, end) events of the permute tables on the side
    stream."""

    def __init__(self):
        self.events = []
        self.names = []
        self.side = []

    def __call__(self, name):
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        self.events.append(e)
        self.names.append(name)

    def durations(self):
        out = []
        for i in range(len(self.events) - 1):
            if self.names[i] is None:
                continue
            out.append((self.names[i],
                        self.events[i].elapsed_time(self.events[i + 1])))
        return out


HOLD_CYCLES = 1_000_000   # about 0.5 ms at 2 GHz


def table_launches(tokens, shards):
    """Permute-table kernels of one pass over `tokens` tokens: block counts,
    expert scan, assign, and the dedup scan when the block x shard table
    holds more than 1024 counts (with shards = 0, never)."""
    if tokens <= 0:
        return 1
    nb = (tokens + 127) // 128
    return 3 + (1 if shards and nb * shards > 1024 else 0)


def launches_per_step(passes, mode, dispatch_only=False, planned=0,
                      shards=0):
    """Kernel launches of one step: router 1, route 1 (+ check 1 with the
    fallback, + the plan), then per pass the permute tables
    (table_launches) and the row scatter, GEMM1 1, GEMM2 1, combine 1 (no
    GEMMs in the sweep)."""
    per = 2 if dispatch_only else 4
    return 1 + (2 if mode == "fallback" else 1) + planned + \
        sum(table_launches(t1 - t0, shards) + per
            for (t0, t1, _) in passes if t1 > t0)


def pass_accounting(layer, passes):
    """Rows and active experts of each pass (bench bookkeeping with torch,
    outside any timed region)."""
    w = layer.wl
    idx = layer.b["topk_idx"].long()
    C = layer.moe.moe_capacity_rows(layer.cfg)
    out = []
    for (t0, t1, capped) in passes:
        if capped and layer.cfg.redundant_slots > 0:
            # virtual groups of the plan: rows kept, distinct experts used
            G = w.E + w.S * layer.cfg.redundant_slots
            off = layer.b["group_offsets"][:G + 1].cpu().numpy()
            gexp = layer.b["group_expert"][:G].cpu().numpy()
            sizes = np.diff(off)
            out.append({"T": t1 - t0, "R": int(off[G]),
                        "E_act": len(set(int(gexp[g]) for g in range(G)
                                         if sizes[g] > 0))})
            continue
        sub = idx[t0:t1].reshape(-1)
        counts = torch.bincount(sub, minlength=w.E).cpu().numpy()
        if capped and C >= 0:
            Es = w.E // w.S
            kept = np.zeros_like(counts)
            for s in range(w.S):
                room = C
                for e in range(s * Es, (s + 1) * Es):
                    kept[e] = min(counts[e], max(room, 0))
                    room -= counts[e]
            counts = kept
        out.append({"T": t1 - t0, "R": int(counts.sum()),
                    "E_act": int((counts > 0).sum())})
    return out


def stage_work(w, acc):
    """Algorithmic bytes and flops of each stage for one pass."""
    b = 2 if w.dtype == "bf16" else 4
    T, R, Ea = acc["T"], acc["R"], acc["E_act"]
    H, F, k = w.H, w.F, w.k
    return {
        "permute": {"bytes": T * H * b + R * H * b + 16 * R, "flops": 0},
        "gmm_gate_up": {"bytes": 2 * Ea * H * F * b + R * H * b + R * F * b,
                        "flops": 4 * R * H * F},
        "gmm_down": {"bytes": Ea * F * H * b + R * F * b + R * H * b,
                     "flops": 2 * R * F * H},
        "combine": {"bytes": R * H * b + T * H * b + T * k * 8, "flops": 0},
    }


def router_work(w, with_offset):
    """Algorithmic bytes and flops of the router GEMM over the batch."""
    b = 2 if w.dtype == "bf16" else 4
    return {"bytes": w.T * w.H * b + w.H * w.E * b +
            w.T * w.E * 4 * (2 if with_offset else 1),
            "flops": 2 * w.T * w.H * w.E}


# ------------------------------------------------------------ the oracle --
def oracle_sample_run(wl, x_dev, wr, offset, W, n_tok, t0=0,
                      mode="fallback"):
    """Runs the oracle layer on tokens [t0, t0+n_tok) as a batch of its own
    (same shape parameters and factor), from the router logits on; returns
    (seconds, tokens)."""
    from oracle import moe_ref as ref
    n_tok = min(n_tok, wl.T - t0)
    xs = x_dev[t0:t0 + n_tok].to("cpu", torch.float64).numpy()
    wr64 = wr.to("cpu", torch.float64).numpy()
    off = None if offset is None else offset[t0:t0 + n_tok]
    Ls = ref.router_logits(xs, wr64, off)
    oi, _, _ = ref.route(Ls, wl.k, wl.renorm)
    touched = sorted(set(int(e) for e in oi.reshape(-1)))
    host = {e: (W[0][e].cpu(), W[1][e].cpu(), W[2][e].cpu()) for e in touched}

    def weights(e):
        g, u, d = host[e]
        return (g.to(torch.float64).numpy(), u.to(torch.float64).numpy(),
                d.to(torch.float64).numpy())
    cfg = ref.MoEConfig(n_tok, wl.H, wl.E, wl.k, wl.F, wl.S, wl.factor,
                        wl.n_chunks, wl.renorm)
    run = {"fallback": ref.layer, "capped": ref.layer_capped,
           "dropless": ref.layer_dropless}[mode]
    t = time.perf_counter()
    run(cfg, xs, ref.router_logits(xs, wr64, off), weights)
    return time.perf_counter() - t, n_tok


# ------------------------------------------------------------ main -------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dsv3",
                    choices=["dsv3", "l4mav", "small", "tiny", "profile",
                             "profile_bwd", "sweep"],
                    help="sweep: routing/permute/dedup only (no expert FFN)")
    ap.add_argument("--sweep-T", type=int, default=65536)
    ap.add_argument("--redundant-slots", type=int, default=0,
                    help="duplicate-expert slots per shard (dynamic "
                         "redundancy; 0 = off)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count T")
    ap.add_argument("--mode", default="fallback",
                    choices=["fallback", "capped", "dropless"],
                    help="fallback: moe_dropless_fallback=layer (default); "
                         "capped: capped path only; dropless: one uncapped "
                         "pass")
    ap.add_argument("--routing", default=None,
                    choices=["zipf", "uniform", "adversarial"],
                    help="override the workload's routing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' short runs (the default "
                         "DeepSeek-V3 run adds them under \"configs\")")
    ap.add_argument("--backward", action="store_true",
                    help="time the layer's backward pass (own JSON line)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    wl = workload_by_name(args.workload, args.sweep_T, args.routing)
    if args.redundant_slots > 0:
        wl = wl.with_(redundant_slots=args.redundant_slots,
                      name=f"{wl.name}_B{args.redundant_slots}")
    if args.tokens > 0:
        wl = wl.with_(T=args.tokens, name=f"{wl.name}_T{args.tokens}")
    if args.routing and args.workload != "sweep":
        wl = wl.with_(routing=args.routing, zipf_s=wl.zipf_s or 1.2,
                      name=f"{wl.name}_{args.routing}")

    if args.impl == "reference":
        if rank == 0:
            reference_arm(args, wl, device)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    layer = Layer(wl, device, seed_offset=rank, mode=args.mode)
    if args.backward:
        backward_main(layer, args, world, rank, device)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    clocks = ClockSampler(device)
    res = measure_layer(layer, args.steps, args.warmup, device, flush,
                        world=world, clocks=clocks, graph_too=True)
    w = layer.wl
    out = {
        "metric": METRIC, "value": res["value"], "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": res["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded; router logits x @ Wr + offset, the "
                "offset a Zipf/uniform expert popularity by Gumbel-max; "
                "random N(0,0.02) router and expert weights)",
        "config": config_of(layer, args.mode, res, world),
    }
    for key in ("timed_step", "ms_per_step_median", "wall_s_timed_loop",
                "warm_l2", "gpu_launches", "kernels", "roofline",
                "check_us", "permute_frac", "combine_frac", "untraced_graph",
                "stepwise", "clocks"):
        if res.get(key) is not None:
            out[key] = res[key]
    if not args.no_e2e and not layer.dispatch_only:
        if args.mode == "fallback":
            e2e = e2e_pipelined(layer, args, world, device)
            e2e["serial"] = e2e_run(layer, args, world, device, None)
        else:
            e2e = e2e_run(layer, args, world, device, None)
        out["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline and \
            not layer.dispatch_only:
        out["cpu_baseline"] = cpu_baseline(layer)
    if world == 1 and args.workload == "dsv3" and args.mode == "fallback" \
            and args.tokens == 0 and args.redundant_slots == 0 \
            and args.routing is None and not args.no_configs:
        # every other workload of the benchmark, a short timed run each
        del layer
        torch.cuda.empty_cache()
        out["configs"] = config_runs(args, device, flush, res)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def config_of(layer, mode, res, world):
    w = layer.wl
    return {
        "workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k,
        "F": w.F, "S": w.S, "ragged_buffer_factor": w.factor,
        "routing": w.routing + (f" s={w.zipf_s}" if w.routing == "zipf"
                                else ""),
        "redundant_slots": w.redundant_slots,
        "mode": {"fallback": "moe_dropless_fallback=layer",
                 "capped": "capped path only",
                 "dropless": "one uncapped pass"}[mode],
        "overflow": res["overflow"], "passes": res["passes"],
        "capacity": res["capacity"],
        "l2": "flushed between steps (256 MiB write, outside the events)",
        "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
    }


# ------------------------------------------------ timed layer steps ------
STAGES = ("permute", "gmm_gate_up", "gmm_down", "combine")


def trace_stage_ms(stamps, n_pass):
    """Stage durations (ms) of one traced graph launch from its stamps
    (slot layout of moe_layer_graph_create_traced)."""
    d = {"route": (stamps[1] - stamps[0]) / 1e6,
         "check": (stamps[2] - stamps[1]) / 1e6}
    for p in range(n_pass):
        b = 3 + 5 * p
        for j, name in enumerate(STAGES):
            d[name] = d.get(name, 0.0) + (stamps[b + j + 1] -
                                          stamps[b + j]) / 1e6
    return d


def graph_launches(passes, T, shards, planned, chunk_tokens, n_chunks):
    """Kernels of one traced graph step: the router, route, check, (plan),
    the branch select, the stamps (3 + 5 per pass); before the branch, on
    side branches, the capped pass's permute tables (not with a plan) and the
    first fallback chunk's (when the fallback has two chunks or more); then
    per pass the scatter, GEMM1, GEMM2 and combine, and the permute tables
    the side branches did not compute (the later chunks', or the capped
    pass's with a plan)."""
    n = 1 + 3 + planned + 3 + 5 * len(passes)
    if not planned:
        n += table_launches(T, shards)
    if n_chunks >= 2:
        n += table_launches(chunk_tokens, shards)
    overflow = bool(passes) and not passes[0][2]
    for i, (t0, t1, _) in enumerate(passes):
        if t1 <= t0:
            continue
        n += 4
        if overflow and (i >= 1 or n_chunks < 2):
            n += table_launches(t1 - t0, shards)
        if not overflow and planned:
            n += table_launches(t1 - t0, shards)
    return n


def stage_table(layer, passes, stage_ms, mean_ms, steps):
    """kernels dict (per-stage time, share, GB/s, TFLOP/s) and the
    algorithmic work per stage."""
    acc = pass_accounting(layer, passes)
    work = {"router": router_work(layer.wl, layer.offset is not None)}
    for a in acc:
        for name, wv in stage_work(layer.wl, a).items():
            t = work.setdefault(name, {"bytes": 0, "flops": 0})
            t["bytes"] += wv["bytes"]
            t["flops"] += wv["flops"]
    kernels = {}
    for name, ms in stage_ms.items():
        per_step = ms / steps
        ent = {"ms_per_step": round(per_step, 4),
               "share": round(per_step / mean_ms, 4)}
        if name in work and per_step > 0:
            wv = work[name]
            ent["GBps"] = round(wv["bytes"] / (per_step / 1e3) / 1e9, 1)
            if wv["flops"]:
                ent["TFLOPs"] = round(wv["flops"] / (per_step / 1e3) / 1e12,
                                      1)
        kernels[name] = ent
    return kernels, work


def roofline_of(layer, passes, stage_ms, work, steps):
    peaks, peak_src = load_peaks()
    cand = [n for n in work if n in stage_ms and n != "router"]
    dom = max(cand, key=lambda n: stage_ms[n])
    wv = work[dom]
    n_launch = max(1, len(passes))
    dur = stage_ms[dom] / steps / n_launch / 1e3     # per launch
    bytes_l, flops_l = wv["bytes"] / n_launch, wv["flops"] / n_launch
    t_mem = bytes_l / (peaks["hbm_gbs"] * 1e9)
    t_flop = flops_l / (peaks["bf16_tflops_sustained"] * 1e12) \
        if flops_l else 0
    if t_mem >= t_flop:
        achieved = bytes_l / dur / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        achieved = flops_l / dur / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1),
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s"}
    roof["frac"] = round(achieved / roof["peak"], 4)
    roof["traffic"] = profiled_traffic(dom, layer.wl.name)
    roof["kernel"] = dom
    roof["algorithmic_bytes_per_launch"] = int(bytes_l)
    roof["algorithmic_flops_per_launch"] = int(flops_l)
    roof["launch_ms"] = round(dur * 1e3, 4)
    if flops_l:
        roof["tensor_TFLOPs"] = round(flops_l / dur / 1e12, 1)
        roof["tensor_frac_of_burst"] = round(
            flops_l / dur / 1e12 / peaks["bf16_tflops"], 4)
    roof["peak_source"] = f"{peak_src} MEASURED_PEAKS.json" \
        if peak_src == "measured" else "fallback"
    return roof


def hbm_frac(kernels, name):
    peaks, _ = load_peaks()
    k = kernels.get(name)
    if not k or "GBps" not in k:
        return None
    return round(k["GBps"] / peaks["hbm_gbs"], 4)


def steps_for(step_ms, steps, min_s=0.4, cap=400):
    """Timed steps: at least `steps`, and enough for about min_s seconds so
    that the clock sampler sees the loop."""
    return int(max(steps, min(cap, math.ceil(min_s * 1e3 / max(step_ms,
                                                                1e-3)))))


def measure_layer(layer, steps, warmup, device, flush, world=1, clocks=None,
                  graph_too=False, exact=True):
    """One workload: the stepwise entry points checked against moe_layer,
    then the timed steps -- the traced layer graph (router + one graph
    launch per step) for fallback=layer, else the stepwise entry points
    with CUDA events between stages.  exact: time exactly `steps` steps;
    else at least ~0.4 s of steps (for the clock sampler).  Returns the
    bench fields."""
    moe = layer.moe
    passes = layer.step()
    torch.cuda.synchronize()
    b = layer.b
    y_api = torch.empty_like(b["y"])
    info = layer.api_layer(layer.x, layer.logits, y_api)
    torch.cuda.synchronize()
    if not torch.equal(y_api, b["y"]):
        raise SystemExit("stepwise path and moe_layer disagree")
    overflow = info["overflow"]
    del y_api
    if int(b["status"].item()) != 0:
        raise SystemExit(f"device status {int(b['status'].item())}")
    res = {"overflow": overflow, "passes": len(passes),
           "capacity": moe.moe_capacity_rows(layer.cfg)}
    planned = int(layer.cfg.redundant_slots > 0 and layer.mode == "fallback")
    use_graph = layer.mode == "fallback"

    # the stepwise entry points, CUDA events between stages
    for _ in range(warmup):
        flush.zero_()
        layer.step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = StageTimer()
    layer.step(st)
    torch.cuda.synchronize()
    one_ms = sum(d for _, d in st.durations())
    n_sw = steps if (use_graph or exact) else steps_for(one_ms, steps)
    timers = []
    if not use_graph and clocks is not None:
        clocks.start()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for _ in range(n_sw):
        flush.zero_()
        st = StageTimer()
        layer.step(st)
        timers.append(st)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clock_rec = clocks.stop() if (not use_graph and clocks) else None
    sw_ms = [sum(d for _, d in t.durations()) for t in timers]
    sw_mean = max_over_ranks(sum(sw_ms) / len(sw_ms), device)
    sw_stage = {}
    for t in timers:
        for name, d in t.durations():
            sw_stage[name] = sw_stage.get(name, 0.0) + d
    sw_kernels, work = stage_table(layer, passes, sw_stage, sw_mean, n_sw)
    T = layer.wl.T
    if not use_graph:
        res.update({
            "timed_step": "stepwise entry points (moe_router_logits, "
                          "moe_route, moe_check_overflow, host flag read, "
                          "per pass moe_permute_tables/scatter, "
                          "moe_gmm_gate_up, moe_gmm_down, moe_combine), CUDA "
                          "events on the launch stream between stages",
            "value": round(whole_job_tokens_per_s(world, T, sw_mean), 1),
            "ms_per_step": round(sw_mean, 4),
            "ms_per_step_median": round(float(np.median(sw_ms)), 4),
            "wall_s_timed_loop": round(wall, 3), "steps_timed": n_sw,
            "kernels": sw_kernels,
            "roofline": roofline_of(layer, passes, sw_stage, work, n_sw),
            "gpu_launches": launches_per_step(
                passes, layer.mode, layer.dispatch_only, planned,
                layer.wl.S) * n_sw,
            "clocks": clock_rec})
        res["permute_frac"] = hbm_frac(sw_kernels, "permute")
        res["combine_frac"] = hbm_frac(sw_kernels, "combine")
        if "check" in sw_kernels:
            res["check_us"] = round(sw_kernels["check"]["ms_per_step"] * 1e3,
                                    2)
        return res

    # the traced graph: router + one graph launch per step
    n_slots = moe.moe_layer_graph_trace_slots(layer.cfg)
    trace = torch.zeros(n_slots, dtype=torch.int64, device=device)
    x_d = layer.x.clone()
    L_d = torch.empty_like(layer.logits)
    y_d = torch.empty_like(b["y"])
    ws = moe.layer_workspace(layer.cfg, moe.MOE_WS_LAYER, device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    W = layer.W if layer.W is not None else (None, None, None)
    g = moe.MoeLayerGraph(layer.cfg, x_d, L_d, *W, y_d, ws, status,
                          trace=trace)

    def run():
        moe.moe_router_logits(layer.cfg, x_d, layer.wr, layer.offset, L_d,
                              status)
        g.launch()
    run()
    torch.cuda.synchronize()
    if not torch.equal(y_d, b["y"]):
        raise SystemExit("traced graph and stepwise path disagree")
    for _ in range(warmup):
        flush.zero_()
        run()
    torch.cuda.synchronize()
    n = steps if exact else steps_for(sw_mean, steps)
    hist = torch.empty((n, n_slots), dtype=torch.int64, device=device)
    evs = []
    if clocks is not None:
        clocks.start()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(n):
        flush.zero_()
        a, r, z = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record()
        moe.moe_router_logits(layer.cfg, x_d, layer.wr, layer.offset, L_d,
                              status)
        r.record()
        g.launch()
        z.record()
        hist[i].copy_(trace, non_blocking=True)
        evs.append((a, r, z))
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clock_rec = clocks.stop() if clocks is not None else None
    if int(status.item()) != 0:
        raise SystemExit(f"device status {int(status.item())}")
    ms = [a.elapsed_time(z) for a, _, z in evs]
    mean_ms = max_over_ranks(sum(ms) / len(ms), device)
    stamps = hist.cpu().numpy()
    stage_ms = {"router": sum(a.elapsed_time(r) for a, r, _ in evs)}
    for i in range(n):
        for name, d in trace_stage_ms(stamps[i], len(passes)).items():
            if layer.dispatch_only and name.startswith("gmm"):
                continue    # no expert FFN: two adjacent stamps
            stage_ms[name] = stage_ms.get(name, 0.0) + d
    kernels, work = stage_table(layer, passes, stage_ms, mean_ms, n)
    staged = sum(stage_ms.values()) / n
    kernels["graph_gaps"] = {
        "ms_per_step": round(mean_ms - staged, 4),
        "share": round((mean_ms - staged) / mean_ms, 4),
        "note": "step time not inside a stage: graph launch, the branch "
                "select kernel and the stamp kernels between stages"}
    # warm L2: the same launches without the flush
    wz = []
    for _ in range(min(n, 20)):
        a, z = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        a.record()
        run()
        z.record()
        wz.append((a, z))
    torch.cuda.synchronize()
    warm = sum(a.elapsed_time(z) for a, z in wz) / len(wz)
    res.update({
        "timed_step": "moe_router_logits + moe_layer_graph_launch of the "
                      "traced layer graph (route, check, conditional node: "
                      "capped pass | chunked fallback); CUDA events around "
                      "each step on the launch stream, stage times from the "
                      "graph's device timestamps at every stage boundary",
        "value": round(whole_job_tokens_per_s(world, T, mean_ms), 1),
        "ms_per_step": round(mean_ms, 4),
        "ms_per_step_median": round(float(np.median(ms)), 4),
        "wall_s_timed_loop": round(wall, 3), "steps_timed": n,
        "kernels": kernels,
        "roofline": roofline_of(layer, passes, stage_ms, work, n),
        "check_us": round(kernels["check"]["ms_per_step"] * 1e3, 2),
        "gpu_launches": graph_launches(
            passes, layer.wl.T, layer.wl.S, planned, layer.chunk,
            moe.moe_num_chunks(layer.cfg)) * n,
        "warm_l2": {"value": round(whole_job_tokens_per_s(world, T, warm),
                                   1),
                    "unit": UNIT, "ms_per_step": round(warm, 4),
                    "note": "the timed launches without the L2 flush"},
        "stepwise": {"value": round(whole_job_tokens_per_s(world, T,
                                                           sw_mean), 1),
                     "ms_per_step": round(sw_mean, 4),
                     "note": "the same layer through the stepwise entry "
                             "points with the host reading the overflow "
                             "flag, CUDA events between stages",
                     "permute_frac": hbm_frac(sw_kernels, "permute"),
                     "combine_frac": hbm_frac(sw_kernels, "combine")},
        "clocks": clock_rec})
    res["permute_frac"] = hbm_frac(kernels, "permute")
    res["combine_frac"] = hbm_frac(kernels, "combine")
    g.close()
    if graph_too:
        gr = graph_run(layer, steps, warmup, device)
        if gr is not None:
            gr["graph"].close()
            res["untraced_graph"] = {
                "value": round(whole_job_tokens_per_s(world, T,
                                                      gr["ms_per_step"]), 1),
                "ms_per_step": round(gr["ms_per_step"], 4),
                "note": "moe_router_logits + moe_layer_graph_launch without "
                        "the stage stamps"}
    del hist, trace, ws, x_d, L_d, y_d
    return res


CONFIG_STEPS = 10


def config_runs(args, device, flush, head):
    """Every other workload of the benchmark at 1 GPU, each a short timed
    run of its own (few steps; at least ~0.4 s of timed work for the clock
    sampler): the tiny and small layers, the DeepSeek-V3 layer as one
    uncapped pass under uniform and Zipf routing (the regime in which the
    GEMMs lean on the tensor cores), the Llama4-Maverick layer, and the
    routing/permute/dedup sweep.  Returns a list of compact records."""
    from synth import SWEEP_ROUTINGS, SWEEP_TOKENS, sweep_workload
    runs = [("dsv3", WORKLOADS["dsv3"], "fallback")]
    runs += [(n, WORKLOADS[n], "fallback") for n in ("tiny", "small")]
    runs += [("dsv3_uncapped_uniform",
              WORKLOADS["dsv3"].with_(routing="uniform", zipf_s=0.0,
                                      name="dsv3_uniform"), "dropless"),
             ("dsv3_uncapped_zipf", WORKLOADS["dsv3"], "dropless"),
             ("l4mav", WORKLOADS["l4mav"], "fallback")]
    runs += [(f"sweep_T{T}_{r}", sweep_workload(T, r), "fallback")
             for T in SWEEP_TOKENS for r in SWEEP_ROUTINGS]
    out = []
    for label, wl, mode in runs:
        if label == "dsv3":
            res = head
        else:
            layer = Layer(wl, device, mode=mode)
            res = measure_layer(layer, CONFIG_STEPS, 3, device, flush,
                                clocks=ClockSampler(device), exact=False,
                                graph_too=mode == "fallback")
            del layer
            torch.cuda.empty_cache()
        rec = {"config": label, "T": wl.T, "mode": mode,
               "routing": wl.routing, "dtype": wl.dtype,
               "value": res["value"], "unit": UNIT,
               "ms_per_step": res["ms_per_step"],
               "overflow": res["overflow"], "passes": res["passes"],
               "timed": "traced graph" if res["timed_step"].startswith(
                   "moe_router_logits + moe_layer_graph") else "stepwise",
               "steps_timed": res.get("steps_timed")}
        roof = res["roofline"]
        rec["dominant"] = {k: roof[k] for k in (
            "kernel", "bound", "achieved", "unit", "peak", "frac")}
        if "tensor_TFLOPs" in roof:
            rec["dominant"]["tensor_TFLOPs"] = roof["tensor_TFLOPs"]
            rec["dominant"]["tensor_frac_of_burst"] = \
                roof["tensor_frac_of_burst"]
        gm = [res["kernels"][n] for n in ("gmm_gate_up", "gmm_down")
              if n in res["kernels"]]
        if len(gm) == 2 and all("TFLOPs" in g_ for g_ in gm):
            ms = gm[0]["ms_per_step"] + gm[1]["ms_per_step"]
            fl = sum(g_["TFLOPs"] * g_["ms_per_step"] for g_ in gm) / ms
            peaks, _ = load_peaks()
            rec["gmm_TFLOPs"] = round(fl, 1)
            rec["gmm_tensor_frac_of_burst"] = round(
                fl / peaks["bf16_tflops"], 4)
            rec["gmm_tensor_frac_of_sustained"] = round(
                fl / peaks["bf16_tflops_sustained"], 4)
        rec["permute_frac"] = res.get("permute_frac")
        rec["combine_frac"] = res.get("combine_frac")
        if "untraced_graph" in res:
            # the same graph without the stage stamps (1 µs a stage, which
            # matters in steps of a few tens of µs)
            rec["untraced_value"] = res["untraced_graph"]["value"]
            rec["untraced_ms_per_step"] = \
                res["untraced_graph"]["ms_per_step"]
        if "check_us" in res:
            rec["check_us"] = res["check_us"]
        rec["clocks"] = res.get("clocks")
        out.append(rec)
    return out


def graph_run(layer, steps, warmup, device):
    """The same layer as one CUDA graph launch per step (moe_layer_graph):
    device-resident throughput, and the bits checked against the stepwise
    result."""
    if layer.mode != "fallback":
        return None
    moe = layer.moe
    x_d = layer.x.clone()
    L_d = layer.logits.clone()
    y_d = torch.empty_like(layer.b["y"])
    ws = moe.layer_workspace(layer.cfg, moe.MOE_WS_LAYER, device)
    W = layer.W if layer.W is not None else (None, None, None)
    g = moe.MoeLayerGraph(layer.cfg, x_d, L_d, *W, y_d, ws)

    def run():   # router logits, then the layer graph
        moe.moe_router_logits(layer.cfg, x_d, layer.wr, layer.offset, L_d)
        g.launch()
    run()
    torch.cuda.synchronize()
    if not torch.equal(y_d, layer.b["y"]):
        raise SystemExit("graph path and stepwise path disagree")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    for _ in range(warmup):
        flush.zero_()
        run()
    ms = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), \
            torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    mean = max_over_ranks(sum(ms) / len(ms), device)
    return {"graph": g, "x": x_d, "logits": L_d, "y": y_d, "ws": ws,
            "ms_per_step": mean}


def e2e_pipelined(layer, args, world, device):
    """Same metric end to end through moe_layer_graph with two buffer sets:
    every step copies its x and logits from pinned host memory and its y
    back, on a copy stream that overlaps the neighbouring steps' compute
    (step i+1's inputs go in while step i runs; step i's output comes back
    while step i+1 runs).  One workspace, one compute stream: the layers
    themselves run one after another."""
    moe = layer.moe
    x_h = layer.x.cpu().pin_memory()
    O_h = None if layer.offset is None else layer.offset.cpu().pin_memory()
    y_h = [torch.empty(layer.b["y"].shape, dtype=layer.b["y"].dtype,
                       pin_memory=True) for _ in range(2)]
    ws = moe.layer_workspace(layer.cfg, moe.MOE_WS_LAYER, device)
    L_d = torch.empty_like(layer.logits)   # one compute stream: one copy
    sets = []
    for _ in range(2):
        x_d = torch.empty_like(layer.x)
        O_d = None if O_h is None else torch.empty_like(layer.offset)
        y_d = torch.empty_like(layer.b["y"])
        g = moe.MoeLayerGraph(layer.cfg, x_d, L_d, *layer.W, y_d, ws)
        sets.append((x_d, O_d, y_d, g))
    comp = torch.cuda.current_stream()
    up = torch.cuda.Stream(device=device)     # host -> device
    down = torch.cuda.Stream(device=device)   # device -> host
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
    free = [ev(), ev()]
    for e in free:
        e.record(down)

    def steps(n):
        for i in range(n):
            b = i % 2
            x_d, O_d, y_d, g = sets[b]
            with torch.cuda.stream(up):
                up.wait_event(free[b])       # buffer b's last output is out
                x_d.copy_(x_h, non_blocking=True)
                if O_d is not None:
                    O_d.copy_(O_h, non_blocking=True)
                h2d = ev()
                h2d.record(up)
            comp.wait_event(h2d)
            moe.moe_router_logits(layer.cfg, x_d, layer.wr, O_d, L_d,
                                  stream=comp)
            g.launch(comp)
            done = ev()
            done.record(comp)
            with torch.cuda.stream(down):
                down.wait_event(done)
                y_h[b].copy_(y_d, non_blocking=True)
                free[b].record(down)

    steps(max(1, args.warmup))
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record(comp)
    up.wait_event(a)
    down.wait_event(a)
    steps(args.steps)
    comp.wait_stream(up)
    comp.wait_stream(down)
    z.record(comp)
    z.synchronize()
    mean = max_over_ranks(a.elapsed_time(z) / args.steps, device)
    # the last step's output reached the host and equals the device result
    if not torch.equal(y_h[(args.steps - 1) % 2], layer.b["y"].cpu()):
        raise SystemExit("pipelined end-to-end output differs")
    for s_ in sets:
        s_[3].close()
    h2d = x_h.numel() * x_h.element_size() + \
        (0 if O_h is None else O_h.numel() * O_h.element_size())
    d2h = y_h[0].numel() * y_h[0].element_size()
    return {"value": round(whole_job_tokens_per_s(world, layer.wl.T, mean), 1),
            "unit": UNIT, "ms_per_step": round(mean, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "api": "moe_router_logits + moe_layer_graph_launch (C ABI), "
                   "pinned host buffers (x and the logit offset in, y out), "
                   "copies on two copy streams overlapping neighbouring "
                   "steps"}


def e2e_run(layer, args, world, device, graph=None):
    """Same metric end to end: pinned host x and logit offset copied in, the
    router and the layer, y copied out, every step.  Through moe_layer_graph
    when available (one launch per layer), else moe_layer."""
    moe = layer.moe
    x_h = layer.x.cpu().pin_memory()
    O_h = None if layer.offset is None else layer.offset.cpu().pin_memory()
    y_h = torch.empty(layer.b["y"].shape, dtype=layer.b["y"].dtype,
                      pin_memory=True)
    O_d = None if O_h is None else torch.empty_like(layer.offset)
    if graph is not None:
        x_d, L_d, y_d = graph["x"], graph["logits"], graph["y"]
        api = "moe_router_logits + moe_layer_graph_launch (C ABI), pinned " \
            "host buffers"

        def run_layer():
            graph["graph"].launch()
    else:
        x_d = torch.empty_like(layer.x)
        L_d = torch.empty_like(layer.logits)
        y_d = torch.empty_like(layer.b["y"])
        api = "moe_router_logits + moe_layer (C ABI), pinned host buffers"

        def run_layer():
            layer.api_layer(x_d, L_d, y_d)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def one():
        x_d.copy_(x_h, non_blocking=True)
        if O_d is not None:
            O_d.copy_(O_h, non_blocking=True)
        moe.moe_router_logits(layer.cfg, x_d, layer.wr, O_d, L_d)
        run_layer()
        y_h.copy_(y_d, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        flush.zero_()
        one()
    torch.cuda.synchronize()
    ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), \
            torch.cuda.Event(enable_timing=True)
        a.record()
        one()
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    mean = max_over_ranks(sum(ms) / len(ms), device)
    h2d = x_h.numel() * x_h.element_size() + \
        (0 if O_h is None else O_h.numel() * O_h.element_size())
    d2h = y_h.numel() * y_h.element_size()
    return {"value": round(whole_job_tokens_per_s(world, layer.wl.T, mean), 1),
            "unit": UNIT, "ms_per_step": round(mean, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "api": api}


def cpu_baseline(layer):
    wl = layer.wl
    n = CPU_SAMPLE.get(wl.name, 32)
    sec, n = oracle_sample_run(wl, layer.x, layer.wr, layer.offset_np,
                               layer.W, n, mode=layer.mode)
    return {"value": round(n / sec, 4), "unit": UNIT, "cores": _CORES,
            "kind": "oracle",
            "sample": f"first {n} tokens of the {wl.name} batch run as a "
                      f"layer of their own (same H, E, k, F, S, factor; "
                      f"float64 numpy oracle incl. router logits, routing, "
                      f"check, fallback, "
                      f"FFN and combine); {sec:.1f} s"}


# ------------------------------------------------------------ backward ----
class Backward:
    """Buffers and the stepwise backward of one layer (inputs and forward
    buffers shared with the Layer)."""

    def __init__(self, layer):
        moe, c, w = layer.moe, layer.cfg, layer.wl
        dev = layer.x.device
        T, H, E, k, F = w.T, w.H, w.E, w.k, w.F
        R = T * k
        dt = layer.x.dtype
        self.layer = layer
        self.dy = make_dy(w, dev)
        self.g, self.u, self.dg, self.du = (
            torch.empty((R, F), dtype=dt, device=dev) for _ in range(4))
        self.dys = torch.empty((R, H), dtype=dt, device=dev)
        self.dxs = torch.empty((R, H), dtype=dt, device=dev)
        self.dtw = torch.empty((T, k), dtype=torch.float32, device=dev)
        # the split combine backward (bf16 with regrouped weight gradients):
        # each row's combine weight and the down dgrad's row dots
        self.parts = max(1, moe.moe_row_dot_parts(c))
        self.wrow = torch.empty(R, dtype=torch.float32, device=dev)
        self.rdot = torch.empty(R * self.parts, dtype=torch.float32,
                                device=dev)
        self.dx = torch.empty((T, H), dtype=dt, device=dev)
        self.dl = torch.empty((T, E), dtype=torch.float32, device=dev)
        self.dw = [torch.empty((E, H, F), dtype=torch.float32, device=dev),
                   torch.empty((E, H, F), dtype=torch.float32, device=dev),
                   torch.empty((E, F, H), dtype=torch.float32, device=dev)]
        n_max = max(1, moe.moe_num_chunks(c))
        G = E + w.S * w.redundant_slots     # groups with duplicate slots
        self.G = G
        self.goff = [torch.empty(G + 1, dtype=torch.int32, device=dev)
                     for _ in range(n_max)]
        # the passes' rows regrouped for the weight gradients (bf16, as
        # moe_layer_backward does)
        self.regroup = w.dtype == "bf16"
        rr = R + 16 * G
        self.rr = rr
        if self.regroup:
            self.xs2 = torch.empty((rr, H), dtype=dt, device=dev)
            self.dys2 = torch.empty((rr, H), dtype=dt, device=dev)
            self.dg2, self.du2, self.h2 = (
                torch.empty((rr, F), dtype=dt, device=dev) for _ in range(3))
            self.off2 = torch.empty(G + 1, dtype=torch.int32, device=dev)
        self.ws = moe.layer_workspace(c, moe.MOE_WS_LAYER_BACKWARD, dev)
        # every pass keeps its own rows, row_of rows and group offsets; the
        # dedup outputs and the permute scratch come in two sets, so that a
        # pass's permute tables can run on the side stream ahead of it
        b = layer.b
        keys = ("uniq_offsets", "uniq_tokens", "n_dropped", "permute_ws")
        self.tabs = [{k: b[k] for k in keys},
                     {k: torch.empty_like(b[k]) for k in keys}]
        self.pass_events = []   # (tables ready, scatter done) per pass

    def tables(self, pas, i, stream, ready, after=None, on_plan=False):
        """Permute tables of backward pass i (tokens pas = (t0, t1, capped))
        into its own row ranges and dedup set i % 2, on `stream`."""
        lay = self.layer
        moe, b, k = lay.moe, lay.b, lay.cfg.k
        t0, t1, capped = pas
        sc = lay.sub(t0, t1, capped)
        tb = self.tabs[i % 2]
        plan = dict(divert=b["divert"], slot_of=b["slot_of"]) if on_plan \
            else {}
        if after is not None:
            stream.wait_event(after)
        moe.moe_permute_tables(
            sc, b["topk_idx"][t0:t1], capped, b["row_of"][t0:t1],
            b["sorted_token"][t0 * k:], self.goff[i], tb["uniq_offsets"],
            tb["n_dropped"], tb["permute_ws"], stream=stream, **plan)
        ready.record(stream)

    def step(self, ev=None):
        L = self
        lay = self.layer
        moe, b, c, W = lay.moe, lay.b, lay.cfg, lay.W
        k = c.k
        mark = ev or (lambda name: None)
        mark("route")
        moe.moe_route(c, lay.logits, b["topk_idx"], b["topk_w"], b["status"])
        lay.routed.record()   # the side stream's tables start after it
        # duplicate-expert slots: check and plan first (as moe_layer_backward)
        planned = c.redundant_slots > 0 and lay.mode != "dropless"
        if planned or lay.mode == "fallback":
            mark("check")
            moe.moe_check_overflow(c, b["topk_idx"], b["expert_counts"],
                                   b["expert_offsets"], b["shard_counts"],
                                   b["overflow_flag"], b["required_factor"],
                                   b["capacity"])
        if planned:
            mark("plan")
            moe.moe_plan_duplication(c, b["expert_counts"], b["divert"],
                                     b["slot_of"], b["group_expert"],
                                     b["shard_after"], b["flag_after"])
        main, side = torch.cuda.current_stream(), lay.side
        if lay.mode != "fallback":
            passes = [(0, c.T, lay.mode == "capped")]
        else:
            mark("flag")
            flag = b["flag_after"] if planned else b["overflow_flag"]
            if int(flag.item()):
                passes = [(t0, min(c.T, t0 + lay.chunk), False)
                          for t0 in range(0, c.T, lay.chunk)]
            else:
                passes = [(0, c.T, True)]
        # the plan's virtual groups for a capped pass, else the experts'
        on_plan = planned and passes[0][2]
        grp = dict(n_groups=L.G, group_expert=b["group_expert"]) \
            if on_plan else {}
        xs, h, ys = b["x_sorted"], b["h"], b["y_sorted"]
        # as moe_layer_backward: with bf16 and regrouped weight gradients the
        # combine weights' gradient comes from the down dgrad (no GEMM2)
        split = L.regroup and len(passes) <= 64
        while len(L.pass_events) < len(passes):
            L.pass_events.append((torch.cuda.Event(), torch.cuda.Event()))
        ready = [e[0] for e in L.pass_events]
        scattered = [e[1] for e in L.pass_events]
        for i, (t0, t1, capped) in enumerate(passes):
            sc = lay.sub(t0, t1, capped)
            r0 = t0 * k
            go = L.goff[i]
            tb = L.tabs[i % 2]
            mark("permute")
            if i == 0:
                L.tables(passes[0], 0, main, ready[0], on_plan=on_plan)
            else:
                main.wait_event(ready[i])
            moe.moe_permute_scatter(sc, lay.x[t0:t1], b["row_of"][t0:t1],
                                    tb["uniq_offsets"], xs[r0:],
                                    tb["uniq_tokens"], b["expand_idx"][r0:],
                                    tb["permute_ws"])
            scattered[i].record(main)
            mark("gmm_gate_up_saved")
            moe.moe_gmm_gate_up_saved(sc, xs[r0:], go, W[0], W[1], L.g[r0:],
                                      L.u[r0:], h[r0:], b["status"], **grp)
            if i + 1 < len(passes):
                # queued once the GPU has this pass's GEMM to run; the next
                # pass's tables reuse the dedup set of pass i-1, which only
                # that pass's scatter reads
                L.tables(passes[i + 1], i + 1, side, ready[i + 1],
                         scattered[i - 1] if i >= 1 else lay.routed)
            if split:
                mark("combine_bwd")
                moe.moe_combine_backward_rows(
                    sc, L.dy[t0:t1], b["row_of"][t0:t1], b["topk_w"][t0:t1],
                    L.dys[r0:], L.wrow[r0:])
                mark("gmm_down_dgrad")
                rd = L.rdot[r0 * L.parts:]
                moe.moe_gmm_down_dgrad_rows(sc, go, W[2], L.g[r0:], L.u[r0:],
                                            h[r0:], L.dys[r0:], L.wrow[r0:],
                                            L.dg[r0:], L.du[r0:], rd,
                                            b["status"], **grp)
                mark("combine_wgrad")
                moe.moe_combine_weight_grad(sc, b["row_of"][t0:t1], rd,
                                            L.dtw[t0:t1])
            else:
                mark("gmm_down")
                moe.moe_gmm_down(sc, h[r0:], go, W[2], ys[r0:], b["status"],
                                 **grp)
                mark("combine_bwd")
                moe.moe_combine_backward(sc, L.dy[t0:t1], ys[r0:],
                                         b["row_of"][t0:t1],
                                         b["topk_w"][t0:t1], L.dys[r0:],
                                         L.dtw[t0:t1])
                mark("gmm_down_dgrad")
                moe.moe_gmm_down_dgrad(sc, go, W[2], L.g[r0:], L.u[r0:],
                                       L.dys[r0:], L.dg[r0:], L.du[r0:],
                                       b["status"], **grp)
            mark("gmm_gate_up_dgrad")
            moe.moe_gmm_gate_up_dgrad(sc, go, W[0], W[1], L.dg[r0:],
                                      L.du[r0:], L.dxs[r0:], b["status"],
                                      **grp)
            mark("permute_bwd")
            moe.moe_permute_backward(sc, L.dxs[r0:], b["row_of"][t0:t1],
                                     L.dx[t0:t1])
        mark("route_bwd")
        moe.moe_route_backward(c, lay.logits, b["topk_idx"], L.dtw, L.dl)
        segs = [(L.goff[i], t0 * k) for i, (t0, _, _) in enumerate(passes)]
        if L.regroup and len(passes) <= 64:
            mark("regroup")
            moe.moe_regroup_rows(c, segs, L.rr, xs, L.dg, L.du, h, L.dys,
                                 L.xs2, L.dg2, L.du2, L.h2, L.dys2, L.off2,
                                 n_groups=L.G if on_plan else 0,
                                 w_row=L.wrow)
            segs, rows = [(L.off2, 0)], L.rr
            wx, wdg, wdu, wh, wdy = L.xs2, L.dg2, L.du2, L.h2, L.dys2
            flags = moe.MOE_WGRAD_ROWS16     # 16-row groups, zero pad rows
        else:
            rows = c.T * k
            wx, wdg, wdu, wh, wdy = xs, L.dg, L.du, h, L.dys
            flags = 0
        mark("gmm_gate_up_wgrad")
        moe.moe_gmm_gate_up_wgrad(c, segs, rows, wx, wdg, wdu,
                                  L.dw[0], L.dw[1], flags, b["status"], **grp)
        mark("gmm_down_wgrad")
        moe.moe_gmm_down_wgrad(c, segs, rows, wh, wdy, L.dw[2], flags,
                               b["status"], **grp)
        mark(None)
        return passes

    def api(self, x, logits, dy, dx, dl):
        moe = self.layer.moe
        mode = {"fallback": moe.MOE_MODE_FALLBACK_LAYER,
                "capped": moe.MOE_MODE_CAPPED,
                "dropless": moe.MOE_MODE_DROPLESS}[self.layer.mode]
        return moe.moe_layer_backward(self.layer.cfg, x, logits,
                                      *self.layer.W, dy, dx, dl, *self.dw_api,
                                      mode, self.ws, self.layer.b["status"])


def backward_launches(passes, mode, regroup, planned=False, shards=0):
    """Kernel launches of one backward step: route (+ check, + the plan with
    duplicate slots), per pass the permute tables (table_launches) + scatter
    + GEMM1-saved + the combine backward's dy rows + the down dgrad + the
    combine weights' gradient + the gate/up dgrad + permute backward (with
    the row segments in batches: GEMM2 + combine backward + the two dgrads +
    permute backward), route backward, the regrouping of the rows (2) or the
    row segments in batches of 16, and per batch the two weight-gradient
    GEMMs, plus the two fills in the first batch that zero the experts not
    written by exactly one group."""
    n = len(passes)
    batches = 1 if regroup else (n + 15) // 16
    head = 1 + (1 if (mode == "fallback" or planned) else 0) + \
        (1 if planned else 0)
    return head + sum(table_launches(t1 - t0, shards) + 7
                      for (t0, t1, _) in passes) + 1 + \
        (2 if regroup else 0) + 2 * batches + 2


def backward_work(w, accs):
    """Algorithmic bytes and flops of each backward stage over the step."""
    b = 2 if w.dtype == "bf16" else 4
    H, F, k, E = w.H, w.F, w.k, w.E
    split = w.dtype == "bf16" and len(accs) <= 64
    parts = F // 256 if F % 256 == 0 else F // 128
    out = {}

    def add(name, by, fl):
        t = out.setdefault(name, {"bytes": 0, "flops": 0, "launches": 0})
        t["bytes"] += by
        t["flops"] += fl
        t["launches"] += 1
    R_tot = 0
    T_tot = 0
    for a in accs:
        T, R, Ea = a["T"], a["R"], a["E_act"]
        R_tot += R
        T_tot += T
        add("permute", T * H * b + R * H * b + 16 * R, 0)
        add("gmm_gate_up_saved", 2 * Ea * H * F * b + R * H * b + 3 * R * F * b,
            4 * R * H * F)
        if split:
            # dy rows unscaled + each row's weight; the dgrad also reads h
            # and writes the row dots; the weights' gradient sums them
            add("combine_bwd", T * H * b + R * H * b + 12 * T * k + 4 * R, 0)
            add("gmm_down_dgrad", Ea * F * H * b + R * H * b + 5 * R * F * b
                + 4 * R + 4 * R * parts, 2 * R * H * F)
            add("combine_wgrad", 4 * R * parts + 8 * T * k, 0)
        else:
            add("gmm_down", Ea * F * H * b + R * F * b + R * H * b,
                2 * R * F * H)
            add("combine_bwd", T * H * b + 2 * R * H * b + 12 * T * k, 0)
            add("gmm_down_dgrad", Ea * F * H * b + R * H * b + 4 * R * F * b,
                2 * R * H * F)
        add("gmm_gate_up_dgrad", 2 * Ea * H * F * b + 2 * R * F * b + R * H * b,
            4 * R * H * F)
        add("permute_bwd", R * H * b + T * H * b + 4 * T * k, 0)
    add("route_bwd", 8 * T_tot * E + 8 * T_tot * k, 0)
    # the five row buffers read once and written once (pad rows not counted)
    add("regroup", 2 * R_tot * (2 * H + 3 * F) * b + (4 * R_tot if split
                                                       else 0), 0)
    add("gmm_gate_up_wgrad", R_tot * H * b + 2 * R_tot * F * b + 2 * E * H * F * 4,
        4 * R_tot * H * F)
    add("gmm_down_wgrad", R_tot * F * b + R_tot * H * b + E * F * H * 4,
        2 * R_tot * H * F)
    return out


def oracle_backward_sample(wl, x_dev, wr, offset, W, dy_dev, n_tok, mode):
    """The oracle's backward of the mode on tokens [0, n_tok) as a layer of
    their own: routing (on the oracle's own router logits), check, the
    capped pass or the chunked passes, each pass's full backward (weight
    gradients of the experts it touched)."""
    from oracle import moe_ref as ref
    n = min(n_tok, wl.T)
    xs = x_dev[:n].to("cpu", torch.float64).numpy()
    dys = dy_dev[:n].to("cpu", torch.float64).numpy()
    Ls = ref.router_logits(xs, wr.to("cpu", torch.float64).numpy(),
                           None if offset is None else offset[:n])
    idx, _, _ = ref.route(Ls, wl.k, wl.renorm)
    touched = sorted(set(int(e) for e in idx.reshape(-1)))
    host = {e: (W[0][e].cpu(), W[1][e].cpu(), W[2][e].cpu()) for e in touched}

    def weights(e):
        g, u, d = host[e]
        return (g.to(torch.float64).numpy(), u.to(torch.float64).numpy(),
                d.to(torch.float64).numpy())
    t = time.perf_counter()
    idx, _, _ = ref.route(Ls, wl.k, wl.renorm)
    C = ref.capacity(n, wl.k, wl.S, wl.factor)
    counts = ref.expert_counts(idx, wl.E)
    groups = None
    load = ref.shard_counts(counts, wl.S)
    if wl.redundant_slots > 0 and mode != "dropless":
        B = wl.redundant_slots
        plan = ref.plan_duplication(counts, wl.S, B)
        vidx = ref.reroute(idx, plan, wl.E, wl.S)
        G = wl.S * (wl.E // wl.S + B)
        groups = (vidx, G, plan.group_expert)
        load = ref.shard_counts(ref.expert_counts(vidx, G), wl.S)
    if mode == "dropless":
        passes = [(0, n, None)]
    elif mode == "capped":
        passes = [(0, n, C)]
    elif ref.overflow_flag(load, C):
        passes = [(t0, t1, None) for (t0, t1) in
                  ref.chunk_plan(n, wl.k, wl.E, wl.S, C, wl.n_chunks)]
        groups = None    # the fallback's chunks run plain
    else:
        passes = [(0, n, C)]
    for (t0, t1, Cp) in passes:
        sub = ref.MoEConfig(t1 - t0, wl.H, wl.E, wl.k, wl.F, wl.S,
                            wl.factor if Cp is not None else -1.0, 0,
                            wl.renorm)
        ref.pass_backward_touched(sub, xs[t0:t1], Ls[t0:t1], weights,
                                  dys[t0:t1], Cp, groups)
    return time.perf_counter() - t, n


def backward_main(layer, args, world, rank, device):
    moe = layer.moe
    bw = Backward(layer)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    # identical bits: stepwise entry points vs moe_layer_backward
    passes = bw.step()
    torch.cuda.synchronize()
    dx_api = torch.empty_like(bw.dx)
    dl_api = torch.empty_like(bw.dl)
    bw.dw_api = [torch.empty_like(t) for t in bw.dw]
    info = bw.api(layer.x, layer.logits, bw.dy, dx_api, dl_api)
    torch.cuda.synchronize()
    same = torch.equal(dx_api, bw.dx) and torch.equal(dl_api, bw.dl) and \
        all(torch.equal(a, b) for a, b in zip(bw.dw_api, bw.dw))
    if not same:
        raise SystemExit("stepwise backward and moe_layer_backward disagree")
    if int(layer.b["status"].item()) != 0:
        raise SystemExit(f"device status {int(layer.b['status'].item())}")
    del bw.dw_api
    for _ in range(args.warmup):
        flush.zero_()
        bw.step()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
    clocks = ClockSampler(device)
    timers = []
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    wall0 = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()
        st = StageTimer()
        passes = bw.step(st)
        timers.append(st)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier()
    clock_rec = clocks.stop()
    step_ms = [sum(d for _, d in st.durations()) for st in timers]
    mean_ms = max_over_ranks(sum(step_ms) / len(step_ms), device)
    stage = {}
    for st in timers:
        for name, d in st.durations():
            s_ = stage.setdefault(name, {"ms": 0.0, "n": 0})
            s_["ms"] += d
            s_["n"] += 1
    planned = layer.cfg.redundant_slots > 0 and layer.mode != "dropless"
    on_plan = planned and passes[0][2]
    if on_plan:   # the virtual groups' offsets, for the accounting only
        layer.b["group_offsets"][:bw.G + 1].copy_(bw.goff[0])
    work = backward_work(layer.wl, pass_accounting(layer, passes))
    peaks, peak_src = load_peaks()
    kernels = {}
    for name, s_ in stage.items():
        per_step = s_["ms"] / args.steps
        ent = {"ms_per_step": round(per_step, 4),
               "launch_groups_per_step": s_["n"] // args.steps,
               "share": round(per_step / mean_ms, 4)}
        if name in work:
            wv = work[name]
            sec = per_step / 1e3
            ent["GBps"] = round(wv["bytes"] / sec / 1e9, 1)
            if wv["flops"]:
                ent["TFLOPs"] = round(wv["flops"] / sec / 1e12, 1)
        kernels[name] = ent
    # dominant kernel: the single-kernel stage with the most time
    single = [n for n in work if n in stage and n != "permute"]
    dom = max(single, key=lambda n: stage[n]["ms"])
    wv = work[dom]
    n_launch = wv["launches"]
    dur = stage[dom]["ms"] / args.steps / n_launch / 1e3
    bytes_l, flops_l = wv["bytes"] / n_launch, wv["flops"] / n_launch
    t_mem = bytes_l / (peaks["hbm_gbs"] * 1e9)
    t_flop = flops_l / (peaks["bf16_tflops_sustained"] * 1e12) if flops_l else 0
    if t_mem >= t_flop:
        achieved = bytes_l / dur / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        achieved = flops_l / dur / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1),
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s"}
    roof["frac"] = round(achieved / roof["peak"], 4)
    roof["traffic"] = profiled_traffic(dom, layer.wl.name)
    roof["kernel"] = dom
    roof["algorithmic_bytes_per_launch"] = int(bytes_l)
    roof["algorithmic_flops_per_launch"] = int(flops_l)
    roof["launch_ms"] = round(dur * 1e3, 4)
    roof["peak_source"] = f"{peak_src} MEASURED_PEAKS.json" \
        if peak_src == "measured" else "fallback"
    w = layer.wl
    out = {
        "metric": METRIC_BWD, "value": None, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded; router logits, x, dy N(0,1), expert "
                "weights N(0,0.02))",
        "config": {
            "workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k,
            "F": w.F, "S": w.S, "ragged_buffer_factor": w.factor,
            "routing": w.routing + (f" s={w.zipf_s}" if w.routing == "zipf"
                                    else ""),
            "mode": layer.mode, "overflow": info["overflow"],
            "passes": len(passes), "capacity": info["capacity"],
            "redundant_slots": w.redundant_slots,
            "pass": "backward: forward recomputed per pass, dW float32 "
                    "written once over all passes",
            "l2": "flushed between steps (256 MiB write, outside the events)",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
        },
        "wall_s_timed_loop": round(wall, 3),
        "gpu_launches": backward_launches(
            passes, layer.mode, bw.regroup and len(passes) <= 64,
            planned, layer.wl.S) * args.steps,
        "kernels": kernels,
        "roofline": roof,
    }
    out["value"] = round(whole_job_tokens_per_s(world, w.T, mean_ms), 1)
    if clock_rec:
        out["clocks"] = clock_rec
    if not args.no_e2e:
        out["e2e"] = backward_e2e_pipelined(bw, args, world, device)
        out["e2e"]["serial"] = backward_e2e(bw, args, world, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = BWD_CPU_SAMPLE.get(w.name, 8)
        sec, n = oracle_backward_sample(w, layer.x, layer.wr, layer.offset_np,
                                         layer.W,
                                        bw.dy, n, layer.mode)
        out["cpu_baseline"] = {
            "value": round(n / sec, 4), "unit": UNIT, "cores": _CORES,
            "kind": "oracle",
            "sample": f"backward of the first {n} tokens of the {w.name} "
                      f"batch as a layer of their own (float64 oracle: "
                      f"routing, check, passes, FFN backward, weight "
                      f"gradients of the touched experts); {sec:.1f} s"}
    if rank == 0:
        print(json.dumps(out))


def backward_e2e(bw, args, world, device):
    """moe_layer_backward with pinned host x, logits and dy copied in and
    dx and dlogits copied out inside the timed region, every step."""
    lay = bw.layer
    x_h = lay.x.cpu().pin_memory()
    L_h = lay.logits.cpu().pin_memory()
    dy_h = bw.dy.cpu().pin_memory()
    dx_h = torch.empty(bw.dx.shape, dtype=bw.dx.dtype, pin_memory=True)
    dl_h = torch.empty(bw.dl.shape, dtype=bw.dl.dtype, pin_memory=True)
    x_d, L_d, dy_d = (torch.empty_like(t) for t in (lay.x, lay.logits, bw.dy))
    dx_d, dl_d = torch.empty_like(bw.dx), torch.empty_like(bw.dl)
    bw.dw_api = bw.dw
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def one():
        x_d.copy_(x_h, non_blocking=True)
        L_d.copy_(L_h, non_blocking=True)
        dy_d.copy_(dy_h, non_blocking=True)
        bw.api(x_d, L_d, dy_d, dx_d, dl_d)
        dx_h.copy_(dx_d, non_blocking=True)
        dl_h.copy_(dl_d, non_blocking=True)
    for _ in range(max(1, args.warmup)):
        flush.zero_()
        one()
    torch.cuda.synchronize()
    ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), \
            torch.cuda.Event(enable_timing=True)
        a.record()
        one()
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    mean = max_over_ranks(sum(ms) / len(ms), device)
    if not torch.equal(dx_h, bw.dx.cpu()):
        raise SystemExit("end-to-end backward output differs")
    h2d = sum(t.numel() * t.element_size() for t in (x_h, L_h, dy_h))
    d2h = sum(t.numel() * t.element_size() for t in (dx_h, dl_h))
    return {"value": round(whole_job_tokens_per_s(world, lay.wl.T, mean), 1),
            "unit": UNIT, "ms_per_step": round(mean, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "api": "moe_layer_backward (C ABI), pinned host buffers"}


def backward_e2e_pipelined(bw, args, world, device):
    """moe_layer_backward end to end with two sets of device inputs and
    outputs: step i+1's x, logits and dy go in on one copy stream while step
    i runs, step i's dx and dlogits come out on another while step i+1 runs.
    One workspace and one compute stream: the backward steps themselves run
    one after another."""
    lay = bw.layer
    x_h = lay.x.cpu().pin_memory()
    L_h = lay.logits.cpu().pin_memory()
    dy_h = bw.dy.cpu().pin_memory()
    outs_h = [(torch.empty(bw.dx.shape, dtype=bw.dx.dtype, pin_memory=True),
               torch.empty(bw.dl.shape, dtype=bw.dl.dtype, pin_memory=True))
              for _ in range(2)]
    sets = [tuple(torch.empty_like(t) for t in
                  (lay.x, lay.logits, bw.dy, bw.dx, bw.dl)) for _ in range(2)]
    bw.dw_api = bw.dw
    comp = torch.cuda.current_stream()
    up = torch.cuda.Stream(device=device)     # host -> device
    down = torch.cuda.Stream(device=device)   # device -> host
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
    free = [ev(), ev()]
    for e in free:
        e.record(down)

    def steps(n):
        for i in range(n):
            b = i % 2
            x_d, L_d, dy_d, dx_d, dl_d = sets[b]
            with torch.cuda.stream(up):
                up.wait_event(free[b])       # set b's last outputs are out
                x_d.copy_(x_h, non_blocking=True)
                L_d.copy_(L_h, non_blocking=True)
                dy_d.copy_(dy_h, non_blocking=True)
                h2d = ev()
                h2d.record(up)
            comp.wait_event(h2d)
            bw.api(x_d, L_d, dy_d, dx_d, dl_d)
            done = ev()
            done.record(comp)
            with torch.cuda.stream(down):
                down.wait_event(done)
                outs_h[b][0].copy_(dx_d, non_blocking=True)
                outs_h[b][1].copy_(dl_d, non_blocking=True)
                free[b].record(down)

    steps(max(1, args.warmup))
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record(comp)
    up.wait_event(a)
    down.wait_event(a)
    steps(args.steps)
    comp.wait_stream(up)
    comp.wait_stream(down)
    z.record(comp)
    z.synchronize()
    mean = max_over_ranks(a.elapsed_time(z) / args.steps, device)
    if not torch.equal(outs_h[(args.steps - 1) % 2][0], bw.dx.cpu()):
        raise SystemExit("pipelined end-to-end backward output differs")
    h2d = sum(t.numel() * t.element_size() for t in (x_h, L_h, dy_h))
    d2h = sum(t.numel() * t.element_size() for t in outs_h[0])
    return {"value": round(whole_job_tokens_per_s(world, lay.wl.T, mean), 1),
            "unit": UNIT, "ms_per_step": round(mean, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "api": "moe_layer_backward (C ABI), pinned host buffers, copies "
                   "on two copy streams overlapping neighbouring steps"}


def reference_arm(args, wl, device):
    """The float64 oracle as the reference implementation, on host cores."""
    x = make_x(wl, device)
    wr = make_router_weight(wl, device)
    off = make_logit_offset(wl)
    W = make_weights(wl, device)
    n = REF_SAMPLE.get(wl.name, 8)
    for i in range(args.warmup):
        oracle_sample_run(wl, x, wr, off, W, n,
                          t0=(i * n) % max(1, wl.T - n))
    secs = []
    toks = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        s, m = oracle_sample_run(wl, x, wr, off, W, n,
                                 t0=((args.warmup + i) * n) % max(1, wl.T - n))
        secs.append(s)
        toks += m
    wall = time.perf_counter() - t0
    value = toks / sum(secs)
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4),
           "unit": UNIT, "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * sum(secs) / len(secs), 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f64", "data": "synthetic",
           "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "E": wl.E,
                      "k": wl.k, "F": wl.F, "S": wl.S,
                      "ragged_buffer_factor": wl.factor,
                      "sample_tokens_per_step": n},
           "cpu_baseline": {"value": round(value, 4), "unit": UNIT,
                            "cores": _CORES, "kind": "oracle",
                            "sample": f"{n} tokens of the {wl.name} batch per "
                                      f"step as a layer of their own"},
           "e2e": {"value": round(value, 4), "unit": UNIT,
                   "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "wall_s": round(wall, 2)}
    print(json.dumps(out))


if __name__ == "__main__":
    main()
