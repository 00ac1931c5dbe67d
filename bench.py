"""Benchmark of the SP boundary hot path on GB300.

One step = one pass of the whole boundary over one batch: the fused forward
(g* reduce-scatter + bias + dropout + residual + LayerNorm + g all-gather)
and the backward (norm / dropout backward, all-gather of the partials'
gradient, parameter gradients), on the 70B-shape workload (t = 8 emulated
ranks, b = 1, s = 16384, h = 8192, bf16).

Prints one JSON line (rank 0).  ``value`` times K whole steps (replayed as
CUDA graphs of up to 8 steps) between two CUDA events on the launching
stream, inputs resident in HBM (larger than L2); the forward / backward split
comes from a second loop with one graph per call, and the roofline of the
dominant kernel (the forward) from its per-launch duration in a third loop
of graphs of 8 back-to-back calls.  ``e2e`` repeats the step through the
public API with pinned host buffers copied in and out.  ``--impl reference``
times the CPU oracle instead, on bounded samples of the same workload.

Launch: ``python bench.py [--gpus N] [--steps K] [--warmup W]``; for N > 1
under torch.distributed.run, each rank processes its own batch (weak
scaling, no collective on the data path).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from datetime import datetime

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from sp_boundary_norm_gb300 import workloads as wl  # noqa: E402

METRIC = "SP-boundary fwd+bwd tokens/s and achieved HBM GB/s (% of GB300 peak) at h=8192,t=8"
UNIT = "tokens/s"
FWD_SOURCES = ("sp_boundary_norm_gb300/csrc/fwd.cu", "sp_boundary_norm_gb300/csrc/fwd_kernel.cuh",
               "sp_boundary_norm_gb300/csrc/sp_device.cuh", "sp_boundary_norm_gb300/csrc/sp_internal.h")
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "rs_norm_fwd_kernel_70b.md")
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e nominal bandwidth (context; the roofline uses the measured copy)
L2_BYTES = 129 * 1000 * 1000   # GB300 L2 capacity, about 129 MB


# ------------------------------------------------------------ byte counts --

def fwd_bytes_per_token(t, h, n_gather, norm="layernorm"):
    """Algorithmic bytes: t partials + residual read; Z, mask, O copies, stats written."""
    stats = 8 if norm == "layernorm" else 4
    return 2 * t * h + 2 * h + 2 * h + h + 2 * h * n_gather + stats


def unfused_fwd_bytes_per_token(t, h, n_gather, norm="layernorm"):
    """The unfused forward: reduce-scatter (t partials in, bf16 shard out), the
    norm on the shard (shard, residual in; Z, mask, O, stats out), all-gather
    (O in, n_gather copies out)."""
    stats = 8 if norm == "layernorm" else 4
    return (2 * t * h + 2 * h) + (2 * h + 2 * h + 2 * h + h + 2 * h + stats) \
        + (2 * h + 2 * h * n_gather)


def bwd_g_bytes_per_token(t, h, n_gather, norm="layernorm", fused=True):
    """Backward entered through g: the t partial gradients of the gathered
    input are read (fused: summed in the kernel; unfused: a reduce-scatter
    writes the bf16 dY shard, which the norm backward reads again)."""
    shard = bwd_bytes_per_token(h, n_gather, norm) - 2 * h   # without reading dY
    rs = 2 * t * h if fused else 2 * t * h + 2 * h + 2 * h
    return rs + shard


def bwd_bytes_per_token(h, n_gather, norm="layernorm", skip=False):
    """Algorithmic bytes: dY, Z, mask, stats (+skip) read; dResidual, dYpre copies written."""
    stats = 8 if norm == "layernorm" else 4
    return 2 * h + 2 * h + h + stats + (2 * h if skip else 0) + 2 * h + 2 * h * n_gather


def step_bytes_per_token(w, n_gather, pipeline="fused", mask="stored", bwd_entry="shard"):
    """(forward, backward) algorithmic bytes per token of one bench step.  The
    mask moves h bytes per token as bytes, h / 8 as bits ("bits") and none in
    the mask-free step ("regen"), in each direction."""
    fused = pipeline == "fused"
    mask_less = {"stored": 0, "regen": w.h, "bits": w.h - w.h // 8}[mask]
    fwd = (fwd_bytes_per_token(w.t, w.h, n_gather, w.norm) if fused else
           unfused_fwd_bytes_per_token(w.t, w.h, n_gather, w.norm)) - mask_less
    if bwd_entry == "g":
        bwd = bwd_g_bytes_per_token(w.t, w.h, n_gather, w.norm, fused) - mask_less
    else:
        bwd = bwd_bytes_per_token(w.h, n_gather, w.norm) - mask_less
    return fwd, bwd


def launches_per_step(fused, n_gather, bwd_entry):
    """Kernels of this library one step launches.  Forward: the fused kernel,
    or reduce-scatter + shard norm (+ all-gather).  Backward: the norm
    backward (fused with the reduce-scatter when entered through g) and the
    parameter-gradient reduce; entered through g unfused, a separate
    reduce-scatter first."""
    fwd = 1 if fused else 2 + (1 if n_gather else 0)
    bwd = 2 + (1 if (bwd_entry == "g" and not fused) else 0)
    return fwd + bwd


# ---------------------------------------------------------- distributed --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world, device=None):
    if world > 1:
        if device is not None and device.type == "cuda":
            torch.distributed.barrier(device_ids=[device.index])
        else:
            torch.distributed.barrier()


def max_over_ranks(value, world, device):
    """The maximum of a float over all ranks (the slowest rank sets the time)."""
    if world == 1:
        return value
    x = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(x, op=torch.distributed.ReduceOp.MAX)
    return float(x.item())


# --------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.lines = []
        ident = None
        try:
            ident = str(torch.cuda.get_device_properties(device).uuid)
            if not ident.startswith("GPU-"):
                ident = "GPU-" + ident
        except Exception:
            ident = None
        self.ident = ident

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.ident:
            cmd += ["-i", self.ident]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0, t1):
        samples = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, smax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            samples.append((ts, sm, smax, parts[5:9]))
        inside = [s for s in samples if t0 - 0.06 <= s[0] <= t1 + 0.06] or samples
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for s in inside for i, v in enumerate(s[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside)}


def clocks_rejected(c):
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if any(r in bad for r in c.get("reasons", [])):
        return True
    if c.get("sm_mhz") and c.get("sm_max_mhz") and not c["reasons"]:
        return c["sm_mhz"] < 0.6 * c["sm_max_mhz"]
    return False


# ----------------------------------------------------------- our arm ------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def fwd_source_sha():
    h = hashlib.sha256()
    for rel in FWD_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, if it is current."""
    try:
        text = open(TRAFFIC_PROFILE).read()
    except OSError:
        return None
    vals = {}
    for ln in text.splitlines():
        if "=" in ln and ln.strip().startswith(("traffic_per_launch_bytes", "source_sha")):
            k, v = ln.split("=", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha") != fwd_source_sha():
        return None
    try:
        return int(vals["traffic_per_launch_bytes"])
    except (KeyError, ValueError):
        return None


def profiled_workload(args):
    """The recorded traffic belongs to the default bench line only (70B shape,
    LayerNorm, p = 0.1, one gathered copy, the byte mask, no size overrides)."""
    return (args.workload == "70b" and not args.s and not args.h and args.p is None
            and args.norm in (None, "layernorm") and args.n_gather == 1
            and args.mask == "stored")


class Step:
    """Device buffers and the fwd + bwd calls of one step.

    pipeline "fused": one forward kernel; "unfused": reduce-scatter, norm on
    the shards, all-gather as three calls (the ablation of the fusion).
    """

    def __init__(self, w, device, n_gather=1, pipeline="fused", mask="stored", bwd_entry="shard"):
        self.pipeline = pipeline
        self.mask_mode = mask
        self.bwd_entry = bwd_entry
        from sp_boundary_norm_gb300 import binding as sp
        self.sp, self.w, self.dev = sp, w, device
        self.inp = wl.forward_inputs(w, device)
        self.dy = wl.backward_inputs(w, device)["dy"]
        sizes = w.shard_sizes()
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)
        self.z = [e((w.b, n, w.h), torch.bfloat16) for n in sizes]
        # mask-free step: the forward stores no mask, the backward draws it
        # again; "bits": the mask stored one bit per element
        self.mask = (None if mask == "regen" else
                     [e((w.b, n, w.h // 8 if mask == "bits" else w.h), torch.uint8)
                      for n in sizes])
        self.mean = [e((w.b, n), torch.float32) for n in sizes]
        self.rstd = [e((w.b, n), torch.float32) for n in sizes]
        self.gathered = [e((w.b, w.s, w.h), torch.bfloat16) for _ in range(n_gather)]
        self.dres = [e((w.b, n, w.h), torch.bfloat16) for n in sizes]
        self.dgat = [e((w.b, w.s, w.h), torch.bfloat16) for _ in range(n_gather)]
        self.dgamma, self.dbeta, self.dbias = (e((w.h,), torch.float32) for _ in range(3))
        self.ws = e((sp.sp_norm_bwd_workspace_bytes(w.b, w.s, w.h, w.t),), torch.uint8)
        self.cu = (torch.from_numpy(wl.cu_seqlens(w.seqlens)).to(device) if w.ragged else None)
        if pipeline == "unfused":
            self.y = [e((w.b, n, w.h), torch.bfloat16) for n in sizes]
            self.o = [e((w.b, n, w.h), torch.bfloat16) for n in sizes]
        if bwd_entry == "g":
            # each rank's partial gradient of the gathered (b, s, h) input
            gen = wl.make_generator(w.draw_seed + 2000, device)
            self.dy_parts = [(torch.randn((w.b, w.s, w.h), generator=gen, device=device)
                              * 0.35).to(torch.bfloat16) for _ in range(w.t)]

    def fwd(self):
        w, i = self.w, self.inp
        if self.pipeline == "unfused":
            self.sp.sp_reduce_scatter_seq(i["partials"], self.y, cu_seqlens=self.cu)
            self.sp.sp_shard_norm_fwd(self.y, i["residual"], i["bias"], i["gamma"], i["beta"],
                                      s=w.s, eps=w.eps, p=w.p, seed=w.seed, offset=w.offset,
                                      norm=w.norm, cu_seqlens=self.cu, z_out=self.z,
                                      mask_out=self.mask, mean_out=self.mean,
                                      rstd_out=self.rstd, o_shards=self.o)
            if self.gathered:
                self.sp.sp_allgather_seq(self.o, self.gathered, s=w.s, cu_seqlens=self.cu)
            return
        if self.mask_mode == "bits":
            self.sp.sp_rs_norm_fwd_bitmask(
                i["partials"], i["residual"], i["bias"], i["gamma"], i["beta"], eps=w.eps,
                p=w.p, seed=w.seed, offset=w.offset, norm=w.norm, cu_seqlens=self.cu,
                z_out=self.z, mask_bits_out=self.mask, mean_out=self.mean, rstd_out=self.rstd,
                gathered=self.gathered)
            return
        self.sp.sp_rs_norm_fwd(i["partials"], i["residual"], i["bias"], i["gamma"], i["beta"],
                               eps=w.eps, p=w.p, seed=w.seed, offset=w.offset, norm=w.norm,
                               cu_seqlens=self.cu, z_out=self.z, mask_out=self.mask,
                               mean_out=self.mean, rstd_out=self.rstd, gathered=self.gathered)

    def bwd(self):
        w = self.w
        if self.bwd_entry == "g":
            if self.pipeline == "unfused":
                self.sp.sp_reduce_scatter_seq(self.dy_parts, self.dy, cu_seqlens=self.cu)
            else:
                rs_bwd = (self.sp.sp_rs_norm_bwd_bitmask if self.mask_mode == "bits"
                          else self.sp.sp_rs_norm_bwd)
                rs_bwd(self.dy_parts, self.z, self.mask, self.mean, self.rstd, self.inp["gamma"],
                       None, p=w.p, norm=w.norm, cu_seqlens=self.cu, dresidual=self.dres,
                       dgathered=self.dgat, dgamma=self.dgamma, dbeta=self.dbeta,
                       dbias=self.dbias, workspace=self.ws)
                return
        if self.mask_mode == "regen":
            self.sp.sp_norm_bwd_philox(
                self.dy, self.z, self.mean, self.rstd, self.inp["gamma"], None, s=w.s, p=w.p,
                seed=w.seed, offset=w.offset, norm=w.norm, cu_seqlens=self.cu,
                dresidual=self.dres, dgathered=self.dgat, dgamma=self.dgamma, dbeta=self.dbeta,
                dbias=self.dbias, workspace=self.ws)
            return
        bwd = self.sp.sp_norm_bwd_bitmask if self.mask_mode == "bits" else self.sp.sp_norm_bwd
        bwd(self.dy, self.z, self.mask, self.mean, self.rstd, self.inp["gamma"], None, s=w.s,
            p=w.p, norm=w.norm, cu_seqlens=self.cu, dresidual=self.dres, dgathered=self.dgat,
            dgamma=self.dgamma, dbeta=self.dbeta, dbias=self.dbias, workspace=self.ws)


    def inputs(self):
        """The step's inputs, as a caller would copy them in."""
        return self.inp["partials"] + self.inp["residual"] + self.dy

    def outputs(self):
        """The step's results, as a caller would copy them out."""
        return self.gathered + self.dres + self.dgat + [self.dgamma, self.dbeta, self.dbias]


class BucketedStep:
    """One step of a packed batch bucketed by length: the boundary's forward
    and backward on every bucket (each bucket a packed batch of its own with
    its cu_seqlens), covering the same sequences as the whole batch.  The
    buckets share no buffer, so each runs on a stream of its own, forked from
    and joined back to the caller's stream (one bucket's blocks start while
    another's last blocks finish); serial=True runs them in turn instead."""

    def __init__(self, w, device, buckets, serial=False, **kw):
        self.buckets = buckets
        self.device = device
        self.steps = [Step(w.with_(name=f"{w.name}-bucket{i}", s=b.tokens,
                                   seqlens=tuple(b.lengths), draw_seed=w.draw_seed + 100 + i),
                           device, **kw) for i, b in enumerate(buckets)]
        self.sp = self.steps[0].sp
        self.streams = (None if serial or device.type != "cuda" else
                        [torch.cuda.Stream(device) for _ in buckets])

    def _each(self, call):
        if self.streams is None:
            for st in self.steps:
                call(st)
            return
        main = torch.cuda.current_stream(self.device)
        fork = torch.cuda.Event()
        fork.record(main)
        joins = []
        for st, stream in zip(self.steps, self.streams):
            stream.wait_event(fork)
            with torch.cuda.stream(stream):
                call(st)
                done = torch.cuda.Event()
                done.record(stream)
            joins.append(done)
        for done in joins:
            main.wait_event(done)

    def fwd(self):
        self._each(lambda st: st.fwd())

    def bwd(self):
        self._each(lambda st: st.bwd())

    def inputs(self):
        return [x for st in self.steps for x in st.inputs()]

    def outputs(self):
        return [x for st in self.steps for x in st.outputs()]


def capture(fn, device):
    """One call of the step's forward or backward as a CUDA graph.

    The boundary's entry points validate arguments on the host and then only
    enqueue kernels, so a captured call replays exactly those kernels with the
    same buffers; replaying removes the per-call host cost (argument checks,
    ctypes marshalling), which otherwise exceeds the kernel time of the
    smaller workloads."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize(device)
    return g.replay


B2B_CALLS = 8    # calls per graph in the back-to-back loops
GRAPH_STEPS = 8  # whole steps per graph in the headline loop


def time_device(step, steps, warmup, world, device, launch="graph"):
    """K steps between two events (the headline); then K more with events
    between each step's forward and backward (the per-call split); then K
    forward calls and K backward calls, B2B_CALLS back to back per graph with
    one event pair around each run of graphs (the per-launch duration, without
    the gap an event pair leaves around every graph launch).  With `launch`
    "graph" the headline loop replays CUDA graphs of GRAPH_STEPS whole steps
    (each step its forward and backward calls; the last graph takes the
    remainder, so exactly K steps run), as a training iteration captured in
    one graph would run them, and the split loop replays one graph per
    call."""
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        step.fwd()
        step.bwd()
    torch.cuda.synchronize(device)
    fwd, bwd = step.fwd, step.bwd
    one_step = lambda: (step.fwd(), step.bwd())
    steps_of = lambda n: (lambda: [one_step() for _ in range(n)])
    per_graph = max(1, min(GRAPH_STEPS, steps))
    headline = [one_step] * steps
    fwd_run = lambda: [step.fwd() for _ in range(B2B_CALLS)]
    bwd_run = lambda: [step.bwd() for _ in range(B2B_CALLS)]
    if launch == "graph":
        fwd, bwd = capture(step.fwd, device), capture(step.bwd, device)
        full = capture(steps_of(per_graph), device)
        headline = [full] * (steps // per_graph)
        if steps % per_graph:
            headline.append(capture(steps_of(steps % per_graph), device))
        fwd_run, bwd_run = capture(fwd_run, device), capture(bwd_run, device)
        for _ in range(warmup):
            full()
            fwd()
            bwd()
        fwd_run()
        bwd_run()
        torch.cuda.synchronize(device)
    runs = max(1, steps // B2B_CALLS)
    b2b = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    start, end = (torch.cuda.Event(enable_timing=True) for _ in range(2))
    sampler = ClockSampler(device)
    sampler.start()
    barrier(world, device)
    torch.cuda.synchronize(device)
    t0 = time.time()
    start.record(stream)
    for g in headline:
        g()
    end.record(stream)
    torch.cuda.synchronize(device)
    for k in range(steps):
        ev[k][0].record(stream)
        fwd()
        ev[k][1].record(stream)
        bwd()
        ev[k][2].record(stream)
    torch.cuda.synchronize(device)
    b2b[0].record(stream)
    for _ in range(runs):
        fwd_run()
    b2b[1].record(stream)
    for _ in range(runs):
        bwd_run()
    b2b[2].record(stream)
    torch.cuda.synchronize(device)
    t1 = time.time()
    barrier(world, device)
    sampler.stop()
    step.sp.check_device_status(device)
    total_ms = start.elapsed_time(end)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    n = runs * B2B_CALLS
    back_to_back = {"calls": n, "fwd_ms": b2b[0].elapsed_time(b2b[1]) / n,
                    "bwd_ms": b2b[1].elapsed_time(b2b[2]) / n}
    return total_ms, fwd_ms, bwd_ms, back_to_back, sampler.summary(t0, t1)


def time_each_step(step_list, steps, device):
    """ms per forward + backward of each step, alone: one graph of the pair,
    replayed `steps` times between two events."""
    stream = torch.cuda.current_stream(device)
    out = []
    for st in step_list:
        g = capture(lambda: (st.fwd(), st.bwd()), device)
        for _ in range(3):
            g()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        a.record(stream)
        for _ in range(steps):
            g()
        b.record(stream)
        torch.cuda.synchronize(device)
        out.append(a.elapsed_time(b) / steps)
    return out


def time_e2e(step_a, step_b, steps, device):
    """The step through the public API with host buffers, end to end (wall
    clock, synchronised at both ends): every step copies its inputs in from
    pinned host memory and its results (O, dResidual, dYpre, dgamma, dbeta,
    dbias) out to pinned host memory.  Consecutive steps are pipelined the
    way a streaming caller would run them: two device buffer sets, the copy-in
    of step i+1 and the copy-out of step i on their own streams while step i
    computes."""
    sets = [step_a, step_b]
    ins = lambda st: st.inputs()
    outs = lambda st: st.outputs()
    host_in = [x.cpu().pin_memory() for x in ins(step_a)]
    host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs(step_a)]
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    s_in, s_cmp, s_out = (torch.cuda.Stream(device) for _ in range(3))

    def run(n):
        done_cmp, done_out = {}, {}
        for i in range(n):
            st = sets[i % 2]
            ev_in = torch.cuda.Event()
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(done_cmp[i - 2])      # set i % 2 is free again
                for d, h in zip(ins(st), host_in):
                    d.copy_(h, non_blocking=True)
                ev_in.record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in)
                if i >= 2:
                    s_cmp.wait_event(done_out[i - 2])     # its outputs were read out
                st.fwd()
                st.bwd()
                done_cmp[i] = torch.cuda.Event()
                done_cmp[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_cmp[i])
                for h, d in zip(host_out, outs(st)):
                    h.copy_(d, non_blocking=True)
                done_out[i] = torch.cuda.Event()
                done_out[i].record(s_out)
        torch.cuda.synchronize(device)

    run(2)
    t0 = time.perf_counter()
    run(steps)
    return (time.perf_counter() - t0) * 1e3, h2d, d2h


def _oracle_worker(conn, w):
    """One process of OraclePool: builds its sample on request (untimed), runs
    the oracle's forward + backward on it on request."""
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    torch.set_num_threads(1)
    from oracle import boundary as ob
    f = lambda x: x.float().numpy()
    conn.send("ready")
    job = None
    while True:
        msg = conn.recv()
        if msg is None:
            break
        if msg[0] == "prep":
            _, n_tok, seed = msg
            sample = w.with_(s=n_tok, name=w.name + "-sample")
            inp = wl.forward_inputs(sample, "cpu", seed=seed)
            dy = [f(x) for x in wl.backward_inputs(sample, "cpu", seed=seed)["dy"]]
            job = (([f(x) for x in inp["partials"]], [f(x) for x in inp["residual"]],
                    f(inp["bias"]), f(inp["gamma"]), f(inp["beta"])), dy)
            conn.send("ok")
        else:
            a, dy = job
            fw = ob.rs_norm_fwd(*a, eps=w.eps, p=w.p, seed=w.seed, offset=w.offset, norm=w.norm,
                                n_gather=1)
            ob.norm_bwd(dy, fw["z"], fw["mask"], fw["mean"], fw["rstd"], a[3], None, p=w.p,
                        norm=w.norm, n_gather=1)
            conn.send("done")
    conn.close()


class OraclePool:
    """The oracle (as it stands, numpy) in `procs` spawned processes, one per
    host core: every step each process builds its own sample of `n_tok`
    tokens (untimed), then all run the forward + backward at once under one
    wall clock.  Spawned, not forked, so it is safe after CUDA is up."""

    def __init__(self, w, procs):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        for _ in range(procs):
            here, there = ctx.Pipe()
            proc = ctx.Process(target=_oracle_worker, args=(there, w), daemon=True)
            proc.start()
            self.conns.append(here)
            self.procs.append(proc)
        for c in self.conns:
            c.recv()

    def step(self, n_tok, seed):
        for i, c in enumerate(self.conns):
            c.send(("prep", n_tok, seed * 1000 + i))
        for c in self.conns:
            c.recv()
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(("run",))
        for c in self.conns:
            c.recv()
        return time.perf_counter() - t0

    def close(self):
        for c in self.conns:
            c.send(None)
        for proc in self.procs:
            proc.join(timeout=30)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, seconds=10.0, n_tokens=64):
    """The CPU oracle (as it stands) on bounded samples of the workload: about
    `seconds` of work on every host core (one oracle process per core), and
    the same on one core for reference."""
    n_tok = max(w.t, n_tokens // w.t * w.t)
    out = {}
    for procs in (1, host_cores()):
        pool = OraclePool(w, procs)
        done, elapsed, reps = 0, 0.0, 0
        try:
            while elapsed < seconds / 2 and reps < 1000:
                elapsed += pool.step(n_tok, 100 + reps)
                done += n_tok * procs
                reps += 1
        finally:
            pool.close()
        out[procs] = (done / elapsed, reps, elapsed)
    cores = max(out)
    value, reps, elapsed = out[cores]
    return {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "nproc": os.cpu_count(), "single_thread_value": round(out[1][0], 2),
            "sample": f"{reps} steps of {cores} oracle processes (one per host core) x "
                      f"{n_tok} tokens of the {w.name} shape (t={w.t}, h={w.h}), fwd+bwd, "
                      f"{elapsed:.1f} s wall; one process alone: {out[1][0]:.1f} tokens/s"}


def run_ours(args):
    world, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    from sp_boundary_norm_gb300 import _build
    if rank == 0 or world == 1:
        _build.build_library()
    barrier(world, device)
    w = wl.WORKLOADS[args.workload]
    if args.s:
        w = w.with_(s=args.s, name=f"{w.name}-s{args.s}")
    if args.h:
        if w.ragged or args.h % 8:
            raise SystemExit("--h: dense workloads only, a multiple of 8")
        w = w.with_(h=args.h, name=f"{w.name}-h{args.h}")
    if args.p is not None:
        w = w.with_(p=args.p, name=f"{w.name}-p{args.p}")
    if args.norm is not None:
        w = w.with_(norm=args.norm, eps=1e-5 if args.norm == "layernorm" else 1e-6,
                    name=f"{w.name}-{args.norm}")
    if args.mask == "regen" and args.bwd_entry == "g":
        raise SystemExit("--mask regen: the backward through g reads a stored mask")
    if args.mask == "bits" and args.pipeline != "fused":
        raise SystemExit("--mask bits: the fused forward only")
    kw = dict(n_gather=args.n_gather, pipeline=args.pipeline, mask=args.mask,
              bwd_entry=args.bwd_entry)
    buckets = None
    if args.bucket:
        if not w.ragged:
            raise SystemExit("--bucket: packed workloads only (--workload ragged)")
        from sp_boundary_norm_gb300 import bucketing as bk
        buckets = bk.bucket_by_tokens(w.seqlens, max_cv=args.max_cv)
        make_step = lambda: BucketedStep(w, device, buckets, **kw)
    else:
        make_step = lambda: Step(w, device, **kw)
    step = make_step()
    total_ms, fwd_ms, bwd_ms, b2b, clocks = time_device(step, args.steps, args.warmup, world,
                                                        device, args.launch)
    rejected = False
    if clocks_rejected(clocks):
        rejected = True
        total_ms, fwd_ms, bwd_ms, b2b, clocks = time_device(step, args.steps, args.warmup,
                                                            world, device, args.launch)
    total_ms = max_over_ranks(total_ms, world, device)
    tokens = w.tokens * args.steps * world
    value = tokens / (total_ms / 1e3)
    fused = args.pipeline == "fused"
    fpt, bpt = step_bytes_per_token(w, args.n_gather, args.pipeline, args.mask, args.bwd_entry)
    fb, bb = fpt * w.tokens, bpt * w.tokens
    fwd_avg = statistics.mean(fwd_ms)
    bwd_avg = statistics.mean(bwd_ms)
    peak, peak_kind = measured_peak()
    step_ms = total_ms / args.steps
    achieved = fb / (b2b["fwd_ms"] / 1e3) / 1e9
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    step_b = make_step()
    e2e_ms, h2d, d2h = time_e2e(step, step_b, e2e_steps, device)
    del step_b
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    bucketing = None
    if buckets is not None:
        # each bucket alone, then the same sequences as one packed batch
        per = time_each_step(step.steps, args.steps, device)
        whole = Step(w, device, **kw)
        w_total, _, _, w_b2b, _ = time_device(whole, args.steps, args.warmup, world, device,
                                              args.launch)
        del whole
        bucketing = {
            "max_cv": args.max_cv,
            "buckets": [{"lengths": list(b.lengths), "length_cv": round(b.length_cv, 4),
                         "tokens": b.tokens, "ms_per_step": round(ms, 4),
                         "tokens_per_s": round(b.tokens / (ms / 1e3), 1)}
                        for b, ms in zip(buckets, per)],
            "unbucketed": {"length_cv": round(bk.length_cv(w.seqlens), 4),
                           "ms_per_step": round(w_total / args.steps, 4),
                           "tokens_per_s": round(w.tokens * args.steps / (w_total / 1e3), 1),
                           "fwd_ms_back_to_back": round(w_b2b["fwd_ms"], 4),
                           "bwd_ms_back_to_back": round(w_b2b["bwd_ms"], 4)},
        }
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, seconds=args.cpu_seconds)
    if rank != 0:
        return
    norm_name = "LayerNorm" if w.norm == "layernorm" else "RMSNorm"
    partial_bytes = w.t * w.tokens * w.h * 2
    l2_note = (f"inputs larger than L2 ({partial_bytes / 1e9:.2f} GB of partials per step), "
               "no flush" if partial_bytes > L2_BYTES else
               f"inputs fit in L2 ({partial_bytes / 1e6:.1f} MB of partials): L2-resident "
               "timings, not an HBM measurement")
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "accumulate": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name}: {norm_name} boundary fwd+bwd, t={w.t} emulated ranks, "
                               f"b={w.b}, s={w.s}, h={w.h}, p={w.p}, n_gather={args.n_gather}"
                               + (f", {len(buckets)} length buckets (max_cv={args.max_cv}), "
                                  "one call pair per bucket, each bucket on a stream of its own"
                                  if buckets else ""),
                   "t": w.t, "b": w.b, "s": w.s, "h": w.h, "norm": w.norm, "p": w.p,
                   "n_gather": args.n_gather, "pipeline": args.pipeline,
                   "backward_mask": args.mask, "backward_entry": args.bwd_entry,
                   "mask_storage": {"stored": "1 byte per element",
                                    "bits": "1 bit per element",
                                    "regen": "none (the backward draws it again)"}[args.mask],
                   "launch": f"cuda graphs of {min(GRAPH_STEPS, args.steps)} steps (each step "
                             "its forward and backward calls); the fwd/bwd split from a second "
                             "loop with one graph per call"
                             if args.launch == "graph" else "eager API calls",
                   "l2": l2_note,
                   "parallelism": f"replicas x{world} (independent batches)"},
        "hbm_gbs": round((fb + bb) / (step_ms / 1e3) / 1e9, 1),
        "hbm_frac_of_peak": round((fb + bb) / (step_ms / 1e3) / 1e9 / peak, 4),
        "hbm_frac_of_nominal": round((fb + bb) / (step_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS, 4),
        "fwd": {"ms": round(fwd_avg, 4), "gbs": round(fb / (fwd_avg / 1e3) / 1e9, 1),
                "bytes": fb, "tokens_per_s": round(w.tokens / (fwd_avg / 1e3), 1),
                "ms_back_to_back": round(b2b["fwd_ms"], 4)},
        "bwd": {"ms": round(bwd_avg, 4), "gbs": round(bb / (bwd_avg / 1e3) / 1e9, 1),
                "bytes": bb, "tokens_per_s": round(w.tokens / (bwd_avg / 1e3), 1),
                "ms_back_to_back": round(b2b["bwd_ms"], 4),
                "gbs_back_to_back": round(bb / (b2b["bwd_ms"] / 1e3) / 1e9, 1)},
        "roofline": {"bound": "hbm",
                     "kernel": "rs_norm_fwd_kernel" if fused else
                               "unfused forward (reduce_scatter + shard norm + allgather)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "launch_ms": round(b2b["fwd_ms"], 4),
                     "timing": f"{b2b['calls']} forward calls, {B2B_CALLS} back to back per "
                               "graph replay, one event pair around all of them",
                     "traffic": (profiled_traffic() if fused and profiled_workload(args)
                                 else None),
                     "algorithmic_bytes": fb},
        "e2e": {"value": round(w.tokens * e2e_steps * world / (e2e_ms / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "timing": "wall clock; copy-in, compute, copy-out pipelined across steps"},
        "gpu_launches": launches_per_step(fused, args.n_gather, args.bwd_entry)
                        * (len(buckets) if buckets else 1) * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if bucketing is not None:
        line["bucketing"] = bucketing
    if rejected:
        line["clocks_remeasured"] = True
    print(json.dumps(line), flush=True)


# ------------------------------------------------------ reference arm ----

def run_reference(args):
    """The oracle timed on the host cores (one oracle process per core), on
    bounded samples per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = wl.WORKLOADS[args.workload]
    procs = host_cores()
    pool = OraclePool(w, procs)
    try:
        # calibrate the per-process sample so the run stays within about a minute
        per_tok = pool.step(w.t * 8, 1) / (w.t * 8)
        budget = 60.0 / max(1, args.steps + args.warmup)
        n_tok = int(max(w.t, min(w.t * 16, budget / per_tok)) // w.t * w.t)
        for i in range(args.warmup):
            pool.step(n_tok, 10 + i)
        elapsed = sum(pool.step(n_tok, 1000 + i) for i in range(args.steps))
    finally:
        pool.close()
    value = n_tok * procs * args.steps / elapsed
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name}: "
                               f"{'LayerNorm' if w.norm == 'layernorm' else 'RMSNorm'} boundary "
                               f"fwd+bwd, t={w.t}, b={w.b}, "
                               f"s={w.s}, h={w.h}, p={w.p}, n_gather=1 (sampled: {procs} x "
                               f"{n_tok} tokens per step)", "t": w.t, "s": w.s, "h": w.h},
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": procs, "kind": "oracle",
                         "nproc": os.cpu_count(),
                         "sample": f"{procs} oracle processes (one per host core) x {n_tok} "
                                   f"tokens per step of the {w.name} shape"},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="70b", choices=sorted(wl.WORKLOADS),
                    help="70b (default), bwd70b / bwd70b_rms (the backward configurations' "
                         "draws and norms), trace4k, ragged, tiny")
    ap.add_argument("--s", type=int, default=0,
                    help="override the sequence length (smaller cases for profiling)")
    ap.add_argument("--h", type=int, default=0,
                    help="override the hidden size (dense workloads; a multiple of 8)")
    ap.add_argument("--p", type=float, default=None, help="override the dropout probability")
    ap.add_argument("--norm", choices=["layernorm", "rmsnorm"], default=None,
                    help="override the norm")
    ap.add_argument("--n-gather", type=int, default=1)
    ap.add_argument("--launch", choices=["graph", "eager"], default="graph",
                    help="graph: replay the captured forward / backward calls")
    ap.add_argument("--bwd-entry", choices=["shard", "g"], default="shard",
                    help="g: the backward starts from each rank's partial gradient of the "
                         "gathered input (reduce-scatter fused, or separate if unfused)")
    ap.add_argument("--mask", choices=["stored", "regen", "bits"], default="stored",
                    help="regen: the mask-free step (the forward stores no mask, the "
                         "backward draws it again); bits: the mask stored one bit per "
                         "element")
    ap.add_argument("--pipeline", choices=["fused", "unfused"], default="fused",
                    help="unfused: reduce-scatter, shard norm and all-gather as three calls")
    ap.add_argument("--bucket", action="store_true",
                    help="packed workload: bucket its sequences by length (bucket_by_tokens) "
                         "and run the boundary once per bucket; the unbucketed batch is timed "
                         "beside it")
    ap.add_argument("--max-cv", type=float, default=0.15,
                    help="length-CV bound of a bucket (with --bucket)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
