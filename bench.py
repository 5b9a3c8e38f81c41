"""Benchmark of the hybrid Muon + AdamW optimizer step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One "step" is one full optimizer step of the workload (global grad norm and
clip, Muon momentum, five Newton-Schulz iterations and update, AdamW) with
all inputs resident in HBM. Default workload: full_vla, the largest
single-GPU configuration: the 2048-hidden, 24-layer action expert (168 Muon
matrices, 1.61 G elements) plus a 1.69 G-element AdamW backbone and a frozen
151936 x 2048 embedding, fp32 masters and moments, bf16 gradients, lr from
cosine_with_min_lr at step 1000 of 2000. Each step touches ~83 GB, far above
the 129 MB L2, so no flush is needed between steps. Other workloads:
--workload tiny | h1024 | h2048 | h2048_fp32grad | many_small.

Prints one JSON line (rank 0). value = optimizer steps/s for the whole job;
under torchrun each rank runs an independent replica ("replicas only"), so
value = N * K / (max over ranks of the timed region); --gpus must equal the
number of ranks. The timed region runs the steps as a user does (the
Newton-Schulz chain replayed from its CUDA graph); the per-kernel times come
from as many steps again with the library's per-launch CUDA events on.
Extra keys: per-kernel CUDA-event breakdown, the roofline of the dominant
kernel (the Newton-Schulz GEMM), the step roofline (the step's ideal time
from its flops and bytes against the measured step), the SM clocks seen
during the timed region, an end-to-end figure (gradients copied from pinned
host memory every step, the norm read back), and the fp64 oracle timed on a
bounded sample on the host cores (cpu_baseline).

--impl reference times the fp64 CPU oracle (the only reference that exists:
the source pages ship no code) on the same bounded sample: each timed step
runs the sample once; the line's value is the estimated rate of whole steps.
"""
from __future__ import annotations

import argparse
import gc
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "optimizer steps/s; NS5 TFLOP/s vs bf16 peak; AdamW HBM GB/s vs peak"
KINDS = ("grad_norm", "clip", "momentum", "ns_prep", "ns_gram", "ns_poly", "ns_update", "ns_apply", "ns_fused",
         "ns_narrow", "adamw")
NS_KINDS = ("ns_gram", "ns_poly", "ns_update", "ns_apply", "ns_fused")
STREAM_KINDS = ("grad_norm", "momentum", "adamw")


# DRAM bytes per ns_tc_kernel launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu
# capture of a 3-layer case of the full_vla expert (expert:2048:8192:3:fp32_mixed: the same matrix
# shapes and policy; the ns_tc_kernel summary in profiles/): the 15 launches of one step (5 X X^T,
# 5 A A, 4 B X, 1 last) averaged, 726.1 MB, and scaled to the 24-layer expert by the matrices
# processed (x 8: each launch reads its operands and writes its output once per matrix). It describes
# only the kernel sources it was measured on: any change to them makes it null until it is measured
# again.
NS_TRAFFIC = {"sources_sha256": "bae68366bf9cb926aa40cb7ba7bd0546a19d20cf6a1af3d5352a60e3588fc515",
              "bytes_per_launch": 5808463189, "workload": "full_vla"}
NS_SOURCES = ("ns_tc.cu", "ns_epilogue.cuh", "internal.h")


def ns_traffic_per_launch(workload: str):
    import hashlib

    h = hashlib.sha256()
    for f in NS_SOURCES:
        with open(os.path.join(ROOT, "muon_adamw_hybrid_grad_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != NS_TRAFFIC["sources_sha256"] or workload != NS_TRAFFIC["workload"]:
        return None
    return NS_TRAFFIC["bytes_per_launch"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def pinned_host_buffer(numel: int, dtype):
    """Host buffer of the end-to-end leg's per-step gradient copy: anonymous
    memory advised to transparent huge pages (where the kernel grants them)
    and page-locked with cudaHostRegister, which keeps the host->device copy's
    address translation to a few large pages; plain pinned memory
    (cudaHostAlloc) where that fails. Returns (tensor, kind, release)."""
    import mmap

    import torch

    esz = torch.tensor([], dtype=dtype).element_size()
    numel = max(int(numel), 1)
    size = numel * esz
    try:
        mm = mmap.mmap(-1, size, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        advised = False
        if hasattr(mmap, "MADV_HUGEPAGE"):
            try:
                mm.madvise(mmap.MADV_HUGEPAGE)
                advised = True
            except OSError:
                pass
        t = torch.frombuffer(mm, dtype=dtype, count=numel)
        t.zero_()  # every page present before it is locked
        cudart = torch.cuda.cudart()
        if int(cudart.cudaHostRegister(t.data_ptr(), size, 0)) != 0:
            raise RuntimeError("cudaHostRegister failed")
        kind = ("anonymous memory advised to huge pages" if advised else "anonymous memory") + ", cudaHostRegister"

        def release(t=t, mm=mm):
            cudart.cudaHostUnregister(t.data_ptr())

        return t, kind, release
    except Exception:
        return torch.zeros(numel, dtype=dtype).pin_memory(), "pinned (cudaHostAlloc)", lambda: None


def blas_threads() -> dict:
    """Threads of the BLAS behind the oracle's matrix products: from
    threadpoolctl where it is installed, else the thread-count environment
    variables, else the library's default of one thread per available core."""
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return {"blas_threads": int(max(n)), "blas_threads_source": "threadpoolctl"}
    except Exception:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(k)
        if v and v.isdigit():
            return {"blas_threads": int(v), "blas_threads_source": k}
    return {"blas_threads": host_cores(), "blas_threads_source": "default: one per available core"}


# ---------------------------------------------------------------------------
# multi-rank plumbing (replicas only)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist

    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when dist is None)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(steps: int, n_ranks: int, max_seconds: float) -> float:
    """Whole-job optimizer steps/s: every rank ran `steps` steps of its replica."""
    return n_ranks * steps / max_seconds


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (both the cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

# Workloads at most this large are timed as whole oracle steps; larger ones on a sample.
WHOLE_STEP_MAX_DENSE_FLOPS = 8e12
WHOLE_STEP_MAX_ADAMW_ELEMS = 16_000_000
SAMPLE_ADAMW_ELEMS = 1_000_000


def _dense_ns_flops(shape, steps: int = 5) -> float:
    s, l = min(shape), max(shape)
    return steps * (4.0 * s * s * l + 2.0 * s * s * s)


class OracleSample:
    """A bounded sample of workload ``w`` for the fp64 oracle, and its scaling
    to one full optimizer step.

    Workloads with at most 8 TFLOP of dense Newton-Schulz and 16 M AdamW
    elements per step (tiny, many_small, h1024) are run whole. Otherwise the
    sample is one Muon matrix of each distinct shape and the first AdamW
    tensors up to 1 M elements. Each part is run as its own oracle step
    (norm of its gradients, momentum, Newton-Schulz and update; AdamW) and a
    full step is estimated as
        sum over shapes (matrices of that shape) x (time of its sample matrix)
        + AdamW time x (AdamW elements / sampled AdamW elements).
    Inputs are generated once, outside the timed calls."""

    def __init__(self, w):
        import numpy as np

        import oracle
        import workloads

        self.np, self.oracle = np, oracle
        names = [t.name for t in w.tensors]
        groups = [oracle.route(n, len(t.shape), frozen=t.frozen) for n, t in zip(names, w.tensors)]
        muon = [i for i, g in enumerate(groups) if g == "muon"]
        adam = [i for i, g in enumerate(groups) if g == "adamw"]
        dense = sum(_dense_ns_flops(w.tensors[i].shape) for i in muon)
        adam_elems = sum(w.tensors[i].numel for i in adam)
        self.whole = dense <= WHOLE_STEP_MAX_DENSE_FLOPS and adam_elems <= WHOLE_STEP_MAX_ADAMW_ELEMS
        self.lr = w.lr
        if self.whole:
            idx = muon + adam
            self.parts = [(idx, 1.0)]
            self.desc = (f"fp64 numpy oracle, one whole step of {w.name} ({len(muon)} Muon matrices, "
                         f"{adam_elems} AdamW elements)")
        else:
            by_shape = {}
            for i in muon:
                by_shape.setdefault(tuple(w.tensors[i].shape), []).append(i)
            self.parts = [([ix[0]], float(len(ix))) for ix in by_shape.values()]
            ad, tot = [], 0
            for i in adam:
                if tot >= SAMPLE_ADAMW_ELEMS:
                    break
                ad.append(i)
                tot += w.tensors[i].numel
            if ad:
                self.parts.append((ad, adam_elems / tot))
            shapes = ", ".join(f"{k[0]}x{k[1]} (x{len(v)})" for k, v in by_shape.items())
            self.desc = (f"fp64 numpy oracle on a sample of {w.name}: one Muon matrix of each shape ({shapes}) "
                         f"and {len(ad)} AdamW tensors ({tot} of {adam_elems} elements), each part one oracle "
                         f"step; full step = sum of part times x (matrices of the shape, or AdamW elements / "
                         f"sampled)")
        self.inputs = []
        for idx, scale in self.parts:
            self.inputs.append(([names[i] for i in idx], [w.tensors[i].shape for i in idx],
                                [workloads.master_weight(w, i).astype(np.float64) for i in idx],
                                [workloads.gradient(w, i, 1) for i in idx], scale))

    def run(self):
        """One timed pass over the sample: (seconds that ran, estimated seconds of a full step)."""
        ran = full = 0.0
        for names, shapes, masters, grads, scale in self.inputs:
            params = [m.copy() for m in masters]
            orc = self.oracle.HybridOracle(names, shapes)
            t0 = time.perf_counter()
            orc.step(params, grads, self.lr)
            dt = time.perf_counter() - t0
            ran += dt
            full += dt * scale
        return ran, full


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def adamw_standalone(mx, torch, entries, w, lr, stream, peaks, steps: int = 10, warmup: int = 3) -> dict:
    """The AdamW kernel alone over every trainable tensor of the workload.

    The same tensors are registered with a second optimizer in AdamW-only
    mode (after the main measurements, whose results they no longer carry),
    and its AdamW launches are timed by the library's CUDA events on the
    launching stream. The step's other kernel (the gradient norm) is not part
    of this figure."""
    opt = mx.MuonAdamW(entries, precision=mx.MA_BF16_MIXED if w.policy == "bf16_mixed" else mx.MA_FP32_MIXED,
                       mode=mx.MA_MODE_ADAMW_ONLY, stream=stream)
    for _ in range(warmup):
        opt.step(lr)
    torch.cuda.synchronize()
    mx.muon_adamw_reset_profile(opt.handle)
    mx.muon_adamw_set_profiling(opt.handle, True)
    for _ in range(steps):
        opt.step(lr)
    torch.cuda.synchronize()
    e = opt.profile()["adamw"]
    info = opt.plan_info()
    del opt
    if e["launches"] == 0 or e["ms"] <= 0:
        return {"elements": 0}
    gbs = e["units"] / (e["ms"] / 1e3) / 1e9
    return {"elements": int(info["adamw_elems"]), "bytes": int(e["units"] / e["launches"]),
            "ms_per_launch": round(e["ms"] / e["launches"], 5), "gbs": round(gbs, 1),
            "frac_hbm": round(gbs / peaks["hbm_gbs"], 3), "launches": e["launches"],
            "how": "every trainable tensor of the workload through AdamW (a second optimizer in AdamW-only "
                   "mode), AdamW launches timed by CUDA events on the launching stream; bytes = p, m, v read "
                   "and written, the gradient read, the bf16 shadow written under bf16_mixed"}


def _batches(idx, size: int = 16):
    idx = list(idx)
    for k in range(0, len(idx), size):
        yield idx[k:k + size]


def step_roofline(info, step_s: float, peaks: dict, shadow: bool) -> dict:
    """The step's ideal time t* against the measured step: the Newton-Schulz
    flops at the bf16 peak plus the step's algorithmic HBM bytes at the HBM
    bandwidth, taken one after the other (serial) or fully overlapped (max).
    The bytes are the streaming kernels' (gradient norm, momentum, AdamW) plus
    the Muon update's read and write of p (and its bf16 shadow), which the
    last Newton-Schulz launch does in its epilogue."""
    f = info["ns_flops_per_step"]
    b = info["stream_bytes_per_step"] + info["muon_elems"] * (8 + (2 if shadow else 0))
    out = {"ns_flops_per_step": f, "hbm_bytes_per_step": b, "measured_ms": round(step_s * 1e3, 4),
           "hbm_gbs": peaks["hbm_gbs"], "how": "t* = F_NS / P_bf16 + B_stream / BW_HBM (serial), "
           "max(F_NS / P_bf16, B_stream / BW_HBM) (overlapped); frac = t* / measured step time"}
    for kind, key in (("burst", "bf16_tflops"), ("sustained", "bf16_tflops_sustained")):
        peak = peaks.get(key)
        if not peak:
            continue
        t_ns = f / (peak * 1e12)
        t_st = b / (peaks["hbm_gbs"] * 1e9)
        out[kind] = {"bf16_tflops": peak, "t_serial_ms": round((t_ns + t_st) * 1e3, 4),
                     "t_overlapped_ms": round(max(t_ns, t_st) * 1e3, 4),
                     "frac_serial": round((t_ns + t_st) / step_s, 3),
                     "frac_overlapped": round(max(t_ns, t_st) / step_s, 3)}
    return out


def run_ours(args):
    import numpy as np
    import torch

    import muon_adamw_hybrid_grad_gb300 as mx
    import workloads
    from muon_adamw_hybrid_grad_gb300 import build as _b

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    _b.build()
    mx.load_library()
    dev = torch.device("cuda", local)
    w = workloads.get_workload(args.workload)
    lr = w.lr
    if w.schedule is not None:
        step_, total_, warm_, min_rate = w.schedule
        lr = w.lr * mx.muon_adamw_cosine_with_min_lr(step_, total_, warm_, min_rate)
    gdt = torch.bfloat16 if w.grad_dtype == "bf16" else torch.float32
    # Gradients live in one flat device buffer (per-parameter views at 128-byte
    # aligned offsets, as a data-parallel gradient bucket would hold them), and
    # their host copy in one flat pinned buffer, so that the end-to-end leg
    # moves each step's inputs with one host->device copy. Inputs are made in
    # batches of tensors and uploaded as they are made (full-size workloads
    # never sit whole in host memory).
    align = 128 // torch.tensor([], dtype=gdt).element_size()
    offs, total = [], 0
    for t in w.tensors:
        offs.append(total)
        if not t.frozen:
            total += (t.numel + align - 1) // align * align
    gflat = torch.zeros(max(total, 1), dtype=gdt, device=dev)
    hflat, host_kind, host_release = pinned_host_buffer(total, gdt)
    n = len(w.tensors)
    P, G, S, entries = [None] * n, [None] * n, [None] * n, [None] * n
    for batch in _batches(range(n)):
        ms = workloads.master_weights(w, batch)
        gs = workloads.gradients(w, 1, batch)
        for i, m, g_np in zip(batch, ms, gs):
            t = w.tensors[i]
            P[i] = torch.from_numpy(m).to(dev)
            if not t.frozen:
                k = t.numel
                src = torch.from_numpy(g_np).reshape(-1).to(gdt)
                hflat[offs[i]:offs[i] + k].copy_(src)
                G[i] = gflat[offs[i]:offs[i] + k].view(t.shape)
                G[i].copy_(src.view(t.shape).to(dev))
            if w.policy == "bf16_mixed" and not t.frozen:
                S[i] = torch.empty(t.shape, dtype=torch.bfloat16, device=dev)
            entries[i] = (t.name, P[i], G[i], S[i], mx.MA_GROUP_FROZEN if t.frozen else None)
        del ms, gs
    stream = torch.cuda.current_stream()
    opt = mx.MuonAdamW(entries, precision=mx.MA_BF16_MIXED if w.policy == "bf16_mixed" else mx.MA_FP32_MIXED,
                       stream=stream)
    for _ in range(args.warmup):
        opt.step(lr)
    torch.cuda.synchronize()
    info = opt.plan_info()
    # ---- timed region (device time, CUDA events on the launching stream),
    # the steps as a user runs them (the Newton-Schulz chain replayed from
    # its CUDA graph, no per-launch events) ----
    clocks = ClockSampler(local)
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    # one event between consecutive steps: the region is first to last event,
    # and each step's own time gives the median and minimum
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    gc.disable()
    evs[0].record(stream)
    for k in range(args.steps):
        opt.step(lr)
        evs[k + 1].record(stream)
    torch.cuda.synchronize()
    gc.enable()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    ms = evs[0].elapsed_time(evs[-1])
    step_ms = [evs[k].elapsed_time(evs[k + 1]) for k in range(args.steps)]
    max_s = max_over_ranks(ms / 1e3, dist, dev)
    value = aggregate(args.steps, world, max_s)
    # ---- per-kernel times: as many steps again with the library's per-launch
    # CUDA events on (direct launches; the events sit between them) ----
    mx.muon_adamw_reset_profile(opt.handle)
    mx.muon_adamw_set_profiling(opt.handle, True)
    t_prof = time.perf_counter()
    for _ in range(args.steps):
        opt.step(lr)
    torch.cuda.synchronize()
    t_prof = time.perf_counter() - t_prof
    mx.muon_adamw_set_profiling(opt.handle, False)
    prof = opt.profile()

    # ---- end to end: grads from pinned host memory each step, norm read back ----
    # per step: the flat gradient buffer, plus the library's own copy of the
    # step's lr- and step-dependent scalars (112 bytes); back: the norm and
    # clip factor (16 bytes) and the device error flag (4 bytes)
    h2d = total * gflat.element_size() + 112
    d2h = 16 + 4
    # Each step's gradients are copied on a copy stream as soon as the previous
    # step has read its gradients (muon_adamw_record_grads_consumed), so the
    # copy overlaps that step's Newton-Schulz chain; every step's copy and the
    # read-back of every step's norm are inside the timed region.
    copy_stream = torch.cuda.Stream(device=dev)
    # Two untimed steps through the same path first (the copy stream, its
    # events and the pinned-copy bookkeeping are set up on first use); the
    # timed region still holds every timed step's copy, the first one included.
    for _ in range(2):
        with torch.cuda.stream(copy_stream):
            gflat.copy_(hflat, non_blocking=True)
        stream.wait_event(copy_stream.record_event())
        opt.step(lr)
        mx.muon_adamw_last_norm(opt.handle)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    # CUDA events on the copy stream around every copy (each copy's own
    # duration), and at each step's start on the optimizer's stream (when,
    # within the previous step, the next copy began)
    cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    gc.disable()  # no collector pause inside the host-timed loop
    t0 = time.perf_counter()
    with torch.cuda.stream(copy_stream):
        cev[0][0].record(copy_stream)
        gflat.copy_(hflat, non_blocking=True)  # step 1's gradients
        cev[0][1].record(copy_stream)
    host_t = [t0]
    for k in range(args.steps):
        stream.wait_event(copy_stream.record_event())
        sev[k].record(stream)
        opt.step(lr)
        if k + 1 < args.steps:
            copy_stream.wait_event(opt.record_grads_consumed())
            with torch.cuda.stream(copy_stream):
                cev[k + 1][0].record(copy_stream)
                gflat.copy_(hflat, non_blocking=True)  # step k+2's gradients
                cev[k + 1][1].record(copy_stream)
        mx.muon_adamw_last_norm(opt.handle)  # synchronises and reads this step's norm
        host_t.append(time.perf_counter())
    sev[args.steps].record(stream)
    e2e_s = time.perf_counter() - t0
    gc.enable()
    torch.cuda.synchronize()
    copy_ms = statistics.median(a.elapsed_time(b) for a, b in cev)
    # for steps 1..K-1: when the next step's copy started and ended, after the step's start
    copy_start = [sev[k].elapsed_time(cev[k + 1][0]) for k in range(args.steps - 1)]
    copy_end = [sev[k].elapsed_time(cev[k + 1][1]) for k in range(args.steps - 1)]
    step_dev = [sev[k].elapsed_time(sev[k + 1]) for k in range(args.steps)]
    step_host = [(host_t[k + 1] - host_t[k]) * 1e3 for k in range(args.steps)]
    e2e_s = max_over_ranks(e2e_s, dist, dev)

    peaks = load_peaks()
    # A kernel timed inside a long run of steps is held to the sustained bf16
    # peak, one timed in a short burst to the burst peak.
    sustained = t_prof >= 0.5 and peaks.get("bf16_tflops_sustained")
    tc_peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    tc_peak_kind = ("bf16 dense sustained" if sustained else "bf16 dense burst") + \
        f", {peaks['source']} (MEASURED_PEAKS.json)"
    ns_ms = sum(prof[k]["ms"] for k in NS_KINDS)
    ns_flops = sum(prof[k]["units"] for k in NS_KINDS)
    ns_launches = sum(prof[k]["launches"] for k in NS_KINDS)
    ns_tflops = ns_flops / (ns_ms / 1e3) / 1e12 if ns_ms > 0 else None
    kernels = {}
    for k in KINDS:
        e = prof[k]
        if e["launches"] == 0:
            continue
        d = {"launches": e["launches"], "ms_total": round(e["ms"], 4),
             "ms_per_launch": round(e["ms"] / e["launches"], 5)}
        if k in NS_KINDS:
            d["tflops"] = round(e["units"] / (e["ms"] / 1e3) / 1e12, 1)
            d["frac_bf16_peak"] = round(d["tflops"] / tc_peak, 3)
            d["frac_bf16_burst"] = round(d["tflops"] / peaks["bf16_tflops"], 3)
        elif k == "ns_narrow":
            # fp32 on the CUDA cores: "alu"-bound, against SMs x 128 fp32 lanes x 2 flops x the
            # maximum SM clock (nvidia-smi's clocks.max.sm, else the part's nominal 2070 MHz)
            d["tflops_fp32"] = round(e["units"] / (e["ms"] / 1e3) / 1e12, 2)
            mhz = clk.get("sm_max_mhz") or 2070.0
            peak = torch.cuda.get_device_properties(dev).multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12
            d["fp32_peak_tflops"] = round(peak, 1)
            d["frac_fp32_peak"] = round(d["tflops_fp32"] / peak, 3)
            d["bound"] = "alu"
        elif k in STREAM_KINDS:
            d["gbs"] = round(e["units"] / (e["ms"] / 1e3) / 1e9, 1)
            d["frac_hbm"] = round(d["gbs"] / peaks["hbm_gbs"], 3)
            d["frac_8tbs"] = round(d["gbs"] / 8000.0, 3)
            if k == "adamw":
                d["note"] = ("second stream, beside the momentum pass (the Newton-Schulz chain waits for it when "
                             "it moves more bytes than that pass): the event time includes sharing HBM and SMs "
                             "(adamw_standalone times it alone)")
            elif k == "momentum" and prof["adamw"]["launches"]:
                d["note"] = "runs beside AdamW (second stream): both share HBM bandwidth"
        kernels[k] = d
    launches = sum(prof[k]["launches"] for k in KINDS)
    adam_alone = adamw_standalone(mx, torch, entries, w, lr, stream, peaks)
    out = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_s * 1e3 / args.steps, 4),
        "step_ms_median": round(statistics.median(step_ms), 4) if step_ms else None,
        "step_ms_min": round(min(step_ms), 4) if step_ms else None,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) fp32 masters, N(0,1e-3)+rank-8 bf16 gradients)",
        "config": {
            "workload": f"{w.name}: {len(w.tensors)} tensors, {info['n_muon']} Muon matrices "
                        f"({info['muon_elems']} elements, {info['n_buckets']} shape buckets), "
                        f"{info['adamw_elems']} AdamW elements, {info['n_frozen']} frozen, {w.grad_dtype} grads, "
                        f"{w.policy}",
            "lr": lr,
            "l2": "no flush: each step touches "
                  f"{info['stream_bytes_per_step'] / 1e9:.2f} GB of state and gradients, far above the 129 MB L2",
            "parallelism": f"replicas x{world}",
        },
        "ns5_tflops": round(ns_tflops, 1) if ns_tflops else None,
        "ns5_frac_bf16_peak": round(ns_tflops / tc_peak, 3) if ns_tflops else None,
        "ns5_dense_equiv_tflops": round(info["ns_dense_flops_per_step"] * args.steps / (ns_ms / 1e3) / 1e12, 1)
        if ns_ms > 0 else None,
        "kernels": kernels,
        "roofline": {
            "kernel": ("ns_tc_kernel (tcgen05 Newton-Schulz GEMMs: X X^T, A A, B X; all launches)"
                       + (" and ns_small_kernel (small matrices: every iteration and the update in one launch)"
                          if prof["ns_fused"]["launches"] else "")),
            "bound": "tensor",
            "achieved": round(ns_tflops, 1) if ns_tflops else None,
            "peak": tc_peak,
            "peak_kind": tc_peak_kind,
            "unit": "TFLOP/s",
            "frac": round(ns_tflops / tc_peak, 3) if ns_tflops else None,
            "frac_of_burst": round(ns_tflops / peaks["bf16_tflops"], 3) if ns_tflops else None,
            "traffic": ns_traffic_per_launch(w.name),
            "traffic_unit": "DRAM bytes per launch (ncu, scaled from a smaller case of the same shapes; null "
                            "when stale)",
            "launches_timed": ns_launches,
            "algorithmic_flops_per_launch": round(ns_flops / max(1, ns_launches)),
        },
        "step_roofline": step_roofline(info, max_s / args.steps, peaks, w.policy == "bf16_mixed"),
        "clocks": clk,
        "e2e": {"value": round(args.steps * world / e2e_s, 3), "unit": "steps/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": d2h,
                "gradient_copy_ms_median": round(copy_ms, 3),
                "gradient_copy_gbs": round(total * gflat.element_size() / (copy_ms / 1e3) / 1e9, 1),
                "next_copy_start_ms_median": round(statistics.median(copy_start), 3) if copy_start else None,
                "next_copy_end_ms_median": round(statistics.median(copy_end), 3) if copy_end else None,
                "step_ms_median": round(statistics.median(step_dev), 3),
                "step_ms_max": round(max(step_dev), 3),
                "step_max_index": int(max(range(len(step_dev)), key=lambda k: step_dev[k])),
                "gradient_copy_ms_max": round(max(a.elapsed_time(b) for a, b in cev), 3),
                "host_step_ms_median": round(statistics.median(step_host), 3),
                "host_step_ms_max": round(max(step_host), 3),
                "host_buffer": host_kind,
                "how": "every step: every gradient copied host->device from pinned memory (one copy of the "
                       "flat gradient buffer, issued once the previous step has read its gradients and "
                       "overlapping that step's Newton-Schulz chain), muon_adamw_step, and the step's norm "
                       "read back (synchronising); two untimed steps through the same path first"},
        "gpu_launches": int(launches),
        "adamw_standalone": adam_alone,
    }
    opt.close()
    del opt
    host_release()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleSample(w)
        runs = [smp.run() for _ in range(args.cpu_repeats)]
        full = statistics.median(r[1] for r in runs)
        out["cpu_baseline"] = {"value": round(1.0 / full, 6), "unit": "steps/s", "cores": host_cores(), **blas_threads(),
                               "kind": "oracle", "extrapolated": not smp.whole,
                               "sample": f"{smp.desc}; median of {len(runs)} passes, each "
                                         f"{statistics.median(r[0] for r in runs):.2f} s of oracle work"}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args):
    import workloads

    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = workloads.get_workload(args.workload)
    smp = OracleSample(w)
    for _ in range(args.warmup):
        smp.run()
    t_wall = time.perf_counter()
    runs = [smp.run() for _ in range(args.steps)]
    t_wall = time.perf_counter() - t_wall
    ran = sum(r[0] for r in runs)
    full = sum(r[1] for r in runs)
    value = args.steps / full
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ran * 1e3 / args.steps, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": w.name, "parallelism": "host CPU, rank 0 only"},
        "extrapolated": not smp.whole,
        "sample": {"what_ran": smp.desc, "steps_timed": args.steps,
                   "oracle_s_per_timed_step": round(ran / args.steps, 4),
                   "full_step_s_estimated": round(full / args.steps, 4), "wall_s_timed_region": round(t_wall, 3),
                   "how": "each timed step runs the sample once (ms_per_step is its time); value is the "
                          "estimated rate of whole optimizer steps"},
        "cpu_baseline": {"value": round(value, 6), "unit": "steps/s", "cores": host_cores(), **blas_threads(), "kind": "oracle",
                         "extrapolated": not smp.whole, "sample": smp.desc},
        "e2e": {"value": round(value, 6), "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def run_shard_projection(args):
    """Per-rank compute of the sharded step, projected on one GPU (not a
    multi-GPU measurement): the ranks of a world run one after another on one
    GPU, sharing the parameter tensors (each writes only what it owns), none
    waiting on another. Each rank's step_begin + step_end is timed with CUDA
    events (median of `--steps` steps after `--warmup`); the collectives are
    not included. Prints one JSON line."""
    import statistics

    import torch

    import muon_adamw_hybrid_grad_gb300 as mx
    import workloads

    mx.load_library()
    w = workloads.get_workload(args.workload)
    lr = w.lr
    if w.schedule is not None:
        step_, total_, warm_, min_rate = w.schedule
        lr = w.lr * mx.muon_adamw_cosine_with_min_lr(step_, total_, warm_, min_rate)
    dev = torch.device("cuda")
    gdt = torch.bfloat16 if w.grad_dtype == "bf16" else torch.float32
    n = len(w.tensors)
    entries = [None] * n
    for batch in _batches(range(n)):
        ms = workloads.master_weights(w, batch)
        gs = workloads.gradients(w, 1, batch)
        for i, m, g in zip(batch, ms, gs):
            t = w.tensors[i]
            p = torch.from_numpy(m).to(dev)
            gt = None if t.frozen else torch.from_numpy(g).to(gdt).to(dev)
            sh = torch.empty(t.shape, dtype=torch.bfloat16, device=dev) if (w.policy == "bf16_mixed" and not t.frozen) else None
            entries[i] = (t.name, p, gt, sh, mx.MA_GROUP_FROZEN if t.frozen else None)
        del ms, gs
    prec = mx.MA_BF16_MIXED if w.policy == "bf16_mixed" else mx.MA_FP32_MIXED
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    out = {"shard_projection": {"workload": args.workload, "steps": args.steps, "warmup": args.warmup,
                                "how": run_shard_projection.__doc__.split("\n\n")[0].replace("\n", " ")}}
    opt = mx.MuonAdamW(entries, precision=prec, stream=stream)
    ts = []
    for k in range(args.warmup + args.steps):
        a, b = ev(), ev()
        a.record(stream)
        opt.step(lr)
        b.record(stream)
        torch.cuda.synchronize()
        if k >= args.warmup:
            ts.append(a.elapsed_time(b))
    opt.close()
    out["shard_projection"]["world1_ms"] = round(statistics.median(ts), 3)
    for world in (2, 4, 8):
        opts = [mx.MuonAdamW(entries, precision=prec, stream=stream, shard=(r, world)) for r in range(world)]
        loc = [torch.zeros(1, dtype=torch.float64, device=dev) for _ in range(world)]
        per = [[] for _ in range(world)]
        for k in range(args.warmup + args.steps):
            eb = [(ev(), ev()) for _ in range(world)]
            ee = [(ev(), ev()) for _ in range(world)]
            for r in range(world):
                eb[r][0].record(stream)
                opts[r].step_begin(lr, loc[r])
                eb[r][1].record(stream)
            tot = sum(loc[1:], loc[0].clone())  # what the all-reduce returns
            for r in range(world):
                ee[r][0].record(stream)
                opts[r].step_end(tot)
                ee[r][1].record(stream)
            torch.cuda.synchronize()
            if k >= args.warmup:
                for r in range(world):
                    per[r].append(eb[r][0].elapsed_time(eb[r][1]) + ee[r][0].elapsed_time(ee[r][1]))
        for o in opts:
            o.close()
        med = [statistics.median(x) for x in per]
        out["shard_projection"][f"world{world}"] = {
            "rank_ms": [round(x, 3) for x in med], "max_ms": round(max(med), 3),
            "mean_ms": round(sum(med) / world, 3), "max_over_mean": round(max(med) / (sum(med) / world), 3)}
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="full_vla")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-repeats", type=int, default=2, help="passes of the oracle sample for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shard-projection", action="store_true",
                    help="instead of the benchmark: per-rank compute of the sharded step for worlds of 2, 4 "
                         "and 8, projected on one GPU (ranks run one after another)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE is {world}: launch one process per GPU, e.g. "
                 f"python -m torch.distributed.run --nnodes=1 --nproc-per-node {args.gpus} --master-addr 127.0.0.1 "
                 f"bench.py --gpus {args.gpus}")
    if args.shard_projection:
        if world != 1:
            ap.error("--shard-projection runs on one GPU")
        run_shard_projection(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
