"""Benchmark: one step = route preprocessing + forward + backward of exact
route-set sparse GQA attention on the training-step workload (B=1,
S_q=S_kv=32768, Hq=32, Hkv=4, D=256, K=2048 int32 routes: 48 random causal
64-token blocks clipped to 2048 ids), BF16.  The right-padded block-route
workload (B=2, S=4096, Hq=16, Hkv=2) is timed the same way in the same run and
reported under ``per_config``.

Prints ONE JSON line (rank 0).  ``value`` is useful TFLOP/s over deduplicated
valid routes: forward 4*Hq*D*K_eff and backward 10*Hq*D*K_eff FLOP per query
row, divided by the device time of the step with inputs already in HBM.  The
L2 cache is flushed (a 256 MiB write) before every timed step, outside the
timed events.  ``e2e`` is the same metric through the public API with pinned
host buffers: host->device copies of Q, K, V, dO and the routes and
device->host copies of O, LSE, dQ, dK, dV are inside its timed region.

``--impl reference`` times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload, on the host cores.

``--route-producer`` measures the route producer instead (compressed-block
index scores + top-k selection, ``select_qsa_token_ids``) on the training-step
index workload (B=1, S=32768, H_index=32, D_index=128, c=4, budget 2048): one
step = one ``qsa_select_token_ids`` call (score kernel + selection kernel);
``value`` is useful TFLOP/s of the scoring (2*H*D per visible (row, block)
pair) over the whole step.  The score kernel is also timed alone; the
selection's time is the step's minus that.  With ``--impl reference`` it times
the oracle on sampled rows.

Multi-GPU (torchrun): every rank runs its own replica of the workload (the
path needs no exchange); the barrier and the max-over-ranks timing use
torch.distributed, nothing on the data path does.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from route_sparse_gqa_gb300 import workloads as W  # noqa: E402

METRIC = "route-sparse GQA fwd+bwd useful TFLOP/s on 1 GB300; % of roofline"
UNIT = "TFLOP/s"
FLOP_FWD_PER_KEY = 4   # x Hq x D per valid (row, key)
FLOP_BWD_PER_KEY = 10  # x Hq x D: S recompute, dP, dV, dQ, dK matmuls
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def work_counts(w, counts: np.ndarray):
    keff = int(counts.astype(np.int64).sum())
    rows = int((counts > 0).sum())
    D = w.D
    return {
        "keff_total": keff,
        "rows_nonempty": rows,
        "fwd_flop": FLOP_FWD_PER_KEY * w.Hq * D * keff,
        "bwd_flop": FLOP_BWD_PER_KEY * w.Hq * D * keff,
        # Algorithmic bytes (per query row): gathered bf16 K and V rows of every routed key for each KV head,
        # plus the row's own Q read / O write / LSE write (forward) or Q, dO read and dQ write plus LSE and
        # Delta reads (backward); backward also scatter-adds fp32 dK and dV (8 bytes per routed element).
        "fwd_bytes": 4 * w.Hkv * D * keff + rows * (w.Hq * D * 4 + 4 * w.Hq),
        "bwd_bytes": 12 * w.Hkv * D * keff + rows * (w.Hq * D * 6 + 8 * w.Hq),
    }


def executed_pairs(w, ids: np.ndarray, counts: np.ndarray) -> dict:
    """Tensor-core (query-head row, key) pairs each kernel family computes per KV head, over the useful ones
    (routed pairs x G heads).  The tile kernels compute every key of a T-query tile's union of route sets,
    packed 64 at a time; the key-major kernels compute every key of an aligned 64-key chunk for groups of T
    routing queries inside one query window (the window the library sizes to 32 MiB of fp32 dQ per KV head).
    Host-side bookkeeping from the route sets; the forward's key-major max pass recomputes S once more."""
    G = w.Hq // w.Hkv
    T = 128 // G
    useful = int(counts.astype(np.int64).sum()) * G
    B, S_q, K = ids.shape
    tile_chunks = 0
    for b in range(B):
        for t0 in range(0, S_q, T):
            blk = ids[b, t0:t0 + T]
            tile_chunks += -(-np.unique(blk[blk >= 0]).size // 64)
    n_blk = -(-S_q // 64)
    w_max = max(256, (32 << 20) // (G * w.D * 4))
    n_win = -(-n_blk // (-(-w_max // 64)))
    win_rows = -(-n_blk // n_win) * 64
    NC = -(-w.S_kv // 64)
    groups = 0
    for b in range(B):
        c = np.where(ids[b] >= 0, ids[b] // 64, -1)
        first = np.ones_like(c, dtype=bool)
        first[:, 1:] = c[:, 1:] != c[:, :-1]
        keep = first & (c >= 0)
        win = np.broadcast_to((np.arange(S_q) // win_rows)[:, None], c.shape)
        n = np.bincount((win[keep].astype(np.int64) * NC + c[keep]), minlength=n_win * NC)
        groups += int((-(-n // T)).sum())
    tile = tile_chunks * 64 * 128
    km = groups * 64 * 128
    return {"tile_over_useful": round(tile / max(useful, 1), 3), "keymajor_over_useful": round(km / max(useful, 1), 3),
            "tile_chunks": int(tile_chunks), "keymajor_groups": groups}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"qsa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# Sources each profiled kernel is built from: a recorded DRAM traffic figure stays
# valid until one of them changes.
KERNEL_SOURCES = {
    "qsa_forward": ["qsa_fwd_tc.cu", "qsa_fwd_km.cu", "qsa_tc_host.cu", "qsa_tc_ptx.cuh", "qsa_queue.cuh", "qsa_tc.cuh",
                    "qsa_internal.cuh"],
    "qsa_backward": ["qsa_bwd_km.cu", "qsa_chunks.cu", "qsa_bwd_tc.cu", "qsa_tc_host.cu", "qsa_tc_ptx.cuh",
                     "qsa_queue.cuh", "qsa_tc.cuh", "qsa_internal.cuh"],
    "index_score_kernel": ["qsa_route.cu", "qsa_tc_host.cu", "qsa_tc_ptx.cuh", "qsa_queue.cuh", "qsa_tc.cuh",
                           "qsa_internal.cuh"],
    "select_kernel": ["qsa_route.cu"],
}


def _code_only(src: bytes) -> bytes:
    """C/C++ source with its // and /* */ comments removed and every run of white space reduced to one
    space (string and character literals are kept), so that editing comments or layout alone leaves
    the hash below, and the measurements recorded against it, valid."""
    out = bytearray()
    i, n = 0, len(src)
    while i < n:
        c = src[i]
        if c in (0x22, 0x27):  # a string or character literal, copied through with its escapes
            out.append(c)
            i += 1
            while i < n:
                d = src[i]
                out.append(d)
                i += 1
                if d == 0x5C and i < n:
                    out.append(src[i])
                    i += 1
                elif d == c:
                    break
        elif src.startswith(b"//", i):
            j = src.find(b"\n", i)
            i = n if j < 0 else j
        elif src.startswith(b"/*", i):
            j = src.find(b"*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(0x20)
        else:
            out.append(c)
            i += 1
    return re.sub(rb"\s+", b" ", bytes(out)).strip()


def kernel_source_hash(kernel: str | None = None) -> str:
    """Hash of the code of the kernel's source files, comments and layout aside (every CUDA source when
    `kernel` is None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "route_sparse_gqa_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel) if kernel else None
    for name in sorted(names or os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()) + b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str | None = None):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was
    taken on the kernel's current sources (and, when `workload` is given, on that
    workload)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(f"{kernel}@{workload}") if workload else None
    entry = entry or rec.get(kernel)
    if not entry or entry.get("source_hash") != kernel_source_hash(kernel):
        return None
    if workload and entry.get("workload") not in (None, workload):
        return None
    return entry.get("bytes_per_launch")


def max_over_ranks(local_ms: float, device=None) -> float:
    """The slowest replica's per-step time: every rank's own time reduced with MAX
    (the local time when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(local_ms)
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_step_per_rank: float, world: int, step_ms: float) -> float:
    """Whole-job rate: every rank runs its own replica of the step (weak scaling),
    so the job does world x the per-rank work in the slowest rank's time."""
    return flop_per_step_per_rank * world / (step_ms * 1e-3) / 1e12


def make_device_inputs(case, device):
    import torch

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

    return bf(case.q), bf(case.k), bf(case.v), bf(case.do), torch.from_numpy(case.routes).to(device)


HEADLINE_WORKLOAD = 4   # train-step: the largest workload that fits one GPU
SECOND_WORKLOAD = 1     # right-padded-blocks: the other workload the targets name


def time_attention(args, index, dev, qsa, flush, world, sample_clocks):
    """Times `args.steps` steps (preprocess + forward + backward) of workload `index` with its inputs
    resident in HBM; returns the timings, work counts and roofline of the dominant entry point."""
    import torch
    import torch.distributed as dist

    w = W.WORKLOADS[index]
    case = W.make_case(index)
    q, k, v, do, routes = make_device_inputs(case, dev)
    scale = w.softmax_scale

    def step(timers=None):
        if timers:
            timers[0].record()
        plan = qsa.preprocess(q, k, v, routes, scale)
        if timers:
            timers[1].record()
        o, lse = qsa.forward(plan, q, k, v)
        if timers:
            timers[2].record()
        dq, dk, dv = qsa.backward(plan, q, k, v, o, lse, do, deterministic=args.deterministic)
        if timers:
            timers[3].record()
        return plan, o, lse, dq, dk, dv

    plan, *_ = step()
    ids, counts = plan.route_sets()
    plan.device_status()
    wc = work_counts(w, counts.cpu().numpy())
    pairs = executed_pairs(w, ids.cpu().numpy(), counts.cpu().numpy())
    del ids
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index) if sample_clocks else None
    if clocks:
        clocks.__enter__()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)  # L2 flush between timed steps, outside the events
        step(events[i])
    torch.cuda.synchronize()
    if clocks:
        clocks.__exit__(None, None, None)
    if world > 1:
        dist.barrier()
    per = np.array([[events[i][j].elapsed_time(events[i][j + 1]) for j in range(3)] for i in range(args.steps)])
    step_ms = float(per.sum(1).sum() / args.steps)
    step_ms_max = max_over_ranks(step_ms, dev)
    pre_ms, fwd_ms, bwd_ms = (float(x) for x in per.mean(0))
    plan.device_status()
    del plan
    flop_step = wc["fwd_flop"] + wc["bwd_flop"]

    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tc_peak = float(peaks["bf16_tflops"])  # burst figure: each entry point runs for milliseconds
    fwd_tf = wc["fwd_flop"] / (fwd_ms * 1e-3) / 1e12
    bwd_tf = wc["bwd_flop"] / (bwd_ms * 1e-3) / 1e12
    fwd_gbs = wc["fwd_bytes"] / (fwd_ms * 1e-3) / 1e9
    bwd_gbs = wc["bwd_bytes"] / (bwd_ms * 1e-3) / 1e9
    dominant = "backward" if bwd_ms >= fwd_ms else "forward"
    kern = {"forward": ("qsa_forward", fwd_tf, wc["fwd_flop"], fwd_ms),
            "backward": ("qsa_backward", bwd_tf, wc["bwd_flop"], bwd_ms)}[dominant]
    # The kernels reuse every gathered K/V row for many (query, head) rows, so their DRAM traffic is far
    # below the per-row gathered bytes; the binding peak is the tensor pipe.  Useful FLOP (valid routes only)
    # never exceed executed FLOP, so achieved/peak is a true fraction.  The gathered-bytes view is kept below.
    roofline = {
        "bound": "tensor",
        "achieved": round(kern[1], 2),
        "peak": tc_peak,
        "unit": "TFLOP/s",
        "frac": round(kern[1] / tc_peak, 4),
        "traffic": recorded_traffic(kern[0], w.name),
        "kernel": kern[0],
        "algorithmic_flop_per_launch": kern[2],
        "launch_ms": round(kern[3], 4),
        "peak_source": (f"{peak_src} MEASURED_PEAKS.json bf16_tflops" if peak_src == "measured"
                        else "fallback 1.9 PFLOP/s"),
        "fwd_tflops": round(fwd_tf, 2),
        "bwd_tflops": round(bwd_tf, 2),
        "fwd_frac": round(fwd_tf / tc_peak, 4),
        "bwd_frac": round(bwd_tf / tc_peak, 4),
        "executed_pairs": pairs,
        "gathered_bytes": {
            "note": "per-row K/V gather model (no reuse); DRAM traffic is far lower, so fractions exceed 1",
            "fwd_gbs": round(fwd_gbs, 1),
            "bwd_gbs": round(bwd_gbs, 1),
            "fwd_frac_of_hbm": round(fwd_gbs / hbm, 3),
            "bwd_frac_of_hbm": round(bwd_gbs / hbm, 3),
            "hbm_peak_gbs": hbm,
        },
    }
    return {
        "w": w, "case": case, "wc": wc, "flop_step": flop_step, "step_ms": step_ms_max,
        "value": job_tflops(flop_step, world, step_ms_max),
        "breakdown_ms": {"preprocess": round(pre_ms, 4), "forward": round(fwd_ms, 4), "backward": round(bwd_ms, 4)},
        "roofline": roofline, "clocks": clocks.summary() if clocks else None,
    }


def run_ours(args):
    import torch
    import torch.distributed as dist

    import route_sparse_gqa_gb300 as qsa
    from route_sparse_gqa_gb300 import build as qbuild

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    qbuild.build()
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)

    head = time_attention(args, args.workload, dev, qsa, flush, world, sample_clocks=True)
    w, case = head["w"], head["case"]
    # End to end through the public API with pinned host buffers.
    e2e = run_e2e(case, w, dev, args, qsa, head["flop_step"], world)
    # The other workload the targets name, timed the same way (its own step, breakdown and roofline).
    per_config = {}
    if args.workload != SECOND_WORKLOAD and not args.no_second:
        second = time_attention(args, SECOND_WORKLOAD, dev, qsa, flush, world, sample_clocks=False)
        per_config[second["w"].name] = {
            "value": round(second["value"], 3), "unit": UNIT, "ms_per_step": round(second["step_ms"], 4),
            "workload": f"{second['w'].name}: {second['w'].summary}",
            "useful_flop_per_step": second["flop_step"], "breakdown_ms": second["breakdown_ms"],
            "roofline": second["roofline"],
        }
        del second
    cpu = run_cpu_baseline(case, w, args) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    wc = head["wc"]
    line = {
        "metric": METRIC,
        "value": round(head["value"], 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(head["step_ms"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{w.name}: {w.summary}",
            "step": ("preprocess + forward + deterministic backward (fixed-point dK/dV sums)" if args.deterministic
                     else "preprocess + forward + backward (fp32 dK/dV accumulation)"),
            "parallelism": f"replicas x{world}",
            "l2": "flushed before every timed step (256 MiB write outside the events)",
            "keff_total": wc["keff_total"],
            "rows_nonempty": wc["rows_nonempty"],
            "useful_flop_per_step": head["flop_step"],
        },
        "breakdown_ms": head["breakdown_ms"],
        "roofline": head["roofline"],
        "per_config": per_config,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * LAUNCHES_PER_STEP,
        "clocks": head["clocks"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# libqsa kernels per step on the headline workload.  Preprocess: route rows, the 7 reverse-list kernels
# (masks, column scan, two scans, fill, items, queue), the path choice, route tiles and tile order (both
# return at once when the key-major kernels run both ways) = 11.  Forward: the tile forward (returns at once)
# + the key-major forward's key norms, init, row-max pass (returns at once when every row's bound serves),
# output pass and final division = 6.  Backward: delta, the tile backward (returns at once), the key-major
# kernel, dQ conversion, dK/dV conversion = 5.
LAUNCHES_PER_STEP = 11 + 6 + 5


def pipelined_e2e(dev, host: dict, outs: dict, compute_fn, n: int, n_slots: int) -> float:
    """Milliseconds per step of an end-to-end loop through the public API: every
    step copies its own inputs (`host`, pinned) to the device and its results
    (`compute_fn(device_inputs)` -> {name: tensor}) back into `outs` (pinned).

    Pipelined like a training input pipeline: device inputs are in `n_slots`
    buffers, the host->device copy of a later step runs on its own stream while a
    step computes, and the device->host copy of a step's results on a third
    stream.  Events order each buffer's reuse; all copies stay in the timed region."""
    import torch

    comp = torch.cuda.current_stream(dev)
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dev_in = [{name: torch.empty_like(t, device=dev) for name, t in host.items()} for _ in range(n_slots)]
    copied = [torch.cuda.Event() for _ in range(n_slots)]   # inputs of a slot are on the device
    used = [torch.cuda.Event() for _ in range(n_slots)]     # compute finished with a slot's inputs
    drained = [None] * n_slots                              # results of a slot's last step are on the host

    def copy_in(slot):
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(used[slot])
            for name, t in host.items():
                dev_in[slot][name].copy_(t, non_blocking=True)
            copied[slot].record(h2d_s)

    def compute(slot):
        comp.wait_event(copied[slot])
        res = compute_fn(dev_in[slot])
        used[slot].record(comp)
        done = torch.cuda.Event()
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(used[slot])
            for name, t in res.items():
                t.record_stream(d2h_s)
                outs[name].copy_(t, non_blocking=True)
            done.record(d2h_s)
        drained[slot] = done

    def run(k):
        for i in range(min(n_slots - 1, k)):
            copy_in(i % n_slots)
        for i in range(k):
            if i + n_slots - 1 < k:
                copy_in((i + n_slots - 1) % n_slots)
            compute(i % n_slots)
        for e in drained:
            if e is not None:
                comp.wait_event(e)

    run(2)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    h2d_s.wait_event(t0)
    run(n)
    t1.record(comp)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / n


def run_e2e(case, w, dev, args, qsa, flop_step, world):
    import torch

    host = {}
    for name in ("q", "k", "v", "do"):
        bits = np.ascontiguousarray(getattr(case, name)).view(np.int16)
        host[name] = torch.from_numpy(bits).view(torch.bfloat16).pin_memory()
    host["routes"] = torch.from_numpy(case.routes).pin_memory()
    outs = {
        "o": torch.empty((w.B, w.S_q, w.Hq, w.D), dtype=torch.bfloat16).pin_memory(),
        "lse": torch.empty((w.B, w.Hq, w.S_q), dtype=torch.float32).pin_memory(),
        "dq": torch.empty((w.B, w.S_q, w.Hq, w.D), dtype=torch.bfloat16).pin_memory(),
        "dk": torch.empty((w.B, w.S_kv, w.Hkv, w.D), dtype=torch.bfloat16).pin_memory(),
        "dv": torch.empty((w.B, w.S_kv, w.Hkv, w.D), dtype=torch.bfloat16).pin_memory(),
    }
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs.values())

    def compute_fn(x):
        plan = qsa.preprocess(x["q"], x["k"], x["v"], x["routes"], w.softmax_scale)
        o, lse = qsa.forward(plan, x["q"], x["k"], x["v"])
        dq, dk, dv = qsa.backward(plan, x["q"], x["k"], x["v"], o, lse, x["do"], deterministic=args.deterministic)
        return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}

    n_slots = int(os.environ.get("QSA_E2E_SLOTS", "2"))
    # At least 10 steps, so that the first step's input copy and the last step's result copy (the
    # pipeline's fill and drain, which nothing overlaps) are not most of the figure.
    n = max(10, args.steps)
    ms = max_over_ranks(pipelined_e2e(dev, host, outs, compute_fn, n, n_slots), dev)
    return {"value": round(job_tflops(flop_step, world, ms), 3), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "pipeline": f"inputs in {n_slots} device buffers; later steps' H2D and earlier steps' D2H overlap each step's compute"}


def oracle_sample(case, w, rows_per_sample: int, seed: int = 0):
    """A bounded sample of the workload for the CPU oracle: `rows_per_sample`
    evenly spaced non-empty query rows of batch row 0, with all their keys."""
    import oracle

    _, counts = oracle.route_sets(case.routes[:1], w.S_kv)
    live = np.nonzero(counts[0] > 0)[0]
    rows = live[np.linspace(0, live.size - 1, min(rows_per_sample, live.size)).astype(np.int64)]
    f64 = lambda bits: W.bf16_bits_to_f32(bits).astype(np.float64)  # noqa: E731
    sub = {
        "q": f64(case.q[:1, rows]), "do": f64(case.do[:1, rows]), "routes": case.routes[:1, rows],
        "k": f64(case.k[:1]), "v": f64(case.v[:1]),
    }
    keff = int(counts[0, rows].astype(np.int64).sum())
    return sub, rows.size, keff


def time_oracle_step(sub, w):
    import oracle

    t0 = time.perf_counter()
    o, lse = oracle.forward(sub["q"], sub["k"], sub["v"], sub["routes"], w.softmax_scale)
    oracle.backward(sub["q"], sub["k"], sub["v"], sub["routes"], sub["do"], w.softmax_scale)
    return time.perf_counter() - t0


def run_cpu_baseline(case, w, args):
    import oracle

    oracle.build()
    sub, n_rows, keff = oracle_sample(case, w, args.cpu_rows)
    secs = time_oracle_step(sub, w)
    flop = (FLOP_FWD_PER_KEY + FLOP_BWD_PER_KEY) * w.Hq * w.D * keff
    return {"value": round(flop / secs / 1e12, 6), "unit": UNIT, "cores": oracle.omp_threads(), "kind": "oracle",
            "seconds": round(secs, 2),
            "sample": f"{n_rows} evenly spaced non-empty query rows of batch row 0 ({keff} routed keys), "
                      f"forward + backward with dK/dV over all {w.S_kv} keys, fp64"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    w = W.WORKLOADS[args.workload]
    case = W.make_case(args.workload)
    sub, n_rows, keff = oracle_sample(case, w, args.ref_rows)
    flop = (FLOP_FWD_PER_KEY + FLOP_BWD_PER_KEY) * w.Hq * w.D * keff
    for _ in range(args.warmup):
        time_oracle_step(sub, w)
    secs = [time_oracle_step(sub, w) for _ in range(args.steps)]
    total = sum(secs)
    value = flop * args.steps / total / 1e12
    sample = (f"{n_rows} evenly spaced non-empty query rows of batch row 0 ({keff} routed keys) per step, "
              f"forward + backward with dK/dV over all {w.S_kv} keys, fp64")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.summary}", "step": "oracle forward + backward on a bounded sample",
                   "parallelism": "CPU threads (OpenMP)"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": oracle.omp_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


ROUTE_METRIC = "QSA route producer (index scores + top-k block selection) useful TFLOP/s on 1 GB300"
ROUTE_WORKLOAD = 3  # index-train-step


def route_work(w, lengths):
    """Visible (row, block) pairs of live rows and the scoring FLOP on them."""
    tg = np.arange(w.S_q, dtype=np.int64) + w.offset
    pairs = 0
    for L in lengths:
        live = tg < int(L)
        pairs += int(np.minimum((tg[live] + 1) // w.c, w.n_blocks).sum())
    rows = int(sum(min(w.S_q, max(0, int(L) - w.offset)) for L in lengths))
    return pairs, 2 * w.H * w.D * pairs, rows


def run_route_producer(args):
    import ctypes

    import torch
    import torch.distributed as dist

    import route_sparse_gqa_gb300 as qsa
    from route_sparse_gqa_gb300 import _abi
    from route_sparse_gqa_gb300 import build as qbuild

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    qbuild.build()
    case = W.make_index_case(ROUTE_WORKLOAD)
    w = case.workload
    bf = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)  # noqa: E731
    q, k = bf(case.q).to(dev), bf(case.k).to(dev)
    lens = torch.from_numpy(case.lengths).to(dev)
    prob, qq, kk = qsa.routes._problem(q, k, w.budget, w.c, w.offset, w.S_global)
    lib = _abi.load()
    ws_bytes = lib.qsa_route_workspace_bytes(ctypes.byref(prob))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    scores_ptr = ws.data_ptr() + 512  # the workspace's score tensor
    W_ = w.budget + w.c - 1
    ids = torch.empty((w.B, w.S_q, W_), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
    pairs, flop, live_rows = route_work(w, case.lengths)

    def step(ev=None):
        # The product call: scores into the workspace, then the selection.
        if ev:
            ev[0].record()
        _abi.check(lib.qsa_select_token_ids(ctypes.byref(prob), qq.data_ptr(), kk.data_ptr(), lens.data_ptr(),
                                            ws.data_ptr(), ws_bytes, ids.data_ptr(), stream))
        if ev:
            ev[1].record()

    def scores_only(ev):
        ev[0].record()
        _abi.check(lib.qsa_index_scores(ctypes.byref(prob), qq.data_ptr(), kk.data_ptr(), lens.data_ptr(),
                                        ws.data_ptr(), ws_bytes, scores_ptr, stream))
        ev[1].record()

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    _abi.check(lib.qsa_read_device_status(ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(stream)))
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            step(events[i])
        torch.cuda.synchronize()
        # The score kernel alone (same launches as inside the product call), for the breakdown.
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            scores_only(sev[i])
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # The producer followed by the attention's route preprocessing on its rows, timed as one sequence: the
    # rows arrive sorted, so route_rows copies them through.  Attention shape of the train-step workload
    # (Hq32 Hkv4 D256) over the producer's rows; the tensors' contents are not read by the preprocessing.
    att = W.WORKLOADS[HEADLINE_WORKLOAD]
    aq = torch.empty((w.B, w.S_q, att.Hq, att.D), dtype=torch.bfloat16, device=dev)
    akv = torch.empty((w.B, w.S_global, att.Hkv, att.D), dtype=torch.bfloat16, device=dev)
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    plan = None
    for i in range(args.steps + max(1, args.warmup)):
        timed = i >= max(1, args.warmup)
        flush.fill_(i & 0xFF)
        ev = pev[i - max(1, args.warmup)] if timed else None
        step(ev)
        plan = qsa.preprocess(aq, akv, akv, ids, att.softmax_scale, routes_sorted=True)
        if ev:
            ev[2].record()
    torch.cuda.synchronize()
    plan.device_status()
    del plan, aq, akv
    with_pre_ms = float(np.mean([e[0].elapsed_time(e[2]) for e in pev]))
    pre_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in pev]))

    local_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in events]))
    score_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in sev]))
    sel_ms = max(local_ms - score_ms, 1e-6)  # the selection and the launch between the kernels
    step_ms = max_over_ranks(local_ms, dev)
    value = job_tflops(flop, world, step_ms)
    _abi.check(lib.qsa_read_device_status(ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(stream)))

    # End to end through the public binding with pinned host buffers: H2D of the
    # index states and lengths, the producer, D2H of the route rows (pipelined).
    host = {"q": bf(case.q).pin_memory(), "k": bf(case.k).pin_memory(),
            "lens": torch.from_numpy(case.lengths).pin_memory()}
    outs = {"ids": torch.empty((w.B, w.S_q, W_), dtype=torch.int32).pin_memory()}

    def compute_fn(x):
        return {"ids": qsa.select_qsa_token_ids(x["q"], x["k"], x["lens"], w.budget, w.c,
                                                query_position_offset=w.offset, global_sequence_length=w.S_global)}

    n_slots = int(os.environ.get("QSA_E2E_SLOTS", "2"))
    n_e2e = max(10, args.steps)  # as in run_e2e: fill and drain spread over at least 10 steps
    e2e_ms = max_over_ranks(pipelined_e2e(dev, host, outs, compute_fn, n_e2e, n_slots), dev)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs.values())
    e2e = {"value": round(job_tflops(flop, world, e2e_ms), 3), "unit": UNIT, "ms_per_step": round(e2e_ms, 4),
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
           "pipeline": f"inputs in {n_slots} device buffers; later steps' H2D and earlier steps' D2H overlap each step's compute"}

    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tc_peak = float(peaks["bf16_tflops"])
    score_tf = flop / (score_ms * 1e-3) / 1e12
    sel_bytes = 4 * pairs + 4 * W_ * w.B * w.S_q + 8 * w.B  # scores read once, route rows written, lengths
    sel_gbs = sel_bytes / (sel_ms * 1e-3) / 1e9
    kernels = {
        "index_score_kernel": {"bound": "tensor", "achieved": round(score_tf, 2), "peak": tc_peak,
                               "unit": "TFLOP/s", "frac": round(score_tf / tc_peak, 4), "launch_ms": round(score_ms, 4),
                               "algorithmic_flop_per_launch": flop, "traffic": recorded_traffic("index_score_kernel")},
        "select_kernel": {"bound": "hbm", "achieved": round(sel_gbs, 1), "peak": hbm, "unit": "GB/s",
                          "frac": round(sel_gbs / hbm, 4), "launch_ms": round(sel_ms, 4),
                          "algorithmic_bytes_per_launch": sel_bytes, "traffic": recorded_traffic("select_kernel")},
    }
    dom = "select_kernel" if sel_ms >= score_ms else "index_score_kernel"
    roofline = dict(kernels[dom])
    roofline["kernel"] = dom
    roofline["peak_source"] = f"{peak_src} MEASURED_PEAKS.json" if peak_src == "measured" else "fallback"
    cpu = run_route_cpu_baseline(case, w, flop, live_rows, args) if (rank == 0 and world == 1 and
                                                                     not args.no_cpu_baseline) else None
    line = {
        "metric": ROUTE_METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{w.name}: {w.summary}",
            "step": "index scores (tcgen05) + top-k block selection and expansion",
            "parallelism": f"replicas x{world}",
            "l2": "flushed before every timed step (256 MiB write outside the events)",
            "visible_pairs": pairs,
            "useful_flop_per_step": flop,
        },
        "breakdown_ms": {"index_scores": round(score_ms, 4), "selection": round(sel_ms, 4)},
        "with_preprocess": {
            "ms_per_step": round(with_pre_ms, 4), "preprocess_ms": round(pre_ms, 4),
            "step": "producer, then qsa_preprocess of its route rows (QSA_ROUTES_SORTED: copied through)",
            "attention": f"{att.name}: B{w.B} S{w.S_q} Hq{att.Hq} Hkv{att.Hkv} D{att.D}, K={W_} producer slots",
        },
        "roofline": roofline,
        "kernels": kernels,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * 2,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


ROUTE_GROUP = 16  # contiguous query rows per oracle call (the oracle's threads split a call's rows)


def route_oracle_sample(case, w, n_rows: int):
    """Groups of ROUTE_GROUP contiguous live query rows of batch row 0, evenly
    spaced over the sequence, for the route-producer oracle."""
    live = min(w.S_q, int(case.lengths[0]) - w.offset)
    n_groups = max(1, min(n_rows // ROUTE_GROUP, live // ROUTE_GROUP))
    starts = np.linspace(0, live - ROUTE_GROUP, n_groups).astype(np.int64)
    rows = (starts[:, None] + np.arange(ROUTE_GROUP)[None, :]).reshape(-1)
    tg = rows + w.offset
    pairs = int(np.minimum((tg + 1) // w.c, w.n_blocks).sum())
    return starts, rows, pairs


def time_route_oracle(case, w, starts):
    import oracle

    f64 = lambda bits: W.bf16_bits_to_f32(bits).astype(np.float64)  # noqa: E731
    kd = f64(case.k[:1])
    qs = [f64(case.q[:1, s:s + ROUTE_GROUP]) for s in starts]
    t0 = time.perf_counter()
    for s, qd in zip(starts, qs):
        oracle.select_qsa_token_ids(qd, kd, case.lengths[:1], w.budget, w.c, w.offset + int(s))
    return time.perf_counter() - t0


def run_route_cpu_baseline(case, w, flop, live_rows, args):
    import oracle

    oracle.build()
    starts, rows, pairs = route_oracle_sample(case, w, args.route_cpu_rows)
    secs = time_route_oracle(case, w, starts)
    return {"value": round(2 * w.H * w.D * pairs / secs / 1e12, 6), "unit": UNIT,
            "cores": min(oracle.omp_threads(), ROUTE_GROUP), "kind": "oracle", "seconds": round(secs, 2),
            "sample": f"{starts.size} groups of {ROUTE_GROUP} contiguous query rows of batch row 0, evenly spaced "
                      f"({pairs} visible blocks), scores + selection in fp64"}


def run_route_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    case = W.make_index_case(ROUTE_WORKLOAD)
    w = case.workload
    starts, rows, pairs = route_oracle_sample(case, w, args.route_rows)
    for _ in range(args.warmup):
        time_route_oracle(case, w, starts[:1])
    secs = [time_route_oracle(case, w, starts) for _ in range(args.steps)]
    total = sum(secs)
    value = 2 * w.H * w.D * pairs * args.steps / total / 1e12
    sample = (f"{starts.size} groups of {ROUTE_GROUP} contiguous query rows of batch row 0, evenly spaced "
              f"({pairs} visible blocks) per step, scores + selection in fp64")
    line = {
        "impl": "reference", "metric": ROUTE_METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.summary}", "step": "oracle scores + selection on a bounded sample",
                   "parallelism": "CPU threads (OpenMP)"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": min(oracle.omp_threads(), ROUTE_GROUP),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=HEADLINE_WORKLOAD,
                    help="workload index (4 = train-step, the headline configuration)")
    ap.add_argument("--no-second", action="store_true",
                    help="skip the per_config timing of the right-padded workload")
    ap.add_argument("--cpu-rows", type=int, default=2048, help="query rows in the CPU-baseline oracle sample")
    ap.add_argument("--ref-rows", type=int, default=160, help="query rows per step of the reference (oracle) arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="time the bitwise reproducible backward (qsa_backward_deterministic)")
    ap.add_argument("--route-producer", action="store_true",
                    help="measure the route producer (index scores + top-k selection) instead of the attention")
    ap.add_argument("--route-rows", type=int, default=256,
                    help="query rows per step of the route-producer reference (oracle) arm")
    ap.add_argument("--route-cpu-rows", type=int, default=12288,
                    help="query rows in the route-producer CPU-baseline oracle sample")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.route_producer:
        (run_route_reference if args.impl == "reference" else run_route_producer)(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
