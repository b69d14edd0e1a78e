#!/usr/bin/env python3
"""Benchmark of the fused LM-head loss forward + backward on GB300.

One step = one call of lmloss_forward_backward over the whole workload: every
row's max, non-target sum, collapse-free NLL, z-loss / KL terms, the gradient
written once, and the loss reduction.  Default workload: confident_bf16
(T=16384 rows, V=128256, bf16, 30% of rows with a planted target margin in
[15, 40], CE, gradient in place, token mean) -- the shape the torchtitan PR
measured (there with V split over two GPUs).  On one GPU the line also times
the other large workloads at their full sizes (ce_z_bf16, gspo_z_bf16 and
ce_z_kl_bf16, the last with 2 x 34 GB of inputs), each the same way, under
"also" (`--also none` skips them).

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream.  Between steps, untimed: in-place workloads get their
logits back from a pristine device copy (the step overwrites them with the
gradient), and a 256 MB buffer is written to flush L2.

Output: one JSON line on rank 0.
  value      logit elements per second over all ranks, inputs resident in HBM
  e2e        the same metric through the C ABI with host buffers: each step
             takes the step's inputs from pinned host memory (the logits through
             lmloss_forward_backward_host, which copies them in row chunks and
             runs each chunk's kernel as it lands) and reads the 5 loss values
             back
  roofline   the staged-row kernel's algorithmic bytes (reads of active rows,
             the gradient write, side inputs) / its CUDA-event duration (events
             around each launch, in a second pass of K steps so that they do not
             slow the timed steps), against the measured HBM copy bandwidth
  cpu_baseline  the fp64 oracle on a bounded sample of rows, host cores

--impl reference times the oracle itself on the host cores (rank 0 only).
Multi-GPU (torchrun): each rank holds its own rows of a batch N times as tall
(weak scaling); every rank reduces with SUM over the global active count, a
host-side scalar, so no collective touches the data path.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "fused LM-loss fwd+bwd logit elems/s and HBM GB/s (% of GB300 peak)"
UNIT = "logit elems/s"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
GEN_CHUNK = 2048


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="confident_bf16")
    ap.add_argument("--also", default="auto",
                    help="comma-separated workloads timed after the main one at their full sizes; "
                         "'auto': the other large workloads on a single GPU, none under torchrun; 'none'")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle sample time")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-restore", action="store_true",
                    help="in-place workloads: time steps on the previous step's gradient")
    ap.add_argument("--cluster", type=int, default=0)
    ap.add_argument("--threads", type=int, default=0)
    ap.add_argument("--nbuf", type=int, default=0)
    ap.add_argument("--rows", type=int, default=0, help="profiling only: fewer rows than the workload")
    ap.add_argument("--temperature", type=float, default=0.0,
                    help="distillation temperature for a workload with a teacher (0: the workload's own)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest() -> str:
    """sha256 of the kernel sources (kernels.cuh, then ptx.cuh) with comments
    and blank lines removed: a comment edit leaves the recorded counters valid,
    any code edit does not."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("kernels.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "lm_head_vocab_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip()).encode())
    return h.hexdigest()


def read_traffic(workload: str, rows: int):
    """DRAM bytes per launch of the staged-row kernel from the ncu record
    profiles/traffic.json, if it was taken on the current kernel code (same
    kernel_source_digest); scaled to `rows` (every row is read and written
    once, so traffic grows in proportion).  None otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(workload)
    if not rec or rec.get("kernel_source_sha256") != kernel_source_digest():
        return None
    return int(round(rec["dram_bytes_per_launch"] * rows / rec["rows"]))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for k, nm in enumerate(names):
                if parts[5 + k].lower() in ("active", "1"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ inputs
class RankSlice:
    """This rank's share of workload w: its rows of a batch world x T rows tall
    (rows [r0, r0 + T) of wg), their targets and mask, the global active-row
    count, and for GSPO this rank's segments (renumbered from 0; packed rows
    never straddle ranks), their advantages and the old-log-prob noise.  Host
    only; the rows themselves come from wg.logits_rows / teacher_rows."""

    def __init__(self, w, rank: int, world: int):
        self.w = w
        self.wg = w if world == 1 else w.with_shape(w.T * world, w.V)
        self.r0 = rank * w.T
        self.targets = self.wg.targets()[self.r0:self.r0 + w.T].copy()
        mask = self.wg.loss_mask()
        self.mask = None if mask is None else mask[self.r0:self.r0 + w.T].copy()
        self.n_active_global = self.wg.n_active()
        self.gspo = None
        if w.has_gspo:
            if w.T % w.packed_len:
                raise SystemExit("bench: GSPO rows per rank must be whole packed rows")
            seg_all, _, adv_all = self.wg.segments()
            seg = seg_all[self.r0:self.r0 + w.T].copy()
            s0, s1 = int(seg.min()), int(seg.max()) + 1
            seg -= s0
            self.gspo = dict(seg=seg.astype(np.int32), S=s1 - s0, adv=adv_all[s0:s1].copy(),
                             noise=self.wg.old_logp_noise()[self.r0:self.r0 + w.T].astype(np.float32))

    def host_rows(self, n: int):
        """The first n rows of this rank on the host (logits, teacher)."""
        x = self.wg.logits_rows(self.r0, n)
        u = self.wg.teacher_rows(self.r0, n, x) if self.w.teacher_sigma is not None else None
        return x, u


class Problem(RankSlice):
    """A RankSlice with its rows generated on the host in chunks and copied to
    the device (optionally also kept in pinned host memory for the end-to-end
    leg)."""

    def __init__(self, w, dev, rank: int, world: int, keep_host: bool):
        import torch
        super().__init__(w, rank, world)
        tg_full = self.wg.targets()
        margins = self.wg.margins()
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.logits = torch.empty((w.T, w.row_stride), dtype=tdt, device=dev)
        self.teacher = torch.empty_like(self.logits) if w.teacher_sigma is not None else None
        self.hx = self.hu = None
        if keep_host:
            self.hx = torch.empty((w.T, w.row_stride), dtype=tdt, pin_memory=True)
            if self.teacher is not None:
                self.hu = torch.empty((w.T, w.row_stride), dtype=tdt, pin_memory=True)
        for a in range(0, w.T, GEN_CHUNK):
            n = min(GEN_CHUNK, w.T - a)
            x = self.wg.logits_rows(self.r0 + a, n, targets=tg_full, margins=margins)
            tx = _as_torch(x)
            self.logits[a:a + n].copy_(tx)
            if self.hx is not None:
                self.hx[a:a + n].copy_(tx)
            if self.teacher is not None:
                tu = _as_torch(self.wg.teacher_rows(self.r0 + a, n, x))
                self.teacher[a:a + n].copy_(tu)
                if self.hu is not None:
                    self.hu[a:a + n].copy_(tu)

def _as_torch(a):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


def call_kwargs(w, world, n_active_global):
    kw = dict(ce_weight=w.ce_weight, z_alpha=w.z_alpha, kl_weight=w.kl_weight, temperature=w.temperature)
    if w.has_gspo:
        kw.update(clip_eps_low=w.clip_eps_low, clip_eps_high=w.clip_eps_high)
    if world > 1 or w.reduction == "sum_active":
        kw.update(reduction="sum", denominator=float(n_active_global))
    else:
        kw.update(reduction="token_mean")
    return kw


def with_temperature(w, args):
    """The workload at the temperature asked for on the command line (teacher workloads only)."""
    if args.temperature > 0.0 and w.teacher_sigma is not None:
        from dataclasses import replace
        return replace(w, temperature=float(args.temperature))
    return w


def config_of(w, kw, world, grad_mode, restore):
    extra = {"temperature": w.temperature} if w.teacher_sigma is not None else {}
    return {
        "workload": w.name, "T_per_gpu": w.T, "V": w.V, "logits": w.dtype, **extra,
        "reduction": kw["reduction"], "grad": grad_mode,
        "l2": (f"inputs larger than L2 ({w.T * w.V * w.elem_bytes / 1e9:.2f} GB of logits per step) "
               f"and a {L2_FLUSH_BYTES >> 20} MB L2 flush between steps"),
        "inputs": ("logits restored from a pristine device copy before each step (untimed)"
                   if restore else "as generated"),
        "parallelism": f"rows x{world}" if world > 1 else "single GPU",
    }


# ------------------------------------------------------------ oracle timing
def oracle_sample_time(prob, seconds: float):
    """Time the fp64 oracle (forward + gradient) on the first R rows of the
    problem, R sized for about `seconds` of host work.  Returns (elements/s,
    cores, rows, description).  With GSPO the old log-probs are the seeded noise
    around -10: the oracle's work (forward, seam, gradient) does not depend on
    their values."""
    import oracle
    w = prob.w
    cores = os.cpu_count() or 1

    def run(rows):
        x, u = prob.host_rows(rows)
        P = oracle.Problem(logits=x, V=w.V, targets=prob.targets[:rows],
                           loss_mask=None if prob.mask is None else prob.mask[:rows], ce_weight=w.ce_weight,
                           z_alpha=w.z_alpha, teacher=u, kl_weight=w.kl_weight, temperature=w.temperature)
        if prob.gspo is not None:
            g = prob.gspo
            P.segment_ids = g["seg"][:rows]
            P.num_segments = g["S"]
            P.advantages = g["adv"]
            P.old_logprobs = (g["noise"][:rows] - 10.0).astype(np.float32)
            P.clip_eps_low, P.clip_eps_high = w.clip_eps_low, w.clip_eps_high
        t0 = time.perf_counter()
        oracle.forward_backward(P, nthreads=cores)
        return time.perf_counter() - t0

    probe = min(w.T, max(cores, 16))
    dt = run(probe)
    rows = int(min(w.T, max(probe, probe * seconds / max(dt, 1e-6))))
    rows = max(cores, rows - rows % cores) if rows >= cores else rows
    dt = run(rows)
    desc = (f"first {rows} of {w.T} rows (x {w.V} columns), fp64 forward+gradient, {cores} OpenMP threads, "
            f"input generation excluded")
    return rows * w.V / dt, cores, rows, desc


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import workloads

    w = with_temperature(workloads.get(args.workload), args)
    prob = RankSlice(w, 0, 1)
    per_step = []
    rows = 0
    cores = os.cpu_count() or 1
    for i in range(args.warmup + args.steps):
        v, cores, rows, desc = oracle_sample_time(prob, args.cpu_seconds / 4)
        if i >= args.warmup:
            per_step.append(v)
    value = statistics.median(per_step)
    elems = w.T * w.V
    kw = call_kwargs(w, 1, w.n_active())
    cfg = config_of(w, kw, 1, "inplace" if w.in_place else "new", False)
    cfg["inputs"] = "host arrays (the oracle's inputs)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elems / value,
        "ms_per_step_kind": f"extrapolated ({rows} of {w.T} rows timed per step, scaled to all rows)",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Philox4x32-10 inputs)",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
def time_workload(args, name, dev, world, rank, main: bool):
    """Times one workload; returns the fields of its result (rank 0) or None."""
    import torch
    import workloads
    from lm_head_vocab_gb300 import LMLoss

    wl = workloads.get(name)
    if args.rows and main:
        wl = wl.with_shape(args.rows, wl.V)
    if main:
        wl = with_temperature(wl, args)
    e2e_on = main and not args.no_e2e
    prob = Problem(wl, dev, rank, world, keep_host=e2e_on)
    w = prob.w
    kw = call_kwargs(w, world, prob.n_active_global)
    tg = torch.from_numpy(prob.targets).to(dev)
    mk = None if prob.mask is None else torch.from_numpy(prob.mask).to(dev)
    h = LMLoss(dev.index, max_T=w.T, max_segments=prob.gspo["S"] if prob.gspo else 1)
    if args.cluster or args.threads or args.nbuf:
        h.set_launch_config(args.cluster, args.threads, args.nbuf)
    grad_mode = "inplace" if w.in_place else "new"
    restore = w.in_place and not args.no_restore
    pristine = prob.logits.clone() if restore else None
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    gkw = {}
    old = None
    if prob.gspo is not None:
        # old log-probs for a timing run: this path's own log-probs plus the
        # seeded noise (the policy term's values do not change the work)
        a0, o0, k0 = h.build_args(prob.logits, tg, mk, grad=None, want=("logp",))
        h.call(a0)
        torch.cuda.synchronize(dev)
        old = (o0.logp + torch.from_numpy(prob.gspo["noise"]).to(dev)).contiguous()
        del a0, o0, k0
        gkw = dict(segment_ids=torch.from_numpy(prob.gspo["seg"]).to(dev), num_segments=prob.gspo["S"],
                   advantages=torch.from_numpy(prob.gspo["adv"]).to(dev), old_logprobs=old)
    a, out, keep = h.build_args(prob.logits, tg, mk, teacher_logits=prob.teacher, grad=grad_mode, want=(),
                                **gkw, **kw)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    def between_steps():
        # untimed: the inputs back to what the workload holds, then L2 flushed
        if restore:
            prob.logits.copy_(pristine)
        flush.zero_()

    def timed_steps(k):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        for e0, e1 in evs:
            between_steps()
            e0.record(stream)
            h.call(a, stream)
            e1.record(stream)
        barrier()
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    for _ in range(args.warmup):
        between_steps()
        h.call(a, stream)
    barrier()
    if h.device_error() != 0:
        raise SystemExit("device error during warm-up")
    info = h.call_info()

    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier()
    # the K timed steps, events around each whole call only (an event between a
    # call's kernels would cost a few microseconds and keep the reduction from
    # launching while the staged-row kernel finishes)
    step_list = timed_steps(args.steps)
    step_ms = sum(step_list) / len(step_list)
    # then K more steps with events around the staged-row kernel(s) of each call,
    # on the same stream: their average launch duration for the roofline
    h.set_timing(True)
    timed_steps(args.steps)
    kern_total, kern_calls = h.kernel_time()
    h.set_timing(False)
    clk = clocks.stop()
    kern_ms = kern_total / max(kern_calls, 1)
    if h.device_error() != 0:
        raise SystemExit("device error during the timed steps")

    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([step_ms, kern_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms, kern_ms = float(t[0]), float(t[1])

    elems_rank = w.T * w.V
    value = world * elems_rank / (step_ms / 1e3)
    alg_bytes = w.algorithmic_bytes()
    peak, peak_kind = read_peaks()
    # a distillation temperature other than 1 runs its own kernel instantiation: its own record
    traffic = read_traffic(w.name if w.temperature == 1.0 else f"{w.name}@tau={w.temperature:g}", w.T)
    achieved = alg_bytes / (kern_ms / 1e3) / 1e9

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if e2e_on:
        import torch as _t
        ht = _t.from_numpy(prob.targets).pin_memory()
        hm = None if prob.mask is None else _t.from_numpy(prob.mask).pin_memory()
        hloss = _t.empty(5, dtype=_t.float32).pin_memory()
        h2d = prob.hx.numel() * prob.hx.element_size() + ht.numel() * 8 \
            + (0 if prob.hu is None else prob.hu.numel() * prob.hu.element_size()) \
            + (0 if hm is None else hm.numel())
        hg = None
        if prob.gspo is not None:
            # the policy inputs travel too: segment ids, advantages, old log-probs
            hg = [(gkw["segment_ids"], _t.from_numpy(prob.gspo["seg"]).pin_memory()),
                  (gkw["advantages"], _t.from_numpy(prob.gspo["adv"]).pin_memory()),
                  (gkw["old_logprobs"], gkw["old_logprobs"].cpu().pin_memory())]
            h2d += sum(hs.numel() * hs.element_size() for _, hs in hg)

        # the small inputs by torch copies, the logits (and the teacher's) by the
        # host entry point, which copies them itself in row chunks
        def e2e_step():
            tg.copy_(ht, non_blocking=True)
            if hm is not None:
                mk.copy_(hm, non_blocking=True)
            if hg is not None:
                for dst, src in hg:
                    dst.copy_(src, non_blocking=True)
            h.call_host(a, prob.hx, prob.hu, 0, stream)
            hloss.copy_(out.loss, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        barrier()
        e0 = _t.cuda.Event(enable_timing=True)
        e1 = _t.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        barrier()
        e2e_ms = e0.elapsed_time(e1) / args.steps
        if world > 1:
            import torch.distributed as dist
            t = _t.tensor([e2e_ms], device=dev, dtype=_t.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_ms = float(t[0])
        e2e = {"value": world * elems_rank / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 20, "ms_per_step": e2e_ms}

    cpu = None
    if main and rank == 0 and world == 1 and not args.no_cpu:
        v, cores, _, desc = oracle_sample_time(prob, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    cfg = config_of(w, kw, world, grad_mode, restore)
    cfg["launch"] = {k: info[k] for k in ("cluster", "threads", "nbuf", "grid", "smem_bytes")}
    res = {
        "value": value, "ms_per_step": step_ms, "config": cfg, "dtype": w.dtype,
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": (f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                                     else "fallback 6.8 TB/s"),
                     "kernel_ms": kern_ms, "algorithmic_bytes": alg_bytes},
        "e2e": e2e, "cpu_baseline": cpu,
        "gpu_launches": int(info["launches"]) * args.steps,
        "clocks": clk,
    }
    h.close()
    del prob, pristine, flush, a, out, keep
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()

    main = time_workload(args, args.workload, dev, world, rank, main=True)
    also = {}
    names = args.also
    if names == "auto":
        names = "" if (world > 1 or args.rows) else "ce_z_bf16,gspo_z_bf16,ce_z_kl_bf16"
    for name in [n for n in names.split(",") if n and n not in ("none", args.workload)]:
        try:
            r = time_workload(args, name, dev, world, rank, main=False)
            also[name] = {k: r[k] for k in ("value", "ms_per_step", "roofline", "clocks", "config", "gpu_launches")}
        except Exception as e:   # the main line stands on its own
            also[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
            torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": main["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": main["dtype"],
            "data": "synthetic (seeded Philox4x32-10 inputs)",
            "config": main["config"], "hbm_gbs": main["hbm_gbs"], "roofline": main["roofline"],
            "e2e": main["e2e"], "cpu_baseline": main["cpu_baseline"],
            "gpu_launches": main["gpu_launches"], "clocks": main["clocks"],
        }
        if also:
            line["also"] = also
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
