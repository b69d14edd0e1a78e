#!/usr/bin/env python3
"""Benchmark of the fused LM-head loss forward + backward on GB300.

One step = one call of lmloss_forward_backward over the whole workload: every
row's max, non-target sum, collapse-free NLL, z-loss / KL terms, the gradient
written once, and the loss reduction.  Default workload: confident_bf16
(T=16384 rows, V=128256, bf16, 30% of rows with a planted target margin in
[15, 40], CE, gradient in place, token mean) -- the shape the torchtitan PR
measured (there with V split over two GPUs).

Output: one JSON line on rank 0.
  value      logit elements per second over all ranks, inputs resident in HBM
  e2e        the same metric through the C ABI with host buffers: each step
             copies the logits and targets from pinned host memory, runs the
             call, and reads the 5 loss values back
  roofline   the fused kernel's algorithmic bytes / its CUDA-event duration
             (events around each launch, in a second pass of K steps so that
             they do not slow the timed steps), against the measured HBM copy
             bandwidth
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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="confident_bf16")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle sample time")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cluster", type=int, default=0)
    ap.add_argument("--threads", type=int, default=0)
    ap.add_argument("--nbuf", type=int, default=0)
    ap.add_argument("--rows", type=int, default=0, help="profiling only: fewer rows than the workload")
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


def read_traffic(kernel_tag: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel code (same kernel_source_digest), else None."""
    prof = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(prof):
        return None
    digest = kernel_source_digest()
    vals = {}
    with open(prof) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != digest:
        return None
    try:
        return int(float(vals["dram_bytes_per_launch_full_workload"]))
    except (KeyError, ValueError):
        return None


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
def make_problem(w, rank: int, world: int):
    """This rank's rows of workload w (a batch world x T rows tall when world > 1),
    the global active-row count, and for GSPO this rank's segments (renumbered
    from 0; packed rows never straddle ranks) with their advantages and the
    rows' old-log-prob noise, all computed on the host from the seeds."""
    wg = w if world == 1 else w.with_shape(w.T * world, w.V)
    r0 = rank * w.T
    targets = wg.targets()[r0:r0 + w.T].copy()
    mask = wg.loss_mask()
    mask = None if mask is None else mask[r0:r0 + w.T].copy()
    margins = wg.margins()
    x = np.empty((w.T, w.row_stride), dtype=w.np_dtype)
    chunk = 2048
    tg_full = wg.targets()
    for a in range(0, w.T, chunk):
        n = min(chunk, w.T - a)
        x[a:a + n] = wg.logits_rows(r0 + a, n, targets=tg_full, margins=margins)
    u = None
    if w.teacher_sigma is not None:
        u = np.empty_like(x)
        for a in range(0, w.T, chunk):
            n = min(chunk, w.T - a)
            u[a:a + n] = wg.teacher_rows(r0 + a, n, x[a:a + n])
    n_active_global = wg.n_active()
    gspo = None
    if w.has_gspo:
        if w.T % w.packed_len:
            raise SystemExit("bench: GSPO rows per rank must be whole packed rows")
        seg_all, _, adv_all = wg.segments()
        seg = seg_all[r0:r0 + w.T].copy()
        s0, s1 = int(seg.min()), int(seg.max()) + 1
        seg -= s0
        gspo = dict(seg=seg.astype(np.int32), S=s1 - s0, adv=adv_all[s0:s1].copy(),
                    noise=wg.old_logp_noise()[r0:r0 + w.T].astype(np.float32))
    return w, x, u, targets, mask, n_active_global, gspo


def call_kwargs(w, world, n_active_global):
    kw = dict(ce_weight=w.ce_weight, z_alpha=w.z_alpha, kl_weight=w.kl_weight, temperature=w.temperature)
    if w.has_gspo:
        kw.update(clip_eps_low=w.clip_eps_low, clip_eps_high=w.clip_eps_high)
    if world > 1 or w.reduction == "sum_active":
        kw.update(reduction="sum", denominator=float(n_active_global))
    else:
        kw.update(reduction="token_mean")
    return kw


# ------------------------------------------------------------ oracle timing
def oracle_sample_time(w, x, u, targets, mask, seconds: float, gspo=None):
    """Time the fp64 oracle (forward + gradient) on the first R rows, R sized
    for about `seconds` of host work.  Returns (elements/s, cores, description).
    With GSPO the old log-probs are the seeded noise around -10: the oracle's
    work (forward, seam, gradient) does not depend on their values."""
    import oracle
    cores = os.cpu_count() or 1

    def run(rows):
        P = oracle.Problem(logits=x[:rows], V=w.V, targets=targets[:rows],
                           loss_mask=None if mask is None else mask[:rows], ce_weight=w.ce_weight,
                           z_alpha=w.z_alpha, teacher=None if u is None else u[:rows],
                           kl_weight=w.kl_weight, temperature=w.temperature)
        if gspo is not None:
            P.segment_ids = gspo["seg"][:rows]
            P.num_segments = gspo["S"]
            P.advantages = gspo["adv"]
            P.old_logprobs = (gspo["noise"][:rows] - 10.0).astype(np.float32)
            P.clip_eps_low, P.clip_eps_high = w.clip_eps_low, w.clip_eps_high
        t0 = time.perf_counter()
        oracle.forward_backward(P, nthreads=cores)
        return time.perf_counter() - t0

    probe = min(w.T, max(cores, 16))
    dt = run(probe)
    rows = int(min(w.T, max(probe, probe * seconds / max(dt, 1e-6))))
    rows = max(cores, rows - rows % cores) if rows >= cores else rows
    dt = run(rows)
    return rows * w.V / dt, cores, f"first {rows} of {w.T} rows (x {w.V} columns), fp64 forward+gradient, " \
                                   f"{cores} OpenMP threads, input generation excluded"


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import workloads
    w, x, u, targets, mask, n_glob, gspo = make_problem(workloads.get(args.workload), 0, 1)
    per_step = []
    for i in range(args.warmup + args.steps):
        v, cores, desc = oracle_sample_time(w, x, u, targets, mask, args.cpu_seconds / 4, gspo)
        if i >= args.warmup:
            per_step.append(v)
    value = statistics.median(per_step)
    elems = w.T * w.V
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elems / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Philox4x32-10 inputs)",
        "config": {"workload": w.name, "T": w.T, "V": w.V, "logits": w.dtype},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
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
    from lm_head_vocab_gb300 import LMLoss

    import workloads
    wl = workloads.get(args.workload)
    wl_full_T = wl.T
    if args.rows:
        wl = wl.with_shape(args.rows, wl.V)
    w, x, u, targets, mask, n_glob, gspo = make_problem(wl, rank, world)
    kw = call_kwargs(w, world, n_glob)

    def to_dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    logits = to_dev(x)
    teacher = to_dev(u)
    tg = torch.from_numpy(targets).to(dev)
    mk = None if mask is None else torch.from_numpy(mask).to(dev)
    h = LMLoss(dev.index, max_T=w.T, max_segments=gspo["S"] if gspo else 1)
    if args.cluster or args.threads or args.nbuf:
        h.set_launch_config(args.cluster, args.threads, args.nbuf)
    grad_mode = "inplace" if w.in_place else "new"
    gkw = {}
    if gspo is not None:
        # old log-probs for a timing run: this path's own log-probs plus the
        # seeded noise (the policy term's values do not change the work)
        a0, o0, k0 = h.build_args(logits, tg, mk, grad=None, want=("logp",))
        h.call(a0)
        torch.cuda.synchronize(dev)
        old = (o0.logp + torch.from_numpy(gspo["noise"]).to(dev)).contiguous()
        del a0, o0, k0
        gkw = dict(segment_ids=torch.from_numpy(gspo["seg"]).to(dev), num_segments=gspo["S"],
                   advantages=torch.from_numpy(gspo["adv"]).to(dev), old_logprobs=old)
    a, out, keep = h.build_args(logits, tg, mk, teacher_logits=teacher, grad=grad_mode, want=(), **gkw, **kw)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        h.call(a, stream)
    barrier()
    if h.device_error() != 0:
        raise SystemExit("device error during warm-up")
    info = h.call_info()

    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    # the K timed steps, with no events between a call's kernels (an event there
    # would cost a few microseconds a call and keep the reduction from launching
    # while the staged-row kernel finishes)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    ev0.record(stream)
    for _ in range(args.steps):
        h.call(a, stream)
    ev1.record(stream)
    barrier()
    step_ms = ev0.elapsed_time(ev1) / args.steps
    # then K more steps with events around the staged-row kernel of each call,
    # on the same stream: its average launch duration for the roofline
    h.set_timing(True)
    barrier()
    for _ in range(args.steps):
        h.call(a, stream)
    barrier()
    kern_total, kern_calls = h.kernel_time()
    h.set_timing(False)
    clk = clocks.stop()
    kern_ms = kern_total / max(kern_calls, 1)

    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([step_ms, kern_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms, kern_ms = float(t[0]), float(t[1])

    elems_rank = w.T * w.V
    value = world * elems_rank / (step_ms / 1e3)
    alg_bytes = w.algorithmic_bytes()
    peak, peak_kind = read_peaks()
    # the recorded traffic is per launch over the workload's full rows; a --rows
    # run moves the same bytes per row
    traffic = read_traffic(f"fused_kernel_{w.name}")
    if traffic is not None and w.T != wl_full_T:
        traffic = int(round(traffic * w.T / wl_full_T))
    achieved = alg_bytes / (kern_ms / 1e3) / 1e9

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        hx = torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x).pin_memory()
        ht = torch.from_numpy(targets).pin_memory()
        hu = None if u is None else torch.from_numpy(u.view(np.int16)).pin_memory()
        hm = None if mask is None else torch.from_numpy(mask).pin_memory()
        hloss = torch.empty(5, dtype=torch.float32).pin_memory()
        dl = logits.view(torch.int16) if logits.dtype == torch.bfloat16 else logits
        du = None if teacher is None else teacher.view(torch.int16)
        h2d = hx.numel() * hx.element_size() + ht.numel() * 8 + (0 if hu is None else hu.numel() * 2) \
            + (0 if hm is None else hm.numel())
        hg = None
        if gspo is not None:
            # the policy inputs travel too: segment ids, advantages, old log-probs
            hg = [(gkw["segment_ids"], torch.from_numpy(gspo["seg"]).pin_memory()),
                  (gkw["advantages"], torch.from_numpy(gspo["adv"]).pin_memory()),
                  (gkw["old_logprobs"], gkw["old_logprobs"].cpu().pin_memory())]
            h2d += sum(hs.numel() * hs.element_size() for _, hs in hg)

        def e2e_step():
            dl.copy_(hx, non_blocking=True)
            tg.copy_(ht, non_blocking=True)
            if hu is not None:
                du.copy_(hu, non_blocking=True)
            if hm is not None:
                mk.copy_(hm, non_blocking=True)
            if hg is not None:
                for dst, src in hg:
                    dst.copy_(src, non_blocking=True)
            h.call(a, stream)
            hloss.copy_(out.loss, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        barrier()
        e2e_ms = e0.elapsed_time(e1) / args.steps
        if world > 1:
            import torch.distributed as dist
            t = torch.tensor([e2e_ms], device=dev, dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_ms = float(t[0])
        e2e = {"value": world * elems_rank / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 20, "ms_per_step": e2e_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, cores, desc = oracle_sample_time(w, x, u, targets, mask, args.cpu_seconds, gspo)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded Philox4x32-10 inputs)",
            "config": {
                "workload": w.name, "T_per_gpu": w.T, "V": w.V, "logits": w.dtype,
                "reduction": kw["reduction"], "grad": grad_mode,
                "l2": f"inputs larger than L2 ({w.T * w.V * w.elem_bytes / 1e9:.2f} GB of logits per step)",
                "parallelism": f"rows x{world}" if world > 1 else "single GPU",
                "launch": {k: info[k] for k in ("cluster", "threads", "nbuf", "grid", "smem_bytes")},
            },
            "hbm_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s", "kernel_ms": kern_ms,
                         "algorithmic_bytes": alg_bytes},
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": int(info["launches"]) * args.steps,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    h.close()
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
