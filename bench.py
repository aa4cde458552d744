"""Benchmark of the packed CTC loss forward + backward on GB300.

One step is the loss and its gradient (upstream gradient 1) over the
large-vocabulary workload: 64 utterances, T ~ U[400,800] frames, D = 8193
classes, U ~ U[T/8, T/4] targets, bfloat16 log-softmax of N(0, 3^2) logits,
reduction none.  Its 638 MB of log probabilities exceed the 129 MB L2, so no
flush is needed between steps.  The headline step is one
``ctc_packed_forward`` + one ``ctc_packed_backward``; the same step as one
``ctc_packed_forward_backward`` call is timed beside it.

Prints ONE JSON line (rank 0): frames/s over the whole job, the roofline of
the whole path (algorithmic bytes per step over the step time, against the
measured HBM copy bandwidth) and of the backward call's gradient stream
(timed live with CUDA events on its stream), an end-to-end figure through
the C-ABI with host buffers (inputs copied in and the gradient copied back
every step), the SM clocks sampled during the timed region, and the fp64 CPU
oracle timed on a bounded sample on this host.

``--impl reference`` times the reference arm instead: the fp64 oracle, as it
stands, on the host cores, on a bounded sample of the same workload per step.
Under torchrun every rank runs its own replica of the workload (weak scaling,
no data-path collective).
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

METRIC = "packed CTC fwd+bwd frames/s and achieved HBM GB/s (% of GB300 peak)"
FALLBACK_HBM_GBS = 6800.0
# kernels of one step: prep, emission gather, chains, gradient stream (one more for logits input)
KERNELS_PER_STEP = 4
L2_BYTES = 129 * 2**20


def _profiled_traffic(workload, fused):
    """DRAM bytes of one step (every kernel of it) from the committed ncu
    summary of the launch, while the sources still match the ones profiled."""
    import hashlib
    import re

    if workload != "largevocab":
        return None
    name = "fused_largevocab.md" if fused else "two_call_largevocab.md"
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
    except OSError:
        return None
    t = re.search(r"traffic_bytes_per_step:\s*(\d+)", text)
    if not t:
        return None
    for fname, digest in re.findall(r"source_sha256_16 ([\w.]+): ([0-9a-f]{16})", text):
        try:
            src = open(os.path.join(ROOT, "packed_sequence_ctc_gb300", "csrc", fname), "rb").read()
        except OSError:
            return None
        if hashlib.sha256(src).hexdigest()[:16] != digest:
            return None
    return int(t.group(1))


def _load_workload(args, dev):
    """The named workload on `dev`; with --first N only its first N
    utterances (a smaller case of the same shapes, e.g. for an ncu capture)."""
    import workloads

    batch = workloads.workload(args.workload, device=dev)
    if args.first:
        batch = workloads.select_utterances(batch, list(range(min(args.first, batch.B))))
        batch.log_probs = batch.log_probs.to(dev)
    return batch


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="largevocab")
    p.add_argument("--first", type=int, default=0,
                   help="only the workload's first N utterances (a smaller case of the same shapes)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--input", default="log_probs", choices=["log_probs", "logits"],
                   help="logits: the rows are unnormalised logits and the path takes log_softmax itself")
    p.add_argument("--dtype", default=None, choices=["f64"],
                   help="f64: the workload's log probabilities in float64 through ctc_packed_forward_f64 / "
                        "ctc_packed_backward_f64 (the float64 path)")
    p.add_argument("--topology", default="ctc", choices=["ctc", "fsa"],
                   help="fsa: the same utterances' CTC lattices through the generic FSA path")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    p.add_argument("--path", default="two_call", choices=["fused", "two_call"],
                   help="the headline step: one forward-backward call, or a forward call then a backward call")
    return p.parse_args()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _workload_description(batch, flush=False):
    lengths = batch.lengths.tolist()
    tls = batch.target_lengths.tolist()
    dt = {"torch.float32": "fp32", "torch.bfloat16": "bf16", "torch.float16": "fp16"}[str(batch.log_probs.dtype)]
    return {
        "workload": f"{batch.name}: B={batch.B}, T_total={batch.T_total}, D={batch.D}, {dt} log probs, "
                    f"reduction={batch.reduction}",
        "B": batch.B,
        "T_total": batch.T_total,
        "frames": int(sum(lengths)),
        "D": batch.D,
        "io_dtype": dt,
        "max_target_len": batch.max_target_len,
        "target_len_range": [min(tls), max(tls)] if tls else [0, 0],
        "reduction": batch.reduction,
        "zero_infinity": batch.zero_infinity,
        "l2": (f"L2 flushed between timed steps ({batch.T_total * batch.D * batch.log_probs.element_size() / 1e6:.0f}"
               " MB of log probabilities fit in L2)") if flush else
              (f"inputs larger than L2 ({batch.T_total * batch.D * batch.log_probs.element_size() / 1e6:.0f} MB "
               "of log probabilities per step)"),
    }


def algorithmic_bytes(batch, logits=False):
    """Bytes the path must move: the forward's
    label-column gathers, the alpha store and reload (fp32), the full dense
    read of the log probabilities and write of the gradient; with logits
    input also the forward's dense read of the logits (the row
    log-sum-exp)."""
    e = batch.log_probs.element_size()
    D = batch.D
    gather = alpha = 0
    for T, U in zip(batch.lengths.tolist(), batch.target_lengths.tolist()):
        S = 2 * U + 1
        gather += T * min(U + 1, D) * e
        alpha += 2 * T * S * 4
    dense = 2 * batch.T_total * D * e
    grad_kernel = dense + alpha // 2  # the backward reads lp, writes grad, reloads the stored rows
    lse = batch.T_total * D * e if logits else 0
    return {"gather": gather, "alpha": alpha, "dense": dense, "lse": lse, "total": gather + alpha + dense + lse,
            "grad_kernel": grad_kernel}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_query_id):
        self.samples = []
        self.proc = None
        self.thread = None
        self.gpu = gpu_query_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu is not None:
            cmd += ["-i", str(self.gpu)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def snapshot(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits"]
        if self.gpu is not None:
            cmd += ["-i", str(self.gpu)]
        try:
            out = subprocess.run(cmd, capture_output=True, text=True, timeout=20).stdout.strip().splitlines()
            if out:
                self.samples.append((time.time(), out[0]))
        except Exception:
            pass

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 <= r[0] <= t1 + 0.3]
        use = inside or rows[-1:]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for _, p in use if num(p[1]) is not None]
        smax = [num(p[2]) for _, p in use if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in use for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use), "in_window": len(inside),
                "power_w_max": max([num(p[3]) for _, p in use if num(p[3]) is not None] or [0])}


def _gpu_query_id(torch, dev):
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


def cpu_baseline(batch, seconds, steps=1, warmup=0, logits=False):
    """Time the fp64 oracle (as it stands) on a bounded sample of utterances
    (its logits form when the rows are logits)."""
    import numpy as np

    import oracle
    import workloads

    def run(b, threads):
        if logits:
            return oracle.ctc_loss_packed_logits(b.log_probs, b.cu_seqlens, b.lengths, b.targets, b.target_lengths,
                                                 b.blank, b.zero_infinity, b.reduction, threads=threads)
        return oracle.oracle_batch(b, threads=threads)

    threads = oracle.max_threads()
    lengths = batch.lengths.tolist()
    # calibrate on two utterances, then take as many as fit the time budget
    probe = workloads.select_utterances(batch, [0, 1] if batch.B > 1 else [0])
    t = time.perf_counter()
    run(probe, 1)
    per_frame = (time.perf_counter() - t) / max(1, probe.frames)
    budget_frames = seconds * threads / max(per_frame, 1e-9)
    take, frames = [], 0
    for b in range(batch.B):
        if take and frames + lengths[b] > budget_frames:
            break
        take.append(b)
        frames += lengths[b]
    sample = workloads.select_utterances(batch, take)
    for _ in range(warmup):
        run(sample, threads)
    times = []
    for _ in range(steps):
        t = time.perf_counter()
        run(sample, threads)
        times.append(time.perf_counter() - t)
    dt = float(np.mean(times))
    return {"value": sample.frames / dt, "unit": "frames/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(take)} of {batch.B} utterances ({sample.frames} frames) of the same workload, "
                      f"fp64 {'log_softmax + ' if logits else ''}loss + gradient, OpenMP over utterances",
            "seconds_per_sample": dt}


def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch

    import workloads

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    batch = _load_workload(args, dev)
    batch.log_probs = batch.log_probs.cpu()
    logits = args.input == "logits"
    if logits:
        batch.log_probs = workloads.unnormalised_logits(batch, seed=17)
    # each step is a sample sized so that warmup + steps end within a few minutes
    per_step = max(1.0, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    base = cpu_baseline(batch, per_step, steps=args.steps, warmup=args.warmup, logits=logits)
    cfg = _workload_description(batch)
    cfg["input"] = args.input
    line = {
        "impl": "reference", "metric": METRIC, "value": base["value"], "unit": "frames/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": base["seconds_per_sample"] * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": cfg,
        "cpu_baseline": {k: base[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": base["value"], "unit": "frames/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def job_throughput(total_ms, steps, frames_per_rank, world, device="cpu"):
    """Whole-job throughput of a timed region: the slowest rank's time (a max
    over ranks when world > 1, so every rank must call this) and the frames
    of all ranks.  Returns (ms per step, frames per second)."""
    import torch
    import torch.distributed as dist

    if world > 1:
        tt = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms_per_step = total_ms / steps
    return ms_per_step, frames_per_rank * world / (ms_per_step / 1e3)


def _time_steps(torch, dev, stream, step, K, flush_buf=None, marks=1):
    """Times K steps on `stream` with CUDA events: returns (total ms, per-step
    intervals between the step's marks).  `step(k, ev)` enqueues step k and
    records ev[1..marks-1] between its parts."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(marks + 1)] for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    start.record(stream)
    for k in range(K):
        if flush_buf is not None:  # evict the inputs from L2; not part of the step's time
            with torch.cuda.stream(stream):
                flush_buf.fill_(float(k))
        ev[k][0].record(stream)
        step(k, ev[k])
        ev[k][marks].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    parts = [[ev[k][i].elapsed_time(ev[k][i + 1]) for i in range(marks)] for k in range(K)]
    total = sum(ev[k][0].elapsed_time(ev[k][marks]) for k in range(K)) if flush_buf is not None \
        else start.elapsed_time(end)
    return total, parts


def run_ours(args):
    import torch
    import torch.distributed as dist

    import packed_sequence_ctc_gb300 as pk
    import workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)

    batch = _load_workload(args, dev)
    logits = args.input == "logits"
    lp = batch.log_probs.contiguous()
    fflags = 0
    if logits:  # unnormalised rows: the forward takes their log_softmax itself
        lp = workloads.unnormalised_logits(batch, seed=17).to(dev).contiguous()
        fflags = pk.FLAG_LOGITS
    cu, ln, tg, tl = (x.to(dev) for x in (batch.cu_seqlens, batch.lengths, batch.targets, batch.target_lengths))
    B, T_total, D = batch.B, batch.T_total, batch.D
    mtl = batch.max_target_len
    red = batch.reduction
    ws = pk.Workspace(T_total, B, mtl, D, lp.dtype, dev).tensor
    nloss = B if red == "none" else 1
    loss = torch.empty(nloss, dtype=torch.float32, device=dev)
    g_up = torch.ones(nloss, dtype=torch.float32, device=dev)
    grad = torch.empty_like(lp)
    blank, zi = batch.blank, batch.zero_infinity

    def fused(k=None, ev=None):
        pk.ctc_packed_forward_backward(lp, cu, ln, tg, tl, blank, zi, red, g_up, loss, grad, ws, mtl, flags=fflags,
                                       stream=stream)

    def two_call(k=None, ev=None):
        pk.ctc_packed_forward(lp, cu, ln, tg, tl, blank, zi, red, loss, ws, mtl, flags=fflags, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        pk.ctc_packed_backward(lp, cu, ln, tg, tl, blank, zi, red, g_up, ws, grad, mtl, stream=stream)

    for _ in range(max(3, args.warmup)):
        fused()
        two_call()
    torch.cuda.synchronize(dev)
    status = pk.ctc_packed_read_status(ws)

    K = args.steps
    flush = lp.numel() * lp.element_size() < 2 * L2_BYTES
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    head, other = (fused, two_call) if args.path == "fused" else (two_call, fused)
    sampler = ClockSampler(_gpu_query_id(torch, dev))
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    total_ms, head_parts = _time_steps(torch, dev, stream, head, K, scrub, marks=1 if head is fused else 2)
    t1 = time.time()
    sampler.snapshot()
    if world > 1:
        dist.barrier()
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    # the other form of the step, timed the same way right after (not part of the headline)
    other_ms, other_parts = _time_steps(torch, dev, stream, other, K, scrub, marks=1 if other is fused else 2)
    status |= pk.ctc_packed_read_status(ws)

    ms_per_step, value = job_throughput(total_ms, K, batch.frames, world, dev)
    two_parts = head_parts if head is two_call else other_parts
    fwd_avg_ms = sum(p[0] for p in two_parts) / K
    bwd_avg_ms = sum(p[1] for p in two_parts) / K
    fused_ms = (total_ms if head is fused else other_ms) / K
    two_ms = (total_ms if head is two_call else other_ms) / K

    hbm_peak, peak_kind = _peaks()
    ab = algorithmic_bytes(batch, logits)
    path_gbs = ab["total"] / (ms_per_step / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "whole path: prep, emission gather, chains, gradient stream (" +
                ("one forward-backward call" if head is fused else "a forward call then a backward call") + ")",
                "achieved": round(path_gbs, 1), "peak": hbm_peak, "unit": "GB/s", "frac": round(path_gbs / hbm_peak, 4),
                "traffic": None if args.first else _profiled_traffic(args.workload, head is fused),
                "peak_kind": f"{peak_kind} copy bandwidth (burst)", "algorithmic_bytes_per_launch": ab["total"],
                "avg_launch_ms": round(ms_per_step, 5),
                "bytes": {k: ab[k] for k in ("gather", "alpha", "dense", "lse")}}
    stream_gbs = ab["grad_kernel"] / (bwd_avg_ms / 1e3) / 1e9
    backward_roofline = {"bound": "hbm", "kernel": "stream_kernel (the backward call alone: class sums and dense "
                         "gradient rows)", "achieved": round(stream_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(stream_gbs / hbm_peak, 4), "algorithmic_bytes_per_launch": ab["grad_kernel"],
                         "avg_launch_ms": round(bwd_avg_ms, 5)}
    paths = {"fused": {"ms_per_step": round(fused_ms, 5), "frames_per_s": round(batch.frames / (fused_ms / 1e3), 1),
                       "hbm_frac": round(ab["total"] / (fused_ms / 1e3) / 1e9 / hbm_peak, 4),
                       "call": "ctc_packed_forward_backward"},
             "two_call": {"ms_per_step": round(two_ms, 5), "frames_per_s": round(batch.frames / (two_ms / 1e3), 1),
                          "hbm_frac": round(ab["total"] / (two_ms / 1e3) / 1e9 / hbm_peak, 4),
                          "forward_ms": round(fwd_avg_ms, 5), "backward_ms": round(bwd_avg_ms, 5),
                          "call": "ctc_packed_forward + ctc_packed_backward"}}

    e2e = None
    if not args.no_e2e:
        e2e = _e2e(args, pk, torch, batch, dev, stream, lp, ws, mtl, red, nloss, world, fflags, head is fused)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        batch.log_probs = lp.cpu()
        base = cpu_baseline(batch, args.cpu_seconds, logits=logits)
        cpu = {k: base[k] for k in ("value", "unit", "cores", "kind", "sample")}

    if rank == 0:
        dt = {"fp32": "f32", "bf16": "f32", "fp16": "f32"}
        cfg = _workload_description(batch, flush)
        cfg["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
        cfg["input"] = args.input
        cfg["step"] = paths[args.path]["call"]
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "frames/s", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dt[cfg["io_dtype"]], "data": "synthetic",
            "config": cfg, "hbm_gbs": round(path_gbs, 1), "roofline": roofline,
            "backward_roofline": backward_roofline, "paths": paths,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": (KERNELS_PER_STEP + (1 if logits else 0)) * K,
            "clocks": clocks, "device_status": status,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _e2e(args, pk, torch, batch, dev, stream, lp, ws, mtl, red, nloss, world, fflags=0, fused=True):
    """Same metric through the C-ABI from and to pinned host buffers: every
    step copies its inputs host->device, computes the loss and the gradient,
    and copies the loss and the whole gradient device->host.  Inputs and
    gradients alternate between two device buffers, so step i+1's input copy
    and step i-1's gradient copy (each on its own copy stream) overlap step
    i's compute."""
    host = {
        "lp": lp.cpu().pin_memory(),
        "cu": batch.cu_seqlens.pin_memory(),
        "ln": batch.lengths.pin_memory(),
        "tg": batch.targets.pin_memory(),
        "tl": batch.target_lengths.pin_memory(),
    }
    bufs = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    grads = [torch.empty_like(lp) for _ in range(2)]
    losses = [torch.empty(nloss, dtype=torch.float32, device=dev) for _ in range(2)]
    grad_host = torch.empty(lp.shape, dtype=lp.dtype).pin_memory()
    loss_host = torch.empty(nloss, dtype=torch.float32).pin_memory()
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    inputs_free = [torch.cuda.Event() for _ in range(2)]
    grad_free = [torch.cuda.Event() for _ in range(2)]
    for j in range(2):
        inputs_free[j].record(stream)
        grad_free[j].record(stream)
    g_up = torch.ones(nloss, dtype=torch.float32, device=dev)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = grad_host.numel() * grad_host.element_size() + loss_host.numel() * 4

    def step(i):
        j = i % 2
        d = bufs[j]
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(inputs_free[j])
            for k in host:
                d[k].copy_(host[k], non_blocking=True)
            copied[j].record(h2d_stream)
        stream.wait_event(copied[j])
        stream.wait_event(grad_free[j])
        if fused:
            pk.ctc_packed_forward_backward(d["lp"], d["cu"], d["ln"], d["tg"], d["tl"], batch.blank,
                                           batch.zero_infinity, red, g_up, losses[j], grads[j], ws, mtl,
                                           flags=fflags, stream=stream)
        else:
            pk.ctc_packed_forward(d["lp"], d["cu"], d["ln"], d["tg"], d["tl"], batch.blank, batch.zero_infinity, red,
                                  losses[j], ws, mtl, flags=fflags, stream=stream)
            pk.ctc_packed_backward(d["lp"], d["cu"], d["ln"], d["tg"], d["tl"], batch.blank, batch.zero_infinity,
                                   red, g_up, ws, grads[j], mtl, stream=stream)
        inputs_free[j].record(stream)
        computed[j].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(computed[j])
            loss_host.copy_(losses[j], non_blocking=True)
            grad_host.copy_(grads[j], non_blocking=True)
            grad_free[j].record(d2h_stream)

    for i in range(3):
        step(i)
    torch.cuda.synchronize(dev)
    K = max(3, min(args.steps, 60))
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(h2d_stream)  # the first timed input copy starts after this
    stream.wait_event(s)
    d2h_stream.wait_event(s)
    for i in range(K):
        step(i)
    stream.wait_event(grad_free[(K - 1) % 2])  # the last gradient has reached the host
    e.record(stream)
    torch.cuda.synchronize(dev)
    ms = s.elapsed_time(e) / K
    return {"value": round(batch.frames * world / (ms / 1e3), 1), "unit": "frames/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4), "steps": K,
            "call": "ctc_packed_forward_backward" if fused else "ctc_packed_forward + ctc_packed_backward",
            "overlap": "inputs and gradients alternate between two device buffers: each step's host-to-device "
                       "input copy and device-to-host gradient copy run on their own copy streams beside the "
                       "neighbouring steps' compute"}


def run_fsa(args):
    """The workload's CTC lattices as FSA edge lists through the generic FSA
    path (ctc_packed_fsa_forward + ctc_packed_fsa_backward), timed like the
    CTC path; one JSON line."""
    import numpy as np
    import torch

    import packed_sequence_ctc_gb300 as pk
    import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    batch = _load_workload(args, dev)
    lp = batch.log_probs.contiguous()
    offs = np.concatenate([[0], np.cumsum(batch.target_lengths.cpu().numpy())])
    tg = batch.targets.cpu().numpy()
    fsa_h = workloads.pack_fsas([workloads.ctc_lattice_fsa(tg[offs[b]:offs[b + 1]], batch.blank)
                                 for b in range(batch.B)])
    fsa = tuple(x.to(dev).contiguous() for x in fsa_h)
    so = fsa_h[0]
    max_states = int((so[1:] - so[:-1]).max())
    eo_h, ed_h = fsa_h[3], fsa_h[4]
    max_labels = max(1, max(len(set(ed_h[eo_h[i]:eo_h[i + 1], 2].tolist())) for i in range(batch.B)))
    cu, ln = batch.cu_seqlens.to(dev).to(torch.int32), batch.lengths.to(dev).to(torch.int32)
    T_total, D = lp.shape
    ws = torch.empty(pk.ctc_packed_fsa_workspace_size(T_total, batch.B, int(fsa_h[1].numel()), int(fsa_h[4].shape[0]),
                                                      max_states, max_labels, D), dtype=torch.uint8,
                     device=dev)
    loss = torch.empty(batch.B, device=dev)
    g_up = torch.ones(batch.B, device=dev)
    grad = torch.empty_like(lp)
    zi = batch.zero_infinity

    def fwd():
        pk.ctc_packed_fsa_forward(lp, cu, ln, fsa, max_states, max_labels, zi, loss, ws, stream=stream)

    def bwd():
        pk.ctc_packed_fsa_backward(lp, cu, ln, fsa, max_states, max_labels, zi, g_up, ws, grad, stream=stream)

    for _ in range(max(3, args.warmup)):
        fwd()
        bwd()
    torch.cuda.synchronize(dev)
    status = pk.ctc_packed_read_status(ws)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(_gpu_query_id(torch, dev))
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for k in range(K):
        ev[k][0].record(stream)
        fwd()
        ev[k][1].record(stream)
        bwd()
        ev[k][2].record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    sampler.snapshot()
    time.sleep(0.25)
    sampler.stop()
    fwd_ms = sum(ev[k][0].elapsed_time(ev[k][1]) for k in range(K)) / K
    bwd_ms = sum(ev[k][1].elapsed_time(ev[k][2]) for k in range(K)) / K
    ms = fwd_ms + bwd_ms
    hbm_peak, peak_kind = _peaks()
    e = lp.element_size()
    dense = 2 * T_total * D * e  # the backward reads the rows and writes the gradient
    achieved = dense / (bwd_ms / 1e3) / 1e9
    cfg = _workload_description(batch, False)
    cfg["topology"] = f"fsa: CTC lattices as edge lists ({int(fsa_h[4].shape[0])} edges, up to {max_states} states)"
    cfg["parallelism"] = "single GPU"
    line = {
        "metric": METRIC, "value": round(batch.frames / (ms / 1e3), 1), "unit": "frames/s", "n_gpus": 1,
        "steps": K, "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfg,
        "roofline": {"bound": "hbm", "kernel": "fsa_post_kernel+grad_kernel (the FSA backward call)",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": None,
                     "peak_kind": f"{peak_kind} copy bandwidth (burst)", "algorithmic_bytes_per_launch": dense,
                     "avg_launch_ms": round(bwd_ms, 5)},
        "forward_ms": round(fwd_ms, 5), "backward_ms": round(bwd_ms, 5), "cpu_baseline": None, "e2e": None,
        "gpu_launches": 4 * K, "clocks": sampler.summary(t0, t1), "device_status": status,
    }
    print(json.dumps(line), flush=True)


def run_f64(args):
    """The workload's rows in float64 through the float64 path
    (ctc_packed_forward_f64 + ctc_packed_backward_f64), timed like the CTC
    path; one JSON line.  The dense rows are twice the bytes of the float32
    path; the recursions run in float64 (extended range)."""
    import torch

    import packed_sequence_ctc_gb300 as pk
    import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    batch = _load_workload(args, dev)
    cfg = _workload_description(batch, False)
    lp = batch.log_probs.to(torch.float64).contiguous()
    batch.log_probs = None
    T_total, D = lp.shape
    cu, ln = batch.cu_seqlens.to(dev).to(torch.int32), batch.lengths.to(dev).to(torch.int32)
    tg, tl = batch.targets.to(dev).to(torch.int32), batch.target_lengths.to(dev).to(torch.int32)
    mtl = batch.max_target_len
    ws = pk.Workspace(T_total, batch.B, mtl, D, torch.float64, dev).tensor
    red = batch.reduction
    loss = torch.empty(batch.B if red == "none" else 1, dtype=torch.float64, device=dev)
    g_up = torch.ones(batch.B if red == "none" else 1, dtype=torch.float64, device=dev)
    grad = torch.empty_like(lp)
    zi = batch.zero_infinity

    def fwd():
        pk.ctc_packed_forward(lp, cu, ln, tg, tl, batch.blank, zi, red, loss, ws, mtl, stream=stream)

    def bwd():
        pk.ctc_packed_backward(lp, cu, ln, tg, tl, batch.blank, zi, red, g_up, ws, grad, mtl, stream=stream)

    for _ in range(max(3, args.warmup)):
        fwd()
        bwd()
    torch.cuda.synchronize(dev)
    status = pk.ctc_packed_read_status(ws)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(_gpu_query_id(torch, dev))
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for k in range(K):
        ev[k][0].record(stream)
        fwd()
        ev[k][1].record(stream)
        bwd()
        ev[k][2].record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    sampler.snapshot()
    time.sleep(0.25)
    sampler.stop()
    fwd_ms = sum(ev[k][0].elapsed_time(ev[k][1]) for k in range(K)) / K
    bwd_ms = sum(ev[k][1].elapsed_time(ev[k][2]) for k in range(K)) / K
    ms = fwd_ms + bwd_ms
    hbm_peak, peak_kind = _peaks()
    dense = 2 * T_total * D * 8  # the backward reads the rows and writes the gradient
    achieved = dense / (bwd_ms / 1e3) / 1e9
    cfg["workload"] = cfg["workload"].replace(cfg["io_dtype"] + " log probs", "f64 log probs")
    cfg["io_dtype"] = "f64"
    cfg["l2"] = f"inputs larger than L2 ({T_total * D * 8 / 1e6:.0f} MB of log probabilities per step)"
    cfg["parallelism"] = "single GPU"
    line = {
        "metric": METRIC, "value": round(batch.frames / (ms / 1e3), 1), "unit": "frames/s", "n_gpus": 1,
        "steps": K, "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
        "roofline": {"bound": "hbm", "kernel": "f64_post_kernel+f64_grad_kernel (the float64 backward call)",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": None,
                     "peak_kind": f"{peak_kind} copy bandwidth (burst)", "algorithmic_bytes_per_launch": dense,
                     "avg_launch_ms": round(bwd_ms, 5)},
        "forward_ms": round(fwd_ms, 5), "backward_ms": round(bwd_ms, 5), "cpu_baseline": None, "e2e": None,
        "gpu_launches": (4 + (1 if red != "none" else 0)) * K, "clocks": sampler.summary(t0, t1),
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


def main():
    args = _args()
    if args.impl == "reference":
        run_reference(args)
    elif args.dtype == "f64":
        run_f64(args)
    elif args.topology == "fsa":
        run_fsa(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
