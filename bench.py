"""Benchmark of the ZeRO partitioned optimizer step of one data-parallel rank.

Metric: parameters updated per second (and achieved HBM GB/s against the
measured GB300 copy bandwidth), 1 GPU per rank.  Default workload: the 7.5B
model of the ZeRO Stage-3 memory table, Nd = 64, bf16 gradients, rank 0's
shard of 117,187,500 parameters, fusion bucket 5e8 (one bucket); 64 gradient
contributions (15 GB) resident in HBM.

A step = the whole hot path: the fused reduce + AdamW + cast kernel over the
shard, the read of the nonfinite flag, and the commit (or global skip).  Each
step moves 18 GB, far more than the 129 MB L2, so no L2 flush is needed
between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c4]
    python bench.py --impl reference     # the CPU oracle on a bounded sample

Under torchrun (N > 1) every process runs its own rank's shard (weak scaling;
the only collective is the one-word OR of the skip flag) and rank 0 prints
the max-over-ranks time.
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
sys.path.insert(0, ROOT)

METRIC = "ZeRO shard step: params updated/s and HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "params/s"
KERNEL_SRCS = [os.path.join(ROOT, "zero_sharded_optimizer_02_gb300", "csrc", f)
               for f in ("zero_ring.cuh", "zero_device.cuh")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "k_step_fused_traffic.txt")
NOMINAL_HBM_GBS = 7900.0
L2_BYTES = 129e6
# Row pitch of the emulated gradient rows and state rows, in elements: a
# multiple of 512 puts every row of the 2-byte gradients on a 1 KB boundary.
# With the 7.5B shard's 117,187,504-element pitch (rows 32-byte aligned) the
# step ran 1.5% slower and the read-only pass 3.9% slower than with any
# 1 KB-aligned pitch; shards whose rows were already 128-byte aligned ran the
# same either way.
ROW_ALIGN = 512


def host_available_gb():
    """MemAvailable of this host in GB (None if it cannot be read)."""
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    return int(ln.split()[1]) * 1024 / 1e9
    except (OSError, ValueError, IndexError):
        pass
    return None


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


# Elements a SM covers in one wave of the short-window kernel (3 CTAs of 256
# threads, 4 elements a thread): by default the library runs a launch window
# of at most SMs times this on that kernel instead of the ring.
SMALL_WAVE_ELEMS_PER_SM = 3 * 256 * 4


def kernel_name(shard_elems: int = None) -> str:
    """The fused-step kernel the run uses: ZERO_FUSED_VARIANT if set, else the
    build's ZERO_FUSED_IMPL (0 registers, 1 cp.async ring (default), 2 bulk
    copies), the default ring giving a shard of at most SMs x 3,072 elements
    (one window) to the short-window kernel."""
    import re
    names = {0: "k_step_fused", 1: "k_step_fused_ring", 2: "k_step_fused_tma",
             3: "k_step_fused_small"}
    v = os.environ.get("ZERO_FUSED_VARIANT")
    if v in ("registers", "ring", "tma", "small"):
        return names[{"registers": 0, "ring": 1, "tma": 2, "small": 3}[v]]
    flags = os.environ.get("ZERO_NVCC_FLAGS", "")
    m = re.search(r"ZERO_FUSED_IMPL=(\d)", flags)
    impl = int(m.group(1)) if m else 1
    if impl == 1 and "ZERO_SMALL_WINDOWS=0" not in flags and shard_elems is not None:
        import torch
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        if shard_elems <= sms * SMALL_WAVE_ELEMS_PER_SM:
            return names[3]
    return names.get(impl, "k_step_fused_ring")


def kernel_source_hash() -> str:
    """Hash of the code (comments and whitespace removed) of the sources the
    default fused kernel is compiled from (its header and the shared device
    helpers): any change of the kernel's code changes it; host launch code
    does not."""
    import re
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, shard_elems: int):
    """DRAM bytes per parameter of the fused kernel from the committed ncu
    summary, if it was taken on the current kernel source for this workload."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for ln in f:
                if ":" in ln and not ln.startswith("#"):
                    k, v = ln.split(":", 1)
                    kv[k.strip()] = v.strip()
    except OSError:
        return None
    if kv.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    if kv.get("build_flags", "") != os.environ.get("ZERO_NVCC_FLAGS", ""):
        return None
    if kernel_name(shard_elems) != "k_step_fused_ring":   # recorded for the ring kernel
        return None
    v = kv.get(f"dram_bytes_per_param.{workload}")
    return None if v is None else float(v)


def workload(args):
    """The named workload, with optional --psi / --grad-dtype overrides (for
    experiments; the benchmark line uses the named workload as it is)."""
    import dataclasses

    import synth
    w = synth.WORKLOADS[args.config]
    if args.psi:
        w = dataclasses.replace(w, psi=args.psi, plant=None)
    if args.nd:
        w = dataclasses.replace(w, nd=args.nd, plant=None)
    if args.bucket:
        w = dataclasses.replace(w, bucket=args.bucket)
    if args.grad_dtype and args.grad_dtype != w.grad_dtype:
        w = dataclasses.replace(w, grad_dtype=args.grad_dtype,
                                loss_scale=1024.0 if args.grad_dtype == "f16" else 1.0)
    return w


def bench_config(args, w, dp_rank: int, world: int) -> dict:
    """The workload description both arms print (host arithmetic only): the
    shard this process runs, its row layout and where its parameters go."""
    import synth
    s, begin, n = synth.shard_of(w.psi, w.nd, dp_rank)
    pitch = synth.pitch_of(s, ROW_ALIGN)
    step_bytes = w.bytes_per_param * n
    overridden = bool(args.psi or args.nd or args.grad_dtype or args.bucket)
    return {"workload": f"{args.config}: {w.title}" + (" (overridden)" if overridden else ""),
            "psi": w.psi, "nd": w.nd,
            "rank": dp_rank, "shard_params": n, "grad_dtype": w.grad_dtype,
            "bucket": w.bucket, "loss_scale": w.loss_scale,
            "row_stride_elems": pitch + args.row_pad,
            "gathered": args.gathered + (
                f" (slot at element {begin}, 16-byte phase {(begin * 2) % 16} B)"
                if args.gathered == "full" else " (the rank's own S-element buffer)"),
            "l2": (f"inputs larger than L2 ({step_bytes / 1e9:.1f} GB per step), no flush"
                   if step_bytes > L2_BYTES else
                   f"inputs L2-resident ({step_bytes / 1e6:.1f} MB per step, L2 129 MB), no "
                   "flush: a latency figure, not a bandwidth one"),
            "parallelism": f"zero-dp{w.nd} emulated, {world} process(es)"}


def time_back_to_back(torch, stream, dev, call, reps: int) -> float:
    """Milliseconds per call of `reps` back-to-back calls, CUDA events on
    `stream` (synchronised on both sides)."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps


def time_graph(torch, stream, dev, call, steps: int, reps: int = 5) -> float:
    """Milliseconds per call of `steps` calls captured once as a CUDA graph on
    `stream` and replayed `reps` times, CUDA events on `stream`: the GPU's
    time for the calls with no host issue time between them.  The calls'
    arguments are frozen at capture, so the replays repeat the same steps;
    the driver's bookkeeping (its step count, its current buffers) no longer
    matches the data afterwards."""
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for _ in range(steps):
            call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / (reps * steps)
    del g
    return ms


# The other workloads the default line also times (kernel time only): the
# 1.5B shard is the second target workload; rank 1 of the 1.5B and 7.5B
# shards writes its parameters into its slot of the flat Nd*S buffer, 8 bytes
# off a 16-byte line (S mod 8 = 4), so its cast runs with 8-byte stores.
PER_CONFIG = [("c0", 0, "slot"), ("c1", 0, "slot"), ("c2", 0, "slot"), ("c3", 0, "slot"),
              ("c3", 1, "full"), ("c4", 1, "full")]


def measure_config(key: str, rank: int, gathered: str, dev, stream, peak: float,
                   reps: int = 100) -> dict:
    """The fused step of one more workload's shard (shard-view rows resident
    in HBM), timed like the headline's kernel figure: `reps` back-to-back
    steps, each step's output feeding the next, CUDA events on the launching
    stream.  Checks that no step was skipped."""
    import torch

    import synth
    from zero_sharded_optimizer_02_gb300 import _abi
    from zero_sharded_optimizer_02_gb300.step import DataParallelStep
    w = synth.WORKLOADS[key]
    with torch.cuda.stream(stream):
        dps = DataParallelStep(w.psi, w.nd, [rank], w.grad_dtype, w.hparams, w.loss_scale,
                               w.bucket, dev, gathered=gathered, fused=True, stream=stream,
                               row_align=ROW_ALIGN)
        L = dps.layouts[rank]
        n, pitch = int(L.length), int(L.row_pitch)
        st = dps.state[rank]
        for row, which in zip(st.bufs[st.cur], ("master", "m", "v")):
            synth.fill_shard_state(w, rank, which, row)
        grads = torch.empty(w.nd, pitch, dtype=w.torch_grad_dtype, device=dev)
        synth.fill_shard_rows(w, 0, rank, grads)
    desc = {rank: _abi.grads(grads, pitch, 0, w.nd, w.grad_dtype)}

    def call():
        dps.launch(desc)
        dps.commit(False)
    for _ in range(3):
        call()
    ms = time_back_to_back(torch, stream, dev, call, reps)
    torch.cuda.synchronize(dev)
    skipped = int(dps.flag.item()) != 0
    launches = _abi.fused_launch_count(n, w.bucket, 0)
    step_bytes = w.bytes_per_param * n
    gbs = step_bytes / (ms * 1e-3) / 1e9
    out = {"workload": f"{key}: {w.title}", "rank": rank, "nd": w.nd, "shard_params": n,
           "grad_dtype": w.grad_dtype,
           "gathered": gathered + (f" (slot at element {int(L.begin)}, 16-byte phase "
                                   f"{(int(L.begin) * 2) % 16} B)" if gathered == "full" else ""),
           "kernel": kernel_name(n), "kernel_ms_per_step": ms, "launches_per_step": launches,
           "kernel_ms": ms / launches, "algorithmic_bytes_per_param": w.bytes_per_param,
           "achieved": gbs, "frac": gbs / peak, "params_per_s": n / (ms * 1e-3),
           "steps_timed_back_to_back": reps, "skipped": skipped}
    if step_bytes <= L2_BYTES:
        out["l2"] = (f"L2-resident ({step_bytes / 1e6:.1f} MB per step): a latency figure, not "
                     "a bandwidth one")
        # Such a short step is issued slower than it runs: time its kernels
        # without the host's issue time too, as one CUDA graph of the same
        # back-to-back steps (the last measurement on this driver).
        try:
            gms = time_graph(torch, stream, dev, call, reps)
        except Exception as e:         # a capture this torch build refuses: no figure
            out["graph"] = f"unavailable: {str(e).splitlines()[0][:200]}"
        else:
            gbs_graph = step_bytes / (gms * 1e-3) / 1e9
            out["kernel_ms_per_step_graph"] = gms
            out["achieved_graph"] = gbs_graph
            out["frac_graph"] = gbs_graph / peak
    del dps, grads
    torch.cuda.empty_cache()
    return out


def smi_index(local: int) -> str:
    """nvidia-smi's id of this process's device (honours CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) over a window."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        rows = [r for (ts, r) in self.rows if t0 - 0.15 <= ts <= t1 + 0.15 and len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args) -> None:
    import torch
    import torch.distributed as dist

    import synth
    from zero_sharded_optimizer_02_gb300 import build
    from zero_sharded_optimizer_02_gb300.step import (DataParallelStep, PipelinedStep,
                                                      data_parallel_rank, max_over_ranks,
                                                      sum_over_ranks)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    # One process per GPU over NCCL.  ZERO_DIST_BACKEND=gloo runs the same
    # choreography with host collectives, and then processes may share a GPU
    # (no kernel of this path waits on another process's kernels).
    backend = os.environ.get("ZERO_DIST_BACKEND", "nccl")
    gpu = local % torch.cuda.device_count() if backend == "gloo" else local
    if world > 1:
        if backend == "nccl":
            dist.init_process_group("nccl", device_id=torch.device("cuda", gpu))
        else:
            dist.init_process_group(backend)
    torch.cuda.set_device(gpu)
    dev = torch.device("cuda", gpu)
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
        build.build()          # every rank loads the library (already built)

    w = workload(args)
    dp_rank = data_parallel_rank(args.rank, rank, w.nd)
    group = dist.group.WORLD if world > 1 else None
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        dps = DataParallelStep(w.psi, w.nd, [dp_rank], w.grad_dtype, w.hparams, w.loss_scale,
                               w.bucket, dev, gathered=args.gathered, fused=True,
                               process_group=group, stream=stream, row_align=ROW_ALIGN)
        L = dps.layouts[dp_rank]
        n = int(L.length)
        pitch = int(L.row_pitch)
        st = dps.state[dp_rank]
        for row, which in zip(st.bufs[st.cur], ("master", "m", "v")):
            synth.fill_shard_state(w, dp_rank, which, row)
        row_stride = pitch + args.row_pad
        grads = torch.empty(w.nd, row_stride, dtype=w.torch_grad_dtype, device=dev)
        synth.fill_shard_rows(w, 0, dp_rank, grads)
        from zero_sharded_optimizer_02_gb300 import _abi
        desc = {dp_rank: _abi.grads(grads, row_stride, 0, w.nd, w.grad_dtype)}
        pipe = PipelinedStep(w.psi, w.nd, [dp_rank], w.grad_dtype, w.hparams, w.loss_scale,
                             w.bucket, dev, gathered=args.gathered, process_group=group,
                             stream=stream, row_align=ROW_ALIGN)
        pipe.state[dp_rank].bufs[0].copy_(st.bufs[st.cur])
    torch.cuda.synchronize(dev)

    # -- warm-up, then K timed steps.  The pipelined driver launches up to two
    #    steps ahead of the oldest undecided step's flag read (a skip re-runs
    #    the speculative steps), so the GPU never waits for the host; every
    #    step is the whole path: fused kernels, flag read, commit or global
    #    skip. -----------------------------------------------------------------
    for _ in range(args.warmup):
        pipe.launch(desc)
    pipe.finish()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(smi_index(gpu)) if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launched0 = pipe.kernel_launches
    wall0 = time.time()
    t_start.record(stream)
    decided = []
    for k in range(args.steps):
        decided += pipe.launch(desc)
    decided += pipe.finish()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    if world > 1:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    launches = sum_over_ranks(pipe.kernel_launches - launched0, group, dev)   # whole job
    skipped = sum(decided)
    assert len(decided) == args.steps

    # -- the same steps with the synchronous driver (flag read before the next
    #    launch), for comparison; per-launch events inside its steps ----------
    for _ in range(args.warmup):
        dps.step(desc)
    nsync = max(1, min(args.steps, 100))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(nsync)]
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    s0.record(stream)
    for k in range(nsync):
        ev[k][0].record(stream)
        dps.launch(desc)
        ev[k][1].record(stream)
        dps.commit(dps.decide())
    s1.record(stream)
    torch.cuda.synchronize(dev)
    sync_ms = max_over_ranks(s0.elapsed_time(s1) / nsync, group, dev)
    kernel_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(total_ms, group, dev)

    # -- the fused kernel alone: back-to-back steps' launches (no flag read
    #    between them; each step's output is the next one's input, as in real
    #    steps), timed with events on the launching stream; this removes the
    #    host launch gap that the per-step events above include -----------------
    nk = max(1, min(args.steps, 100))
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    k0.record(stream)
    for _ in range(nk):
        dps.launch(desc)
        dps.commit(False)          # swap the buffers without reading the flag
    k1.record(stream)
    torch.cuda.synchronize(dev)
    back_to_back_ms = k0.elapsed_time(k1) / nk
    # -- a read-only stream over the same rows: the nonfinite pre-check reads
    #    the Nd contribution rows (2 Nd B/param) and writes nothing, in the
    #    same launch windows.  The step is 2 Nd + 12 B read to 14 B written
    #    a parameter; a pure read is the best stream HBM gives that mix, so
    #    the step's fraction of it shows how much is left. --------------------
    def read_pass():
        _abi.zero_check_nonfinite(desc[dp_rank], 0, n, dps.flag, stream)
    for _ in range(3):
        read_pass()
    read_ms = time_back_to_back(torch, stream, dev, read_pass, nk)
    read_gbs = 2 * w.nd * n / (read_ms * 1e-3) / 1e9
    with torch.cuda.stream(stream):
        dps.flag.zero_()
    time.sleep(0.2 if sampler else 0.0)
    clocks = None
    if sampler:
        sampler.stop()
        clocks = sampler.summary(wall0, wall1)

    # -- end to end through host buffers.  Every step: the step's gradients
    #    enter from pinned host memory, the step runs, the new parameters and
    #    the flag come back.  The gradients are fed in transfer buckets by
    #    zero_feed_buckets on a copy stream while the bucket-ready kernel
    #    (zero_step_shard_streamed) runs the optimizer on the buckets that have
    #    landed; results do not depend on the bucket size.  The plain
    #    sequential form (copy everything, then step) is timed beside it. -----
    e2e = None
    if args.e2e_steps > 0:
        # the step's gradients in page-locked host memory (each rank its own);
        # every rank must have them, or no rank runs the end-to-end leg
        pin_gb = (grads.numel() + 3 * n) * grads.element_size() / 1e9
        # every process of this node pins as much at once: leave at least half
        # of the host's available memory to everything else
        local_world = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
        avail_gb = host_available_gb()
        if world > 1:
            dist.barrier()
        host_grads = host_params = None
        if avail_gb is not None and local_world * pin_gb > 0.5 * avail_gb:
            pin_error = (f"{local_world} x {pin_gb:.1f} GB would exceed half of the host's "
                         f"{avail_gb:.0f} GB available")
        else:
            try:
                host_grads = torch.empty(grads.shape, dtype=grads.dtype, pin_memory=True)
                host_grads.copy_(grads)
                host_params = torch.empty(n, dtype=grads.dtype, pin_memory=True)
                pin_error = ""
            except RuntimeError as err:
                host_grads = host_params = None
                pin_error = str(err).splitlines()[0][:160] if str(err) else type(err).__name__
        pinned_everywhere = -max_over_ranks(-float(not pin_error), group, dev) > 0.5
        if not pinned_everywhere:
            e2e = {"unavailable": f"could not pin {pin_gb:.1f} GB of host memory on every rank"
                                  + (f" ({pin_error})" if pin_error else "")}
            host_grads = host_params = None
        else:
            copy_stream = torch.cuda.Stream(dev)
            stream_bucket = max(8, -(-(-(-n // args.e2e_buckets)) // 8) * 8)
            slot0 = int(L.begin) if args.gathered == "full" else 0   # the rank's parameters

            gview = dps.gathered_view(dp_rank)

            def read_back():
                with torch.cuda.stream(stream):
                    host_params.copy_(gview[slot0:slot0 + n], non_blocking=True)
                stream.synchronize()

            fed_timeouts = []

            def host_fed():
                dps.launch_host_fed(dp_rank, host_grads, desc[dp_rank], stream_bucket, copy_stream)
                try:
                    skipped = dps.decide()
                except _abi.ZeroError as err:     # a bucket never arrived within the wait
                    if err.status != _abi.ZERO_ERR_TIMEOUT:
                        raise
                    fed_timeouts.append(1)
                    return
                dps.commit(skipped)
                read_back()

            def sequential():
                with torch.cuda.stream(stream):
                    grads.copy_(host_grads, non_blocking=True)
                dps.step(desc)
                read_back()

            host_desc = {dp_rank: _abi.grads(host_grads, row_stride, 0, w.nd, w.grad_dtype)}

            def zero_copy_read_back():   # the kernels read the gradients in host memory
                dps.step(host_desc)
                read_back()

            # the same step with its gathered slot in pinned host memory: the
            # kernels also write the new parameters in place over the host
            # link, so they are on the host when the step's flag is read
            dps_h = DataParallelStep(w.psi, w.nd, [dp_rank], w.grad_dtype, w.hparams,
                                     w.loss_scale, w.bucket, dev, gathered="slot", fused=True,
                                     process_group=group, stream=stream, gathered_on_host=True,
                                     row_align=ROW_ALIGN)
            with torch.cuda.stream(stream):
                dps_h.state[dp_rank].bufs[0].copy_(dps.state[dp_rank].bufs[dps.state[dp_rank].cur])
            dps_h.t = dps.t

            def zero_copy():
                dps_h.step(host_desc)

            def copies_alone():   # the host link alone: the same bytes, no step
                with torch.cuda.stream(stream):
                    grads.copy_(host_grads, non_blocking=True)
                read_back()

            # The three forms run interleaved, one of each per iteration, so that
            # they see the same host-memory conditions (the host is shared); the
            # first iteration is untimed.  Each is timed on the host around the
            # whole call, its final synchronisation included.
            forms = {"fed": host_fed, "sequential": sequential, "zero_copy": zero_copy,
                     "zero_copy_read_back": zero_copy_read_back, "copies": copies_alone}
            times = {k: [] for k in forms}
            for it in range(args.e2e_steps + 1):
                for k, fn in forms.items():
                    if world > 1:
                        dist.barrier()
                    torch.cuda.synchronize(dev)
                    t0 = time.perf_counter()
                    fn()
                    if it:
                        times[k].append((time.perf_counter() - t0) * 1e3)
            mean = {k: max_over_ranks(statistics.fmean(v), group, dev) for k, v in times.items()}
            best = {k: max_over_ranks(min(v), group, dev) for k, v in times.items()}
            grad_bytes = w.nd * n * host_grads.element_size()
            nbk = -(-n // stream_bucket)

            def form(k, path, h2d):
                return {"ms_per_step": mean[k], "ms_per_step_min": best[k],
                        "value": world * n / (mean[k] * 1e-3), "path": path,
                        "h2d_bytes_per_step": h2d}
            # The headline is the zero-copy form: the kernels read the step's
            # gradients, and write its parameters, in place in pinned host
            # memory, so the same bytes cross the host link every step without
            # a device copy; it runs steadily where the copy engines' time
            # varies with the shared host.
            e2e = {"value": world * n / (mean["zero_copy"] * 1e-3), "unit": UNIT,
                   "h2d_bytes_per_step": grad_bytes,
                   "d2h_bytes_per_step": n * host_params.element_size() + 4,
                   "ms_per_step": mean["zero_copy"], "ms_per_step_min": best["zero_copy"],
                   "steps": args.e2e_steps,
                   "path": "zero_step_shard reading the Nd gradient rows, and writing the new "
                           "parameters, in place in pinned host memory (zero-copy both ways over "
                           "the host link), then the flag device-to-host",
                   "other_forms": {
                       "fed": form("fed", f"zero_feed_buckets (DMA, {nbk} transfer buckets) + "
                                          "zero_step_shard_streamed", grad_bytes + 4 * nbk)
                       if not fed_timeouts else
                       {"unavailable": f"a bucket-ready wait expired (ZERO_ERR_TIMEOUT) in "
                                       f"{len(fed_timeouts)} of {args.e2e_steps + 1} iterations; "
                                       f"its times are not a measurement"},
                       "sequential": form("sequential", "one DMA copy of the gradients, then "
                                                        "zero_step_shard", grad_bytes),
                       "zero_copy_read_back": form(
                           "zero_copy_read_back", "zero_step_shard reading the rows in place in "
                           "host memory into device parameters, then a DMA copy of them",
                           grad_bytes),
                       "copies_alone": form("copies", "the DMA copies alone, no step",
                                            grads.numel() * grads.element_size())},
                   "ms_per_iteration": {k: [round(x, 3) for x in v] for k, v in times.items()},
                   "link": {"bound_ms": best["copies"],
                            "bound": "the fastest iteration of the DMA copies alone",
                            "frac": best["copies"] / mean["zero_copy"]}}
            if best["copies"] > mean["zero_copy"]:
                e2e["link"]["note"] = ("the copy engines ran slower than the kernels' own "
                                       "reads of host memory in this run: not a bound")
            del host_grads, host_params, dps_h

    # -- optionally the back-to-back steps once more as one CUDA graph: their
    #    kernels' time without the host's issue time (for shards whose step is
    #    issued slower than it runs).  Last, since the replays leave the
    #    driver's bookkeeping behind its data. ----------------------------------
    graph_ms = None
    if args.graph:
        def b2b():
            dps.launch(desc)
            dps.commit(False)
        graph_ms = max_over_ranks(time_graph(torch, stream, dev, b2b, nk), group, dev)

    # -- the other workloads' fused step (kernel time), rank 0 at N = 1 only --
    peaks = measured_peaks()
    per_config = None
    if world == 1 and not args.no_per_config and not (args.psi or args.nd or args.grad_dtype or
                                                       args.bucket or args.row_pad):
        pk = peaks.get("hbm_gbs") or 6800.0
        per_config = {f"{k} rank {r}" + (" (flat buffer slot)" if g == "full" else ""):
                      measure_config(k, r, g, dev, stream, pk)
                      for k, r, g in PER_CONFIG if (k, r, g) != (args.config, dp_rank,
                                                                   args.gathered)}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # -- report -----------------------------------------------------------------
    ms_per_step = total_ms / args.steps
    bytes_per_param = w.bytes_per_param
    kern_step_ms = statistics.fmean(kernel_ms)
    from zero_sharded_optimizer_02_gb300 import _abi
    per_step = _abi.fused_launch_count(n, w.bucket, 0)     # launch windows of one step
    kern_avg_ms = back_to_back_ms / per_step                # average launch duration
    launch_bytes = bytes_per_param * n / per_step           # algorithmic bytes per launch
    achieved = launch_bytes / (kern_avg_ms * 1e-3) / 1e9
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    traffic_pp = None if (args.psi or args.nd or args.grad_dtype or args.row_pad or
                          args.bucket) else \
        recorded_traffic(args.config, n)
    line = {
        "metric": METRIC,
        "value": world * n / (ms_per_step * 1e-3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded counter-based generator; no dataset or weights)",
        "config": bench_config(args, w, dp_rank, world),
        "gbs": bytes_per_param * n / (ms_per_step * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src,
                     "frac_of_nominal_7900": achieved / NOMINAL_HBM_GBS,
                     "traffic": None if traffic_pp is None else traffic_pp * n / per_step,
                     "kernel": kernel_name(n), "kernel_ms": kern_avg_ms,
                     "launches_per_step": per_step,
                     "kernel_ms_per_step": back_to_back_ms,
                     **({} if graph_ms is None else {
                         "kernel_ms_per_step_graph": graph_ms,
                         "frac_graph": bytes_per_param * n / (graph_ms * 1e-3) / 1e9 / peak}),
                     "kernel_ms_in_sync_step": kern_step_ms,
                     "kernel_ms_in_sync_step_median": statistics.median(kernel_ms),
                     "kernel_ms_in_sync_step_min": min(kernel_ms),
                     "steps_timed_back_to_back": nk,
                     "algorithmic_bytes_per_launch": launch_bytes,
                     "read_ceiling_gbs": read_gbs,
                     "frac_of_read_ceiling": achieved / read_gbs,
                     "read_ceiling": "zero_check_nonfinite over the same Nd rows (reads "
                                     "2 Nd B/param, writes nothing), same launch windows, "
                                     f"{nk} back-to-back passes"},
        "per_config": per_config,
        "e2e": e2e,
        "gpu_launches": launches,
        "driver": f"pipelined (up to {pipe.depth} steps launched ahead of the oldest "
                  f"undecided step's flag read)",
        "ms_per_step_sync_driver": sync_ms,
        "build_flags": os.environ.get("ZERO_NVCC_FLAGS", ""),
        "skipped_steps": skipped,
        "clocks": clocks,
        "wall_s_timed": wall1 - wall0,
    }
    if not args.no_cpu_baseline and world == 1:      # the host-core baseline: N = 1 only
        line["cpu_baseline"] = cpu_baseline(w, dp_rank, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU oracle timing (the baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def _oracle_sample(w, dp_rank: int, n_sample: int, first: int = 0):
    import numpy as np
    import torch

    import synth
    s, begin, n = synth.shard_of(w.psi, w.nd, dp_rank)
    first = min(first, n)
    n_sample = min(n_sample, n - first)
    idx = torch.arange(begin + first, begin + first + n_sample, dtype=torch.int64)
    rows = np.stack([synth.grad_values(w, 0, j, idx).view(torch.int16).numpy().view(np.uint16)
                     for j in range(w.nd)])
    st = [synth.state_values(w, k, idx).numpy() for k in ("master", "m", "v")]
    return rows, st, n_sample


def _oracle_step(orc, w, rows, st, n_sample, t):
    import numpy as np
    params = np.zeros(n_sample, np.uint16)
    return orc.step_rank(rows, n_sample, 0, n_sample, w.nd, orc.dtype_code(w.grad_dtype),
                         w.bucket, w.loss_scale, w.hparams, t, st[0], st[1], st[2], params, 0)


def _oracle_worker(args):
    """One host core: the oracle, as it stands, on its own contiguous slice of
    the shard, repeated for `seconds` (or `reps` times)."""
    key, dp_rank, n_sample, first, seconds, reps = args
    import torch
    torch.set_num_threads(1)
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    w = synth.WORKLOADS[key]
    rows, st, n = _oracle_sample(w, dp_rank, n_sample, first)
    _oracle_step(oracle, w, rows, st, n, 1)
    done, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(oracle, w, rows, st, n, 1 + done)
        done += 1
        el = time.perf_counter() - t0
        if (reps and done >= reps) or (not reps and el >= seconds):
            return done * n, el


def _cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_pool(key: str, dp_rank: int, n_per_core: int, seconds: float = 0.0,
                 reps: int = 0):
    """Run the oracle on every host core (spawned processes, one slice each)."""
    import multiprocessing as mp
    import oracle
    oracle.build()
    cores = _cores()
    jobs = [(key, dp_rank, n_per_core, i * n_per_core, seconds, reps) for i in range(cores)]
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_worker, jobs)
    params = sum(r[0] for r in res)
    elapsed = max(r[1] for r in res)
    return params / elapsed, cores, params, elapsed


def cpu_model() -> str:
    """The host CPU's model name (or the machine type if the OS does not say)."""
    import platform
    arm_parts = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1",
                 "0xd0c": "Arm Neoverse N1", "0xd49": "Arm Neoverse N2"}
    part = None
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return ln.split(":", 1)[1].strip()
                if key == "cpu part" and part is None:
                    part = ln.split(":", 1)[1].strip().lower()
    except OSError:
        pass
    if part:
        return arm_parts.get(part, f"{platform.machine()} (CPU part {part})")
    return platform.machine()


def cpu_baseline(w, dp_rank: int, seconds: float) -> dict:
    """The oracle as it stands (plain C, one process per host core) on
    contiguous slices of this rank's shard, each core repeating its slice for
    about ``seconds``."""
    n_per_core = 1 << 16
    rate, cores, params, el = _oracle_pool(w.key, dp_rank, n_per_core, seconds=seconds)
    return {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{cores} processes x {n_per_core} contiguous params of rank {dp_rank}'s "
                      f"shard ({w.nd} contributions each), {params} param-steps in {el:.1f} s",
            "per_core_value": rate / cores, "cpu_model": cpu_model(),
            "gbs": rate * w.bytes_per_param / 1e9}


def run_reference(args) -> None:
    """The reference arm: the CPU oracle, as it stands, on the host cores; each
    step is every core running the oracle once on its own slice of the bench
    workload's shard."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import synth
    w = synth.WORKLOADS[args.config]
    n_per_core = args.ref_sample
    _oracle_pool(w.key, args.rank, n_per_core, reps=args.warmup)
    rate, cores, params, el = _oracle_pool(w.key, args.rank, n_per_core, reps=args.steps)
    ms = el * 1e3 / args.steps
    sample = (f"each step: {cores} processes x {n_per_core} contiguous params of rank "
              f"{args.rank}'s shard ({w.nd} contributions each), plain C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded counter-based generator)",
        "config": bench_config(args, w, args.rank, world),
        "sample_params_per_step": params // args.steps,
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample, "per_core_value": rate / cores,
                         "cpu_model": cpu_model()},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_entry(args) -> None:
    """One entry point besides the fused step, on the bench workload's shard
    rows and state (rank --rank, shard view), timed over --steps back-to-back
    calls with CUDA events:
      check    zero_check_nonfinite (the in-place pre-check): 2 Nd B/param read;
      unfused  zero_step_shard_unfused (reduce into the fusion buffer, AdamW
               from it, cast): 2 Nd + 4 + 28 + 6 = 2 Nd + 38 B/param;
      streamed zero_step_shard_streamed with every ready word already set
               (the waits pass at once): 2 Nd + 26 B/param."""
    import torch

    import synth
    from zero_sharded_optimizer_02_gb300 import _abi, build
    from zero_sharded_optimizer_02_gb300.step import DataParallelStep
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = workload(args)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        dps = DataParallelStep(w.psi, w.nd, [args.rank], w.grad_dtype, w.hparams,
                               w.loss_scale, w.bucket, dev, gathered="slot",
                               fused=args.op != "unfused", stream=stream, row_align=ROW_ALIGN)
        L = dps.layouts[args.rank]
        n, pitch = int(L.length), int(L.row_pitch)
        st = dps.state[args.rank]
        for row, which in zip(st.bufs[st.cur], ("master", "m", "v")):
            synth.fill_shard_state(w, args.rank, which, row)
        grads = torch.empty(w.nd, pitch, dtype=w.torch_grad_dtype, device=dev)
        synth.fill_shard_rows(w, 0, args.rank, grads)
    desc = {args.rank: _abi.grads(grads, pitch, 0, w.nd, w.grad_dtype)}
    torch.cuda.synchronize(dev)

    if args.op == "check":
        def call():
            _abi.zero_check_nonfinite(desc[args.rank], 0, n, dps.flag, stream)
        bpp, launches = 2 * w.nd, 1
    elif args.op == "streamed":
        # every bucket's ready word already set: the bucket-ready kernel's own
        # rate, with the rows resident (the buckets of the end-to-end fed form)
        sb = max(8, -(-(-(-n // args.e2e_buckets)) // 8) * 8)
        ready = torch.ones(-(-n // sb), dtype=torch.int32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        st, Lr = dps.state[args.rank], dps.layouts[args.rank]

        def call():
            gbuf, goff = dps._gathered_target(args.rank, 1 - dps.gcur)
            dps.h.step = dps.t + 1
            _abi.zero_step_shard_streamed(desc[args.rank], Lr, st.states[st.cur],
                                          st.states[1 - st.cur], gbuf, goff, sb,
                                          dps.loss_scale, dps.h, ready, 1, 10 ** 10, dps.flag,
                                          status, stream)
            dps.commit(False)
        bpp, launches = 2 * w.nd + 26, _abi.streamed_launch_count(n, sb, w.nd, 0)
    else:
        def call():
            dps.launch(desc)
            dps.commit(False)
        bpp = 2 * w.nd + 38
        launches = _abi.unfused_launch_count(n, w.bucket, 0)
    for _ in range(args.warmup):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(args.steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    assert int(dps.flag.item()) == 0
    if args.op == "streamed":
        assert int(status.item()) == 0
    ms = e0.elapsed_time(e1) / args.steps
    gbs = bpp * n / (ms * 1e-3) / 1e9
    peak = measured_peaks().get("hbm_gbs", 6800.0)
    name = {"check": "zero_check_nonfinite", "unfused": "zero_step_shard_unfused",
            "streamed": "zero_step_shard_streamed"}[args.op]
    print(json.dumps({"op": name, "metric": "params/s", "value": n / (ms * 1e-3),
                      "unit": "params/s", "ms_per_call": ms,
                      "config": {"workload": f"{args.config}: {w.title}", "shard_params": n,
                                 "nd": w.nd, "bucket": w.bucket, "rank": args.rank},
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak,
                                   "unit": "GB/s", "frac": gbs / peak,
                                   "algorithmic_bytes_per_param": bpp},
                      "gpu_launches": args.steps * launches}), flush=True)


def run_gather(args) -> None:
    """ZeRO-3 on-demand gather: zero_gather_range collecting the whole flat
    fp16 parameter vector of a workload from its Nd pitched shards (the worst
    case of a layer gather: every shard segment).  HBM roofline: 2 B read +
    2 B written per parameter."""
    import torch

    import synth
    from zero_sharded_optimizer_02_gb300 import _abi, build
    build.build()
    dev = torch.device("cuda", 0)
    w = synth.WORKLOADS[args.config]
    L = _abi.zero_partition_layout(w.psi, w.nd, 0, 8)
    pitch = int(L.row_pitch)
    shards = torch.randint(-30000, 30000, (w.nd, pitch), dtype=torch.int16, device=dev)
    out = torch.empty(w.psi, dtype=torch.int16, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        _abi.zero_gather_range(shards, pitch, w.psi, w.nd, 0, w.psi, 2, out, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(args.steps):
        _abi.zero_gather_range(shards, pitch, w.psi, w.nd, 0, w.psi, 2, out, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    # spot check against the flat concatenation
    s = int(L.shard_elems)
    for i in (0, 1, s - 1, s, w.psi // 2, w.psi - 1):
        assert int(out[i]) == int(shards[i // s, i % s]), i
    gbs = 4 * w.psi / (ms * 1e-3) / 1e9
    peak = measured_peaks().get("hbm_gbs", 6800.0)
    print(json.dumps({"op": "zero_gather_range", "metric": "params gathered/s", "value":
                      w.psi / (ms * 1e-3), "unit": "params/s", "ms_per_gather": ms,
                      "config": {"workload": f"{args.config}: {w.title}", "psi": w.psi,
                                 "nd": w.nd, "segments": w.nd, "elem_bytes": 2},
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak,
                                   "unit": "GB/s", "frac": gbs / peak,
                                   "algorithmic_bytes_per_param": 4},
                      "gpu_launches": args.steps * _abi.gather_launch_count(
                          w.psi, w.nd, 0, w.psi)}), flush=True)


def run_checkpoint(args) -> None:
    """Sharded checkpoint of every rank's fp32 state (master, m, v): each rank
    saves its file, then one rank of Nd + 1 loads its range from the old
    files (resharding).  Host I/O, timed beside a plain write and read of the
    same bytes in the same directory (the I/O bound of this host)."""
    import tempfile

    import numpy as np

    import synth
    from zero_sharded_optimizer_02_gb300 import _abi, build
    build.build()
    w = synth.WORKLOADS[args.config]
    nd = w.nd
    if 12 * w.psi > 16e9:
        sys.exit(f"--op checkpoint writes 12 B per parameter ({12 * w.psi / 1e9:.0f} GB for "
                 f"{args.config}); use a workload of at most 1.3e9 parameters")
    d = tempfile.mkdtemp(prefix="zero_ckpt_")
    paths, total = [], 0
    saves = []
    for r in range(nd):
        L = _abi.zero_partition_layout(w.psi, nd, r, 8)
        n = int(L.length)
        arr = [np.full(n, k + r, np.float32) for k in range(3)]
        p = os.path.join(d, f"r{r}.zck")
        t0 = time.perf_counter()
        _abi.zero_checkpoint_save(p, L, _abi.adamw(**w.hparams, step=7), *arr)
        saves.append(time.perf_counter() - t0)
        paths.append(p)
        total += 12 * n
    L = _abi.zero_partition_layout(w.psi, nd + 1, 0, 8)
    buf = [np.empty(int(L.length), np.float32) for _ in range(3)]
    t0 = time.perf_counter()
    _abi.zero_checkpoint_load(paths, L, *buf)
    load_s = time.perf_counter() - t0
    # the reshard read every old file it overlaps whole (checksum) plus its range
    s_old = -(-w.psi // nd)
    lo, hi = int(L.begin), int(L.begin) + int(L.length)
    read_files = [r for r in range(nd) if r * s_old < hi and lo < min((r + 1) * s_old, w.psi)]
    load_bytes = sum(os.path.getsize(paths[r]) for r in read_files) + 12 * int(L.length)
    # plain I/O of the same sizes: rank 0's bytes written and read back
    n0 = int(_abi.zero_partition_layout(w.psi, nd, 0, 8).length)
    plain = np.full(3 * n0, 1.0, np.float32)
    q = os.path.join(d, "plain.bin")
    t0 = time.perf_counter()
    with open(q, "wb") as f:
        plain.tofile(f)
        f.flush()
    plain_w = time.perf_counter() - t0
    t0 = time.perf_counter()
    back = np.fromfile(q, np.float32)
    plain_r = time.perf_counter() - t0
    assert back.size == plain.size
    os.remove(q)
    for p in paths:
        os.remove(p)
    os.rmdir(d)
    print(json.dumps({"op": "zero_checkpoint", "metric": "checkpoint GB/s (host)",
                      "save_gbs": total / sum(saves) / 1e9,
                      "load_reshard_gbs": load_bytes / load_s / 1e9,
                      "load_reshard_s": load_s, "files_read": len(read_files),
                      "plain_write_gbs": plain.nbytes / plain_w / 1e9,
                      "plain_read_gbs": plain.nbytes / plain_r / 1e9,
                      "config": {"workload": f"{args.config}: {w.title}", "nd_saved": nd,
                                 "nd_loaded": nd + 1, "bytes_saved": total,
                                 "dir": "tempfile.mkdtemp() (page cache)"}}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=["step", "gather", "checkpoint", "check", "unfused",
                                     "streamed"], default="step",
                    help="step (the benchmark line) or a measurement of another entry point")
    ap.add_argument("--config", default="c4", choices=["c0", "c1", "c2", "c3", "c4"])
    ap.add_argument("--rank", type=int, default=0, help="first data-parallel rank to run")
    ap.add_argument("--variant", choices=["registers", "ring", "tma", "small"], default=None,
                    help="fused-step kernel for every window (sets ZERO_FUSED_VARIANT; "
                         "default: the ring, and the short-window kernel for a shard "
                         "that one wave of it covers, SMs x 3,072 elements)")
    ap.add_argument("--graph", action="store_true",
                    help="also time the back-to-back steps as one CUDA graph (kernel time "
                         "without host issue time)")
    ap.add_argument("--gathered", choices=["slot", "full"], default="slot",
                    help="slot: the rank's own S-element parameter buffer; full: its slot at "
                         "r*S of the flat Nd*S buffer (odd ranks then start off the 16-byte "
                         "boundary when S mod 8 != 0)")
    ap.add_argument("--psi", type=int, default=0, help="override the parameter count")
    ap.add_argument("--nd", type=int, default=0, help="override the data-parallel degree")
    ap.add_argument("--bucket", type=int, default=0, help="override the bucket size")
    ap.add_argument("--grad-dtype", choices=["f16", "bf16"], default=None,
                    help="override the gradient dtype")
    ap.add_argument("--row-pad", type=int, default=0,
                    help="extra elements (multiple of 8) between contribution rows")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--e2e-buckets", type=int, default=16,
                    help="transfer buckets of the host-fed e2e step")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads' kernel timings of the default line")
    ap.add_argument("--ref-sample", type=int, default=1 << 13,
                    help="params per core per step of the reference (oracle) arm")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.row_pad % 8:
        ap.error("--row-pad must be a multiple of 8 elements")
    if args.variant:
        os.environ["ZERO_FUSED_VARIANT"] = args.variant
    if args.impl == "reference":
        run_reference(args)
    elif args.op in ("check", "unfused", "streamed"):
        run_entry(args)
    elif args.op == "gather":
        run_gather(args)
    elif args.op == "checkpoint":
        run_checkpoint(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
