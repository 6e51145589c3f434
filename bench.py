#!/usr/bin/env python3
"""Benchmark of the ZeRO gradient-bucket reduction on GB300.

Workload (one "step" = one pass of the whole path over one batch):
  K = 8 simulated ranks, one 1 GiB bf16 bucket per rank (N = 2**29 elements),
  filled from 32 fragmented 4096x4096 gradients per rank.
    1. flatten   the 32 fragments of every rank into its flat bucket
    2. RS fp32   reduce-scatter, ring-order fp32 sums, 2 micro-batches
                 accumulated first, x1/8, cast into fp32 partition shards
    3. RS hop    the same with bf16 partial sums on the wire, accumulating
                 into existing fp32 partition shards
    4. AG        all-gather of 8 bf16 parameter shards into 8 full replicas
    5. AR        fused all-reduce (ring fp32, x1/8, bf16 replicas)
Inputs stay resident in HBM (45 GiB, far larger than the 129 MB L2, so no
flush is needed between steps).

value  = algorithmic bytes of a step (each input read once, each output
         written once) x steps / device time, in GB/s (1e9 B/s).
e2e    = the same bytes over the time of steps that also copy the step's
         inputs from pinned host memory and read every result back.
roofline = the dominant kernel's algorithmic bytes per launch / its average
         CUDA-event launch time, against the measured HBM copy peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dpr|reference]
                  [--workload zero_bucket|zero3_per_param|bucket_pipeline|bf16_partition|
                              sweep|configs|fragments|point]

The default workload is the headline step above; the others time the
per-parameter path, the stream-overlapped bucket pipeline, the bf16
partitions, configuration 5's sweep, configurations 1-4, the reduce-scatter
straight from fragments, and one point chosen on the command line.

--impl reference times the CPU oracle (its C ring simulation, one process per
host core, each on its own slab) on a bounded sample of the same workload.  With --gpus N > 1 (under torchrun) every rank runs an
independent replica of the workload on its own GPU (the path does not shard
across GPUs); the job value is the bytes of all ranks over the slowest rank's
time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "reduce-scatter/all-gather effective HBM GB/s at K=8, 1 GB/rank; % of GB300 peak"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
STEP_KERNELS = ("flatten", "rs_fp32_m2", "rs_hop_m2_acc", "allgather", "allreduce")
Z3_KERNELS = ("rs_coalesced", "ag_coalesced")
BF16_KERNELS = ("rs_bf16_copy", "rs_bf16_add", "cast")

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per full-size
# launch, scaled from one ncu capture of a small case of the same kernel: the
# bench's step kernels at 2**25 elements per rank (x16 to the full 2**29), the
# per-parameter kernels on one layer of the 7-layer model (x7), the bf16
# partition kernels at 2**25 elements per rank (x16).  Each entry holds only
# while the kernel's sources hash to `src_sha`; otherwise the bench reports
# null.  Dirty lines still in L2 when a kernel ends (at most the L2's 129 MB)
# are not counted at either size, so the scaled write traffic is a slight
# underestimate.
NCU_TRAFFIC = {
    "flatten": {"bytes": 16_290_209_792, "small_case_bytes": 1_018_138_112, "scale": 16,
        "src_sha": "b613c2b04ba85972"},
    "rs_fp32_m2": {"bytes": 19_163_496_448, "small_case_bytes": 1_197_718_528, "scale": 16,
        "src_sha": "9d0af4a9c5c06563"},
    "rs_hop_m2_acc": {"bytes": 21_305_192_448, "small_case_bytes": 1_331_574_528, "scale": 16,
        "src_sha": "9d0af4a9c5c06563"},
    "allgather": {"bytes": 8_736_522_240, "small_case_bytes": 546_032_640, "scale": 16,
        "src_sha": "b613c2b04ba85972"},
    "allreduce": {"bytes": 16_272_740_352, "small_case_bytes": 1_017_046_272, "scale": 16,
        "src_sha": "9d0af4a9c5c06563"},
    "rs_fp32_m1": {"bytes": 10_433_806_336, "small_case_bytes": 652_112_896, "scale": 16,
        "src_sha": "9d0af4a9c5c06563"},
    "rs_hop_m1": {"bytes": 10_429_546_496, "small_case_bytes": 651_846_656, "scale": 16,
        "src_sha": "9d0af4a9c5c06563"},
    "rs_coalesced": {"bytes": 21_887_973_632, "small_case_bytes": 3_126_853_376, "scale": 7,
        "src_sha": "6db8cec815e4b3a0"},
    "ag_coalesced": {"bytes": 19_398_374_912, "small_case_bytes": 2_771_196_416, "scale": 7,
        "src_sha": "9fdeaea1861c48c0"},
    "rs_bf16_copy": {"bytes": 9_522_950_144, "small_case_bytes": 595_184_384, "scale": 16,
        "src_sha": "9d0af4a9c5c06563"},
    "rs_bf16_add": {"bytes": 10_583_232_512, "small_case_bytes": 661_452_032, "scale": 16,
        "src_sha": "9d0af4a9c5c06563"},
    "cast": {"bytes": 2_331_922_432, "small_case_bytes": 145_745_152, "scale": 16,
        "src_sha": "be25e80a1cc2945b"},
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["dpr", "reference"], default="dpr")
    p.add_argument("--e2e-steps", type=int, default=8)
    p.add_argument("--pg-timeout", type=float, default=600.0,
                   help="seconds before a collective of the multi-rank harness gives up on "
                        "a rank that has gone")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--workload", choices=["zero_bucket", "zero3_per_param", "bucket_pipeline",
                                          "bf16_partition", "sweep", "configs", "point",
                                          "fragments", "sequence"],
                   default="zero_bucket",
                   help="zero_bucket: the headline step (default); zero3_per_param: the ZeRO-3 "
                        "discrete path on config 3's 56 gradients; bucket_pipeline: backward "
                        "time under the stream-overlap policies; bf16_partition: reduce-scatter "
                        "into bf16 partitions over two micro steps and the step-time cast; "
                        "sweep: configuration 5; configs: configurations 1-4; fragments: the "
                        "1 GiB bucket reduced straight from its fragments; sequence: 64 "
                        "buckets of 4 MiB per rank back to back, plain, programmatic and "
                        "batched launches; point: one "
                        "reduce-scatter / all-gather / all-reduce point chosen by --K, "
                        "--bytes-per-rank, --mode, --micro, --seed")
    p.add_argument("--K", type=int, default=8, help="point: simulated ranks")
    p.add_argument("--bytes-per-rank", type=int, default=1 << 28, help="point: bf16 bytes per rank")
    p.add_argument("--mode", choices=["ring_fp32", "hop_bf16"], default="ring_fp32",
                   help="point: reduce-scatter summation mode")
    p.add_argument("--micro", type=int, default=1, choices=[1, 2],
                   help="point: micro-batches accumulated before the reduce")
    p.add_argument("--seed", type=int, default=0, help="point: generator seed")
    p.add_argument("--z3-layers", type=int, default=None,
                   help="profile helper: layers of the zero3_per_param model (a small case); "
                        "its bench line is quoted only at the default 7")
    p.add_argument("--bucket-elems", type=int, default=25_000_000,
                   help="configs: bucket cap of configuration 3, in elements per rank")
    p.add_argument("--only", choices=STEP_KERNELS + ("rs_fp32_m1", "rs_hop_m1") + Z3_KERNELS
                   + BF16_KERNELS, default=None,
                   help="profile helper: launch only this kernel per step")
    p.add_argument("--graph", action="store_true",
                   help="capture one step's launches in a CUDA graph and replay it")
    p.add_argument("--n-per-rank", type=int, default=None,
                   help="profile helper: elements per rank (a multiple of 2**24) for a small "
                        "case; the bench line is quoted only at the default 2**29")
    return p.parse_args(argv)


# ---- multi-process harness (host logic; covered by gloo tests) ------------------

def dist_env():
    """(rank, world, local_rank) from torchrun's environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(backend: str, device=None, timeout_s: float = 600.0):
    """Process group over torchrun's environment.  A rank that dies between
    steps makes the others' next barrier or reduction end with an error
    within timeout_s instead of waiting forever."""
    import datetime

    import torch.distributed as dist
    kw = {"timeout": datetime.timedelta(seconds=timeout_s)}
    if device is not None:
        kw["device_id"] = device
    dist.init_process_group(backend, **kw)


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def all_ranks(flag: bool, device=None) -> bool:
    """True only if flag is true on every rank (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return flag
    t = torch.tensor([1 if flag else 0], dtype=torch.int32, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return bool(t.item())


def host_available_bytes() -> int:
    """MemAvailable of this host (Linux), or a very large number elsewhere."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 1 << 62


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def job_value(bytes_per_step: float, steps: int, world: int, max_seconds: float) -> float:
    """GB/s of the whole job: every rank's bytes over the slowest rank's time."""
    return bytes_per_step * steps * world / max_seconds / 1e9


# ---- measurement helpers ---------------------------------------------------------

def ring_busbw(kernel: str, K: int, N: int, seconds: float):
    """Ring-equivalent bus bandwidth in GB/s, the collective libraries' figure
    (CMU 11-868 Lecture 14 notes, section 3.4): a ring reduce-scatter or
    all-gather of N elements per rank moves (K-1)/K of the N-element message
    per rank, a ring all-reduce twice that.  None for the bucket gather."""
    hops = {"rs": 1, "allgather": 1, "allreduce": 2}
    key = "rs" if kernel.startswith("rs_") else kernel
    if key not in hops:
        return None
    return hops[key] * (K - 1) / K * 2 * N / seconds / 1e9


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Source files that determine each timed kernel and its launch (kernel code,
# shared device headers, host-side layout selection and grid sizing).
_COMMON_SRC = ["dpr_device.cuh", "dpr_kernels.h", "dpr_api.cu", "host_checks.h"]
KERNEL_SOURCES = {
    "flatten": ["gather_kernels.cu"] + _COMMON_SRC,
    "allgather": ["gather_kernels.cu"] + _COMMON_SRC,
    "rs_fp32_m2": ["reduce_kernels.cu", "dpr_ring.cuh"] + _COMMON_SRC,
    "rs_hop_m2_acc": ["reduce_kernels.cu", "dpr_ring.cuh"] + _COMMON_SRC,
    "allreduce": ["reduce_kernels.cu", "dpr_ring.cuh"] + _COMMON_SRC,
    "rs_fp32_m1": ["reduce_kernels.cu", "dpr_ring.cuh"] + _COMMON_SRC,
    "rs_hop_m1": ["reduce_kernels.cu", "dpr_ring.cuh"] + _COMMON_SRC,
    "rs_coalesced": ["coalesced.cu", "dpr_ring.cuh", "dpr_device.cuh", "dpr_kernels.h",
                     "host_checks.h"],
    "ag_coalesced": ["coalesced.cu", "dpr_device.cuh", "dpr_kernels.h", "host_checks.h"],
    "rs_bf16_copy": ["reduce_kernels.cu", "dpr_ring.cuh"] + _COMMON_SRC,
    "rs_bf16_add": ["reduce_kernels.cu", "dpr_ring.cuh"] + _COMMON_SRC,
    "cast": ["reduce_kernels.cu"] + _COMMON_SRC,
}


def kernel_src_sha(kernel: str | None = None) -> str:
    """Hash of the sources of one timed kernel (all of csrc/ when None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gradient_reduction_gb300", "csrc")
    files = KERNEL_SOURCES.get(kernel) if kernel else None
    for f in sorted(files or os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip() == "Active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- the device workload -----------------------------------------------------------

class Workload:
    """Device-resident buffers of the bench workload and one step's launches.

    Each kind of buffer is one contiguous allocation with one row per rank
    (fragments: one row per rank and fragment), so that host<->device copies
    move each kind in one call.  With fill=False the buffers are left
    uninitialised (a second buffer set for the pipelined end-to-end steps,
    whose inputs arrive from the host)."""

    def __init__(self, dev, stream, n_per_rank=None, fill=True):
        import dataclasses

        import torch
        import gradient_reduction_gb300 as dpr
        from workloads import configs as C
        from workloads import synthetic as syn
        self.dpr, self.torch = dpr, torch
        w = C.BENCH
        if n_per_rank is not None and n_per_rank != w.N:
            if n_per_rank <= 0 or n_per_rank % w.frag_numel:
                raise ValueError("--n-per-rank must be a positive multiple of 2**24")
            w = dataclasses.replace(w, N=n_per_rank, n_frag=n_per_rank // w.frag_numel)
        self.w, self.dev, self.stream = w, dev, stream
        K, N = w.K, w.N
        S = N // K
        F, P = w.frag_numel, w.n_frag
        self.K, self.N, self.S, self.F, self.P = K, N, S, F, P
        bf, f32 = torch.bfloat16, torch.float32
        with torch.cuda.stream(stream):
            self.frag_all = torch.empty(K * P, F, dtype=bf, device=dev)
            self.ipg0_all = torch.empty(K, N, dtype=bf, device=dev)
            self.ipg1_all = torch.zeros(K, N, dtype=bf, device=dev)
            self.part_f32_all = torch.empty(K, S, dtype=f32, device=dev)
            self.part_hop_all = torch.empty(K, S, dtype=f32, device=dev)
            self.shards_all = torch.empty(K, S, dtype=bf, device=dev)
            self.params_all = torch.empty(K, N, dtype=bf, device=dev)
            self.ar_all = torch.empty(K, N, dtype=bf, device=dev)
            if fill:
                for r in range(K):
                    for p in range(P):
                        w.dist.fill(0, F, w.frag_key(r, p), device=dev,
                                    out=self.frag_all[r * P + p])
                    w.dist.fill(0, N, w.micro0_key(r), device=dev, out=self.ipg0_all[r])
                    self.part_hop_all[r].copy_(
                        syn.gauss_bf16(0, S, w.prev_grad_key(r), 1e-3, device=dev))
                    w.param_dist.fill(r * S, S, w.param_key(), device=dev, out=self.shards_all[r])
            self.frags = [[self.frag_all[r * P + p].view(*w.frag_shape) for p in range(P)]
                          for r in range(K)]
            self.ipg0 = list(self.ipg0_all.unbind(0))
            self.ipg1 = list(self.ipg1_all.unbind(0))
            self.part_f32 = list(self.part_f32_all.unbind(0))
            self.part_hop = list(self.part_hop_all.unbind(0))
            self.shards = list(self.shards_all.unbind(0))
            self.params = list(self.params_all.unbind(0))
            self.ar_out = list(self.ar_all.unbind(0))
            self.plan = dpr.dpr_flatten_plan_create(
                self.frags, [F] * P, [p * F for p in range(P)], N, stream=stream)
        stream.synchronize()
        self.bytes = {
            "flatten": 4 * K * N,
            "rs_fp32_m2": 2 * 2 * K * N + 4 * N,
            "rs_hop_m2_acc": 2 * 2 * K * N + 4 * N + 4 * N,
            "allgather": 2 * N + 2 * K * N,
            "allreduce": 4 * K * N,
            "rs_fp32_m1": 2 * K * N + 4 * N,
            "rs_hop_m1": 2 * K * N + 4 * N,
        }
        self.launches_per_step = len(STEP_KERNELS)

    # inputs a step reads from the host, outputs it returns (e2e steps)
    def inputs(self):
        return [self.frag_all, self.ipg0_all, self.part_hop_all, self.shards_all]

    def outputs(self):
        return [self.part_f32_all, self.part_hop_all, self.params_all, self.ar_all]

    def launch(self, name):
        dpr, K, N, s = self.dpr, self.K, self.N, self.stream
        if name == "flatten":
            dpr.dpr_flatten_bucket(self.plan, self.ipg1, stream=s)
        elif name == "rs_fp32_m2":
            dpr.dpr_reduce_scatter(self.ipg0 + self.ipg1, K, 2, N, self.part_f32,
                                   mode=dpr.RING_FP32, scale=1.0 / K, stream=s)
        elif name == "rs_hop_m2_acc":
            dpr.dpr_reduce_scatter(self.ipg0 + self.ipg1, K, 2, N, self.part_hop,
                                   mode=dpr.HOP_BF16, scale=1.0 / K, accumulate=True, stream=s)
        elif name == "allgather":
            dpr.dpr_allgather(self.shards, K, N, self.params, stream=s)
        elif name == "allreduce":
            dpr.dpr_allreduce(self.ipg1, K, N, self.ar_out, mode=dpr.RING_FP32, scale=1.0 / K,
                              stream=s)
        elif name == "rs_fp32_m1":          # the metric's own reduce-scatter (profile helper)
            dpr.dpr_reduce_scatter(self.ipg0, K, 1, N, self.part_f32, mode=dpr.RING_FP32,
                                   scale=1.0 / K, stream=s)
        elif name == "rs_hop_m1":
            dpr.dpr_reduce_scatter(self.ipg0, K, 1, N, self.part_f32, mode=dpr.HOP_BF16,
                                   scale=1.0 / K, stream=s)
        else:
            raise ValueError(name)

    def step(self, kernels, events=None):
        for name in kernels:
            if events is not None:
                a = self.torch.cuda.Event(enable_timing=True)
                b = self.torch.cuda.Event(enable_timing=True)
                a.record(self.stream)
                self.launch(name)
                b.record(self.stream)
                events.append((name, a, b))
            else:
                self.launch(name)


class Zero3Workload:
    """The ZeRO-3 discrete path on config 3: K=8 ranks, 56 separately allocated
    gradients of a 7-layer hidden-4096 transformer per rank.  A step
    reduce-scatters every gradient into per-parameter shards (fp32 partitions,
    ring fp32, x1/8) and all-gathers bf16 partitions back into 56 full
    parameters per rank."""
    kernels = Z3_KERNELS

    def __init__(self, dev, stream, layers: int | None = None):
        import dataclasses

        import torch
        import gradient_reduction_gb300 as dpr
        from workloads import configs as C
        self.dpr, self.torch, self.dev, self.stream = dpr, torch, dev, stream
        cfg = C.CFG3 if layers is None else dataclasses.replace(C.CFG3, layers=layers)
        K = cfg.K
        arr = cfg.arrival_order()
        numel = [n for *_, n in arr]
        with torch.cuda.stream(stream):
            self.grads = [[cfg.grad(r, p, device=dev) for p in range(len(arr))] for r in range(K)]
            self.params = [[torch.empty(n, dtype=torch.bfloat16, device=dev) for n in numel]
                           for _ in range(K)]
            self.rs_plan = dpr.dpr_coalesced_plan_create(self.grads, numel, stream=stream)
            self.ag_plan = dpr.dpr_coalesced_plan_create(self.params, numel, stream=stream)
            L = self.rs_plan.partition_numel
            self.part = [torch.empty(L, dtype=torch.float32, device=dev) for _ in range(K)]
            self.shards = [torch.empty(L, dtype=torch.bfloat16, device=dev) for _ in range(K)]
            for j in range(K):
                self.shards[j].copy_(cfg.dist.fill(0, L, cfg.key(j, 10_000), device=dev))
        stream.synchronize()
        N = sum(numel)
        self.K, self.N, self.L = K, N, L
        self.bytes = {"rs_coalesced": 2 * K * N + 4 * K * L, "ag_coalesced": 2 * K * L + 2 * K * N}

    def launch(self, name):
        dpr, s = self.dpr, self.stream
        if name == "rs_coalesced":
            dpr.dpr_reduce_scatter_coalesced(self.rs_plan, self.part, mode=dpr.RING_FP32,
                                             scale=1.0 / self.K, stream=s)
        elif name == "ag_coalesced":
            dpr.dpr_allgather_coalesced(self.ag_plan, self.shards, stream=s)
        else:
            raise ValueError(name)

    step = Workload.step

    def close(self):
        self.rs_plan.close()
        self.ag_plan.close()


class Bf16PartitionWorkload:
    """The ZeRO-3 literal partition data flow at K=8, 1 GiB per rank: micro
    step 0 reduce-scatters into bf16 partition shards (copy_), micro step 1
    reduce-scatters the next micro-batch and adds in bf16 (add_), and step()
    casts the partition to fp32."""
    kernels = ("rs_bf16_copy", "rs_bf16_add", "cast")

    def __init__(self, dev, stream, n_per_rank=None):
        import torch
        import gradient_reduction_gb300 as dpr
        from workloads import configs as C
        self.dpr, self.torch, self.dev, self.stream = dpr, torch, dev, stream
        w = C.BENCH
        K, N = w.K, (n_per_rank or w.N)
        if N % (16 * K):
            raise ValueError("--n-per-rank must be a multiple of 16 K")
        S = N // K
        with torch.cuda.stream(stream):
            self.x = torch.empty(2, K, N, dtype=torch.bfloat16, device=dev)
            for m, key in ((0, w.micro0_key), (1, lambda r: w.frag_key(r, 0))):
                for r in range(K):
                    w.dist.fill(0, N, key(r), device=dev, out=self.x[m, r])
            self.part = torch.empty(K, S, dtype=torch.bfloat16, device=dev)
            self.f32 = torch.empty(K * S, dtype=torch.float32, device=dev)
        stream.synchronize()
        self.K, self.N, self.S = K, N, S
        self.bytes = {"rs_bf16_copy": 2 * K * N + 2 * N, "rs_bf16_add": 2 * K * N + 4 * N,
                      "cast": 6 * N}

    def launch(self, name):
        dpr, K, N, s = self.dpr, self.K, self.N, self.stream
        if name == "rs_bf16_copy":
            dpr.dpr_reduce_scatter_bf16(list(self.x[0].unbind(0)), K, 1, N, list(self.part.unbind(0)),
                                        stream=s)
        elif name == "rs_bf16_add":
            dpr.dpr_reduce_scatter_bf16(list(self.x[1].unbind(0)), K, 1, N, list(self.part.unbind(0)),
                                        accumulate=True, stream=s)
        elif name == "cast":
            dpr.dpr_cast_bf16_to_fp32(self.part.view(-1), self.f32, stream=s)
        else:
            raise ValueError(name)

    step = Workload.step

    def close(self):
        pass


class PipelineBackward:
    """A simulated backward pass for the bucket pipeline: 16 buckets (one
    gradient per rank each, K=8, alternately 3 * 2**23 and 2**23 elements),
    each preceded by backward compute stood in for by bf16 4096^3 matmuls on
    the compute stream (alternately 1 and 3), so the reductions of large
    buckets outlast the compute that follows them.  run() times one backward
    under a wait policy ("per_buffer", "reverse_wait") or "serial" (gather and
    reduce on the compute stream, i.e. no overlap)."""

    def __init__(self, dev, n_buckets=16):
        import torch
        import gradient_reduction_gb300 as dpr
        from workloads import synthetic as syn
        self.torch, self.dpr, self.dev = torch, dpr, dev
        self.K = K = 8
        self.sizes = [3 * (1 << 23) if i % 2 == 0 else (1 << 23) for i in range(n_buckets)]
        self.mms = [1 if i % 2 == 0 else 3 for i in range(n_buckets)]
        self.grads = [[syn.gauss_bf16(0, n, syn.stream_key(0x91, r, 0, i), 1e-3, device=dev)
                       for r in range(K)] for i, n in enumerate(self.sizes)]
        self.plans = [dpr.dpr_flatten_plan_create([[g] for g in gi], [n], [0], n)
                      for gi, n in zip(self.grads, self.sizes)]
        self.outs = [[torch.empty(n // K, dtype=torch.float32, device=dev) for _ in range(K)]
                     for n in self.sizes]
        self.a = torch.randn(4096, 4096, device=dev).to(torch.bfloat16)
        self.b = torch.randn(4096, 4096, device=dev).to(torch.bfloat16)
        self.c = torch.empty(4096, 4096, dtype=torch.bfloat16, device=dev)
        self.ipg = [torch.empty(max(self.sizes), dtype=torch.bfloat16, device=dev) for _ in range(K)]
        self.bytes = sum(4 * K * n + 2 * K * n + 4 * n for n in self.sizes)   # gather + RS
        self.cur = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize()

    def compute(self, i):
        for _ in range(self.mms[i]):
            self.torch.matmul(self.a, self.b, out=self.c)

    def run(self, policy: str, max_blocks: int = 0) -> float:
        torch, dpr, K = self.torch, self.dpr, self.K
        cur = self.cur
        pipe = None
        if policy != "serial":
            pipe = dpr.BucketPipeline(K, max(self.sizes), 2,
                                      dpr.WAIT_PER_BUFFER if policy == "per_buffer"
                                      else dpr.WAIT_REDUCTION_STREAM, max_blocks)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(cur):
            t0.record(cur)
            for i, n in enumerate(self.sizes):
                self.compute(i)
                if pipe is None:
                    views = [t[:n] for t in self.ipg]
                    dpr.dpr_flatten_bucket(self.plans[i], views, stream=cur)
                    dpr.dpr_reduce_scatter(views, K, 1, n, self.outs[i], stream=cur)
                else:
                    pipe.submit(self.plans[i], self.outs[i], stream=cur)
            if pipe is not None:
                pipe.flush(stream=cur)
            t1.record(cur)
        torch.cuda.synchronize()
        if pipe is not None:
            pipe.close()
        return t0.elapsed_time(t1) / 1e3

    def run_parts(self):
        """Compute alone and gather+reduce alone (serial), for the overlap bound."""
        torch, dpr, K, cur = self.torch, self.dpr, self.K, self.cur
        res = {}
        for name in ("compute", "reduce"):
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            with torch.cuda.stream(cur):
                t0.record(cur)
                for i, n in enumerate(self.sizes):
                    if name == "compute":
                        self.compute(i)
                    else:
                        views = [t[:n] for t in self.ipg]
                        dpr.dpr_flatten_bucket(self.plans[i], views, stream=cur)
                        dpr.dpr_reduce_scatter(views, K, 1, n, self.outs[i], stream=cur)
                t1.record(cur)
            torch.cuda.synchronize()
            res[name] = t0.elapsed_time(t1) / 1e3
        return res

    def close(self):
        for p in self.plans:
            p.close()


class LaunchTimer:
    """Average launch time of fn() on stream s (CUDA events).  Working sets
    below 1 GiB are timed launch by launch with the L2 flushed before each
    launch by reading 512 MiB, so no point is measured L2-resident (a read
    leaves clean lines; a write-based flush would leave ~129 MB of dirty lines
    whose write-back the timed kernel would pay for)."""

    def __init__(self, s, steps: int, warmup: int):
        import torch
        self.torch, self.s, self.steps, self.warmup = torch, s, steps, warmup
        self.flush = torch.ones(128 << 20, dtype=torch.int32, device=s.device)  # 512 MiB > L2

    def __call__(self, fn, working_set: int) -> float:
        torch, s = self.torch, self.s
        torch.cuda.synchronize()
        for _ in range(self.warmup):
            fn()
        s.synchronize()
        if working_set >= (1 << 30):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            for _ in range(self.steps):
                fn()
            b.record(s)
            s.synchronize()
            return a.elapsed_time(b) / 1e3 / self.steps
        ts = []
        for _ in range(self.steps):
            with torch.cuda.stream(s):
                self.flush.sum()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            ts.append((a, b))
        s.synchronize()
        return sum(a.elapsed_time(b) for a, b in ts) / 1e3 / len(ts)


def run_configs_bench(args):
    """Configurations 1 to 4 as the workload table states them, each timed
    like the sweep (configuration 5): algorithmic bytes over the average time
    of the listed launches.
      1: K=4, N=4096: reduce-scatter ring fp32 x1/4 and all-reduce (launch-bound)
      2: K=8, one 25M-element bucket per rank: reduce-scatter, both modes, x1/8
      3: K=8, 56 fragmented gradients of a 7-layer hidden-4096 model: each
         bucket gathered by offset table, then reduce-scattered (ring fp32) into
         the fp32 partition; one figure for all buckets of a backward pass
      4: K=8, all-gather of one hidden-8192 layer from 1/8 shards."""
    import torch
    import gradient_reduction_gb300 as dpr
    from workloads import configs as C
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = torch.cuda.Stream(device=dev)
    timed = LaunchTimer(s, args.steps, args.warmup)
    bf, f32 = torch.bfloat16, torch.float32
    rows = []

    def row(cfg, op, nbytes, t, launches=1):
        r = {"config": cfg, "op": op, "bytes": int(nbytes), "launches": launches,
             "us": round(t * 1e6, 2), "gbs": round(nbytes / t / 1e9, 1)}
        rows.append(r)
        print(json.dumps(r), file=sys.stderr, flush=True)

    with torch.cuda.stream(s):
        # configuration 1
        K, N = C.CFG1.K, C.CFG1.N
        S = N // K
        x = [C.CFG1.buffer(r, device=dev) for r in range(K)]
        out = [torch.empty(S, dtype=f32, device=dev) for _ in range(K)]
        ar = [torch.empty(N, dtype=bf, device=dev) for _ in range(K)]
        t = timed(lambda: dpr.dpr_reduce_scatter(x, K, 1, N, out, mode=dpr.RING_FP32, stream=s),
                  2 * K * N + 4 * N)
        row(1, "rs_fp32", 2 * K * N + 4 * N, t)
        t = timed(lambda: dpr.dpr_allreduce(x, K, N, ar, mode=dpr.RING_FP32, stream=s), 4 * K * N)
        row(1, "allreduce", 4 * K * N, t)
        del x, out, ar
        # configuration 2
        K, N = C.CFG2.K, C.CFG2.N
        S = N // K
        x = [C.CFG2.buffer(r, device=dev) for r in range(K)]
        out = [torch.empty(S, dtype=f32, device=dev) for _ in range(K)]
        for mode, name in ((dpr.RING_FP32, "rs_fp32"), (dpr.HOP_BF16, "rs_hop")):
            t = timed(lambda: dpr.dpr_reduce_scatter(x, K, 1, N, out, mode=mode, stream=s),
                      2 * K * N + 4 * N)
            row(2, name, 2 * K * N + 4 * N, t)
        del x, out
        torch.cuda.empty_cache()
        # configuration 3
        cfg = C.CFG3
        K = cfg.K
        numel = [n for *_, n in cfg.arrival_order()]
        bucket_of, offset, bucket_numel = dpr.dpr_bucket_assign(numel, args.bucket_elems,
                                                                pad_to=8 * K)
        grads = [[cfg.grad(r, p, device=dev) for p in range(len(numel))] for r in range(K)]
        part = torch.empty(K, sum(bucket_numel) // K, dtype=f32, device=dev)
        ipg = torch.zeros(K, max(bucket_numel), dtype=bf, device=dev)
        steps = []
        at = 0
        for b, nb in enumerate(bucket_numel):
            ps = [p for p in range(len(numel)) if bucket_of[p] == b]
            plan = dpr.dpr_flatten_plan_create([[grads[r][p] for p in ps] for r in range(K)],
                                               [numel[p] for p in ps], [offset[p] for p in ps],
                                               nb, stream=s)
            views = [ipg[r, :nb] for r in range(K)]
            outs = [part[j, at:at + nb // K] for j in range(K)]
            steps.append((plan, views, outs, nb))
            at += nb // K

        def backward():
            for plan, views, outs, nb in steps:
                dpr.dpr_flatten_bucket(plan, views, stream=s)
                dpr.dpr_reduce_scatter(views, K, 1, nb, outs, mode=dpr.RING_FP32, stream=s)

        total = sum(bucket_numel)
        nbytes = 4 * K * total + 2 * K * total + 4 * total
        t = timed(backward, nbytes)
        row(3, "flatten+rs_fp32 per bucket", nbytes, t, launches=2 * len(steps))
        for plan, *_ in steps:
            plan.close()
        # the same reduction straight from the fragments: no bucket is written or re-read
        fused = []
        for b, nb in enumerate(bucket_numel):
            ps = [p for p in range(len(numel)) if bucket_of[p] == b]
            fplan = dpr.dpr_fragments_plan_create([[grads[r][p] for p in ps] for r in range(K)],
                                                  [numel[p] for p in ps], [offset[p] for p in ps],
                                                  nb, stream=s)
            fused.append(fplan)
        outs_by_bucket = []
        at = 0
        for nb in bucket_numel:
            outs_by_bucket.append([part[j, at:at + nb // K] for j in range(K)])
            at += nb // K

        def backward_fused():
            for fplan, outs in zip(fused, outs_by_bucket):
                dpr.dpr_reduce_scatter_fragments(fplan, outs, mode=dpr.RING_FP32, stream=s)

        fbytes = 2 * K * sum(numel) + 4 * total
        t_f = timed(backward_fused, fbytes)
        row(3, "rs_fp32 from fragments per bucket", fbytes, t_f, launches=len(fused))
        prev = dpr.dpr_set_programmatic_launch(False)
        try:
            t_p = timed(backward_fused, fbytes)
        finally:
            dpr.dpr_set_programmatic_launch(prev)
        row(3, "rs_fp32 from fragments per bucket, plain launches", fbytes, t_p,
            launches=len(fused))

        def backward_batched():
            dpr.dpr_reduce_scatter_fragments_batch(fused, outs_by_bucket, mode=dpr.RING_FP32,
                                                   stream=s)

        t_b = timed(backward_batched, fbytes)
        row(3, "rs_fp32 from fragments, all buckets in one batched call", fbytes, t_b,
            launches=len(fused))
        s.synchronize()
        graph_b = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_b, stream=s):
            backward_batched()

        def replay_b():
            with torch.cuda.stream(s):
                graph_b.replay()

        t_bg = timed(replay_b, fbytes)
        row(3, "rs_fp32 from fragments, one batched call, CUDA graph", fbytes, t_bg,
            launches=len(fused))
        del graph_b
        # the 42 launches captured once in a CUDA graph and replayed
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            backward_fused()
        def replay():
            with torch.cuda.stream(s):
                graph.replay()

        t_g = timed(replay, fbytes)
        row(3, "rs_fp32 from fragments per bucket, CUDA graph", fbytes, t_g, launches=len(fused))
        del graph
        for fplan in fused:
            fplan.close()
        del steps, grads, part, ipg
        torch.cuda.empty_cache()
        # configuration 4
        K, N = C.CFG4.K, C.CFG4.N
        S = N // K
        shards = [C.cfg4_shard(j, device=dev) for j in range(K)]
        full = [torch.empty(N, dtype=bf, device=dev) for _ in range(K)]
        t = timed(lambda: dpr.dpr_allgather(shards, K, N, full, stream=s), 2 * N + 2 * K * N)
        row(4, "allgather", 2 * N + 2 * K * N, t)
        del shards, full
        torch.cuda.empty_cache()
    peak, kind = load_peaks()
    head = [r for r in rows if r["config"] == 3][0]
    line = {"metric": METRIC, "value": head["gbs"], "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "config": {"workload": "configs_1_to_4", "bucket_elems": args.bucket_elems},
            "value_is": "configuration 3: gather + reduce-scatter of every bucket of one backward",
            "peak": peak, "peak_kind": kind, "table": rows}
    print(json.dumps(line), flush=True)
    return 0


def run_fragments_bench(args):
    """The bench's 1 GiB bucket (K=8, 32 fragmented 4096x4096 gradients per
    rank) reduce-scattered two ways: gathered into the flat bucket, then
    reduce-scattered (two launches), and straight from the fragments (one
    launch).  Both give the same bits; the line reports both times."""
    import torch
    import gradient_reduction_gb300 as dpr
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = torch.cuda.Stream(device=dev)
    wl = Workload(dev, s, args.n_per_rank)
    K, N, P, F = wl.K, wl.N, wl.P, wl.F
    S = N // K
    timed = LaunchTimer(s, args.steps, args.warmup)
    with torch.cuda.stream(s):
        out = list(torch.empty(K, S, dtype=torch.float32, device=dev).unbind(0))
        ref = list(torch.empty(K, S, dtype=torch.float32, device=dev).unbind(0))
        with dpr.dpr_fragments_plan_create(wl.frags, [F] * P, [p * F for p in range(P)], N,
                                           stream=s) as plan:
            def gather_then_rs():
                dpr.dpr_flatten_bucket(wl.plan, wl.ipg1, stream=s)
                dpr.dpr_reduce_scatter(wl.ipg1, K, 1, N, ref, stream=s)

            def from_fragments():
                dpr.dpr_reduce_scatter_fragments(plan, out, stream=s)

            t2 = timed(gather_then_rs, 1 << 30)
            t1 = timed(from_fragments, 1 << 30)
            s.synchronize()
            same = all(torch.equal(a.view(torch.int32), b.view(torch.int32)) for a, b in zip(out, ref))
    wl.plan.close()
    b1 = 2 * K * N + 4 * N
    b2 = 4 * K * N + 2 * K * N + 4 * N
    peak, kind = load_peaks()
    line = {"metric": METRIC, "value": round(b1 / t1 / 1e9, 1), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "config": {"workload": "fragments_k8_1GiB", "K": K, "elements_per_rank": N,
                       "fragments_per_rank": f"{P} x (4096x4096)"},
            "value_is": "reduce-scatter straight from the fragments, GB/s of its algorithmic bytes",
            "from_fragments": {"ms": round(t1 * 1e3, 3), "bytes": b1, "launches": 1},
            "gather_then_reduce_scatter": {"ms": round(t2 * 1e3, 3), "bytes": b2, "launches": 2},
            "speedup": round(t2 / t1, 3), "bit_identical": same, "peak": peak, "peak_kind": kind}
    print(json.dumps(line), flush=True)
    return 0 if same else 1


def run_sequence_bench(args):
    """A backward pass's worth of small buckets issued back to back: 64
    buckets of 4 MiB per rank at K=8 (2 micro-batches, ring fp32, x1/8),
    reduce-scattered with plain launches, with programmatic dependent launches
    (one call per bucket), as persistent requests and in one batched call;
    then the same 64 buckets all-gathered the same four ways.  Each figure is
    the sequence's algorithmic bytes over its CUDA-event time, averaged over
    --steps sequences (4.8 GB per reduce-scatter sequence, far larger than
    L2, so no flush is needed).  The three reduce-scatter forms must give the
    same bits."""
    import torch
    import gradient_reduction_gb300 as dpr
    from workloads import synthetic as syn
    K, M, nb = 8, 2, 64
    N = (4 << 20) // 2
    S = N // K
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = torch.cuda.Stream(device=dev)
    bf, f32 = torch.bfloat16, torch.float32
    with torch.cuda.stream(s):
        x = torch.empty(nb, M * K, N, dtype=bf, device=dev)
        for i in range(M * K):      # 16 distinct rank buffers, copied into every bucket
            syn.gauss_bf16(0, N, syn.stream_key(args.seed, i % K, i // K), 1e-3, device=dev,
                           out=x[0, i])
        x[1:].copy_(x[0].expand(nb - 1, M * K, N))
        ins = [x[b] for b in range(nb)]              # one [M*K, N] tensor per bucket
        outs = {k: torch.empty(nb, K, S, dtype=f32, device=dev) for k in ("plain", "pdl", "batch")}
        out_l = {k: [v[b] for b in range(nb)] for k, v in outs.items()}   # [K, S] per bucket
        ins_list = [list(x[b].unbind(0)) for b in range(nb)]              # the list form
        outs_list = [list(outs["plain"][b].unbind(0)) for b in range(nb)]
        full = torch.empty(nb, K, N, dtype=bf, device=dev)
        full_l = [full[b] for b in range(nb)]
        # shard j of bucket b is chunk j of rank j's buffer: rows N + S elements apart
        shards_all = torch.as_strided(x, (nb, K, S), (M * K * N, N + S, 1))
        shards = [shards_all[b] for b in range(nb)]
    s.synchronize()

    def rs_single(key):
        for b in range(nb):
            dpr.dpr_reduce_scatter(ins[b], K, M, N, out_l[key][b], mode=dpr.RING_FP32, stream=s)

    def rs_batch():
        dpr.dpr_reduce_scatter_batch(x, K, M, [N] * nb, outs["batch"], mode=dpr.RING_FP32,
                                     stream=s)

    # persistent requests: every bucket's call checked once, started every step
    reqs = [dpr.dpr_reduce_scatter_init(ins[b], K, M, N, out_l["pdl"][b], mode=dpr.RING_FP32)
            for b in range(nb)]

    def rs_requests():
        for rq in reqs:
            rq.start(s)

    def host_us(fn, calls):
        """Host time per call of fn (no synchronisation inside the loop)."""
        s.synchronize()
        t0 = time.perf_counter()
        fn()
        t1 = time.perf_counter()
        s.synchronize()
        return (t1 - t0) / calls * 1e6

    def ag_single():
        for b in range(nb):
            dpr.dpr_allgather(shards[b], K, N, full_l[b], stream=s)

    ag_reqs = [dpr.dpr_allgather_init(shards[b], K, N, full_l[b]) for b in range(nb)]

    def ag_requests():
        for rq in ag_reqs:
            rq.start(s)

    def ag_batch():
        dpr.dpr_allgather_batch(shards_all, K, [N] * nb, full, stream=s)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        s.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(args.steps):
            fn()
        e.record(s)
        s.synchronize()
        return a.elapsed_time(e) / 1e3 / args.steps

    def graphed(fn):
        """fn's launches captured once in a CUDA graph (programmatic launches
        become programmatic edges), so the host's per-call cost drops out."""
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()

        def replay():
            with torch.cuda.stream(s):
                g.replay()
        return replay, g

    rs_bytes = nb * (2 * M * K * N + 4 * N)
    ag_bytes = nb * (2 * N + 2 * K * N)
    graphs = []
    prev = dpr.dpr_set_programmatic_launch(False)
    try:
        t_rs_plain = timed(lambda: rs_single("plain"))
        t_ag_plain = timed(ag_single)
        r, g = graphed(lambda: rs_single("plain"))
        graphs.append(g)
        t_rs_plain_g = timed(r)
        r, g = graphed(ag_single)
        graphs.append(g)
        t_ag_plain_g = timed(r)
    finally:
        dpr.dpr_set_programmatic_launch(prev)
    dpr.dpr_set_programmatic_launch(True)
    t_rs_pdl = timed(lambda: rs_single("pdl"))
    t_rs_req = timed(rs_requests)
    t_rs_batch = timed(rs_batch)
    t_ag_pdl = timed(ag_single)
    t_ag_req = timed(ag_requests)
    r, g = graphed(lambda: rs_single("pdl"))
    graphs.append(g)
    t_rs_pdl_g = timed(r)
    r, g = graphed(rs_batch)
    graphs.append(g)
    t_rs_batch_g = timed(r)
    r, g = graphed(ag_single)
    graphs.append(g)
    t_ag_pdl_g = timed(r)
    t_ag_batch = timed(ag_batch)
    r, g = graphed(ag_batch)
    graphs.append(g)
    t_ag_batch_g = timed(r)
    dpr.dpr_set_programmatic_launch(prev)
    same = all(torch.equal(outs["plain"].view(torch.int32), outs[k].view(torch.int32))
               for k in ("pdl", "batch"))
    # the binding's host cost per call, with rank buffers passed as lists of tensors and
    # as one stacked tensor per bucket
    host = {
        "list_args_us_per_call": round(host_us(lambda: [
            dpr.dpr_reduce_scatter(ins_list[b], K, M, N, outs_list[b], stream=s)
            for b in range(nb)], nb), 2),
        "stacked_args_us_per_call": round(host_us(lambda: rs_single("plain"), nb), 2),
        "batched_call_us_per_bucket": round(host_us(rs_batch, nb), 2),
        "persistent_request_us_per_start": round(host_us(rs_requests, nb), 2),
    }
    for rq in reqs + ag_reqs:
        rq.close()
    peak, kind = load_peaks()

    def fig(nbytes, t):
        return {"ms": round(t * 1e3, 4), "gbs": round(nbytes / t / 1e9, 1),
                "frac_of_peak": round(nbytes / t / 1e9 / peak, 4),
                "us_per_bucket": round(t / nb * 1e6, 2)}

    line = {"metric": METRIC, "value": round(rs_bytes / t_rs_batch / 1e9, 1), "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "config": {"workload": "sequence_k8_64x4MiB", "K": K, "buckets": nb,
                       "bytes_per_rank_per_bucket": 2 * N, "micro_batches": M,
                       "l2": "4.8 GB per sequence, far larger than L2; no flush needed"},
            "value_is": "64 reduce-scatters of 4 MiB per rank in one batched call, GB/s",
            "peak": peak, "peak_kind": kind,
            "reduce_scatter": {"plain_launches": fig(rs_bytes, t_rs_plain),
                               "programmatic_launches": fig(rs_bytes, t_rs_pdl),
                               "persistent_requests": fig(rs_bytes, t_rs_req),
                               "one_batched_call": fig(rs_bytes, t_rs_batch),
                               "graph_plain_launches": fig(rs_bytes, t_rs_plain_g),
                               "graph_programmatic_launches": fig(rs_bytes, t_rs_pdl_g),
                               "graph_one_batched_call": fig(rs_bytes, t_rs_batch_g),
                               "bytes": rs_bytes, "bit_identical": same},
            "allgather": {"plain_launches": fig(ag_bytes, t_ag_plain),
                          "programmatic_launches": fig(ag_bytes, t_ag_pdl),
                          "persistent_requests": fig(ag_bytes, t_ag_req),
                          "one_batched_call": fig(ag_bytes, t_ag_batch),
                          "graph_plain_launches": fig(ag_bytes, t_ag_plain_g),
                          "graph_programmatic_launches": fig(ag_bytes, t_ag_pdl_g),
                          "graph_one_batched_call": fig(ag_bytes, t_ag_batch_g),
                          "bytes": ag_bytes},
            "host_cost": host,
            "host_note": "eager rows include the Python binding's per-call cost (one call per "
                         "bucket with stacked-tensor arguments, except the batched call); graph "
                         "rows replay the same launches from a CUDA graph"}
    del graphs
    print(json.dumps(line), flush=True)
    return 0 if same else 1


def run_point_bench(args):
    """One point chosen on the command line: the reduce-scatter (--mode,
    --micro), all-gather and all-reduce at --K ranks and --bytes-per-rank,
    seeded gradients ~N(0, 1e-3), timed like the sweep."""
    import torch
    import gradient_reduction_gb300 as dpr
    from workloads import synthetic as syn
    K, M = args.K, args.micro
    N = args.bytes_per_rank // 2
    if N <= 0 or N % K:
        raise SystemExit("--bytes-per-rank / 2 must be a positive multiple of --K")
    S = N // K
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = torch.cuda.Stream(device=dev)
    timed = LaunchTimer(s, args.steps, args.warmup)
    mode = dpr.RING_FP32 if args.mode == "ring_fp32" else dpr.HOP_BF16
    with torch.cuda.stream(s):
        x = torch.empty(M * K, N, dtype=torch.bfloat16, device=dev)
        for i in range(M * K):
            syn.gauss_bf16(0, N, syn.stream_key(args.seed, i % K, i // K), 1e-3, device=dev,
                           out=x[i])
        xs = list(x.unbind(0))
        out = list(torch.empty(K, S, dtype=torch.float32, device=dev).unbind(0))
        rows = {}
        b_rs = 2 * M * K * N + 4 * N
        t = timed(lambda: dpr.dpr_reduce_scatter(xs, K, M, N, out, mode=mode, stream=s), b_rs)
        rows["reduce_scatter"] = {"bytes": b_rs, "us": round(t * 1e6, 2), "gbs": round(b_rs / t / 1e9, 1)}
        del out
        y = list(torch.empty(K, N, dtype=torch.bfloat16, device=dev).unbind(0))
        b_ag = 2 * N + 2 * K * N
        shards = [xs[j][:S] for j in range(K)]
        t = timed(lambda: dpr.dpr_allgather(shards, K, N, y, stream=s), b_ag)
        rows["allgather"] = {"bytes": b_ag, "us": round(t * 1e6, 2), "gbs": round(b_ag / t / 1e9, 1)}
        b_ar = 4 * K * N
        t = timed(lambda: dpr.dpr_allreduce(xs[:K], K, N, y, mode=mode, stream=s), b_ar)
        rows["allreduce"] = {"bytes": b_ar, "us": round(t * 1e6, 2), "gbs": round(b_ar / t / 1e9, 1)}
    peak, kind = load_peaks()
    line = {"metric": METRIC, "value": rows["reduce_scatter"]["gbs"], "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "config": {"workload": "point", "K": K, "bytes_per_rank": args.bytes_per_rank,
                       "mode": args.mode, "micro_batches": M, "seed": args.seed},
            "value_is": "the reduce-scatter's GB/s", "peak": peak, "peak_kind": kind,
            "ops": rows}
    print(json.dumps(line), flush=True)
    return 0


def run_sweep_bench(args):
    """Configuration 5's sweep: effective GB/s of the reduce-scatter (both
    modes, 2 micro-batches, and 1 micro-batch beside them), all-gather and
    all-reduce for K in
    {2,4,8,16,64} and 1 KiB .. 1 GiB per rank.  Each figure is algorithmic
    bytes over the average launch time (CUDA events); small sizes show the
    launch-bound regime."""
    import torch
    import gradient_reduction_gb300 as dpr
    from workloads import configs as C
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s = torch.cuda.Stream(device=dev)

    timed = LaunchTimer(s, args.steps, args.warmup)

    table = []
    for K, nbytes in C.cfg5_points():
        N = nbytes // 2
        S = N // K
        row = {"K": K, "bytes_per_rank": nbytes}
        gen = torch.Generator(device=dev)
        gen.manual_seed(C.BASE_SEED + 5)            # N(0, 1e-3), seeded, drawn on the device
        x = torch.empty(2 * K, N, dtype=torch.bfloat16, device=dev).normal_(0.0, 1e-3,
                                                                             generator=gen)
        xs = list(x.unbind(0))
        out = torch.empty(K, S, dtype=torch.float32, device=dev)
        outs = list(out.unbind(0))
        for mode, name in ((dpr.RING_FP32, "rs_fp32_m2"), (dpr.HOP_BF16, "rs_hop_m2")):
            t = timed(lambda: dpr.dpr_reduce_scatter(xs, K, 2, N, outs, mode=mode, stream=s),
                      4 * K * N + 4 * N)
            row[name] = round((4 * K * N + 4 * N) / t / 1e9, 1)
        for mode, name in ((dpr.RING_FP32, "rs_fp32_m1"), (dpr.HOP_BF16, "rs_hop_m1")):
            t = timed(lambda: dpr.dpr_reduce_scatter(xs[:K], K, 1, N, outs, mode=mode, stream=s),
                      2 * K * N + 4 * N)
            row[name] = round((2 * K * N + 4 * N) / t / 1e9, 1)
        del xs, x, out, outs
        torch.cuda.empty_cache()
        x = torch.empty(K, N, dtype=torch.bfloat16, device=dev).normal_(0.0, 1e-3, generator=gen)
        y = torch.empty(K, N, dtype=torch.bfloat16, device=dev)
        xs, ys = list(x.unbind(0)), list(y.unbind(0))
        t = timed(lambda: dpr.dpr_allreduce(xs, K, N, ys, stream=s), 4 * K * N)
        row["allreduce"] = round(4 * K * N / t / 1e9, 1)
        shards = [xs[j][:S] for j in range(K)]
        t = timed(lambda: dpr.dpr_allgather(shards, K, N, ys, stream=s), 2 * N + 2 * K * N)
        row["allgather"] = round((2 * N + 2 * K * N) / t / 1e9, 1)
        del xs, ys, x, y, shards
        torch.cuda.empty_cache()
        table.append(row)
        print(json.dumps(row), file=sys.stderr, flush=True)
    peak, kind = load_peaks()
    head = [r for r in table if r["K"] == 8 and r["bytes_per_rank"] == 1 << 30][0]
    line = {"metric": METRIC, "value": head["rs_fp32_m2"], "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "config": {"workload": "cfg5_sweep", "K": [2, 4, 8, 16, 64],
                       "bytes_per_rank": "1 KiB .. 1 GiB by 4x", "micro_batches": 2},
            "value_is": "reduce-scatter ring fp32 M=2 at K=8, 1 GiB per rank",
            "peak": peak, "peak_kind": kind, "table": table}
    print(json.dumps(line), flush=True)
    return 0


def run_pipeline_bench(args):
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pb = PipelineBackward(dev)
    budgets = (0, 608, 304, 152, 64)
    keys = ["serial"] + [f"{pol}@{mb}" for mb in budgets for pol in ("reverse_wait", "per_buffer")]

    def run(key):
        if key == "serial":
            return pb.run("serial")
        pol, mb = key.split("@")
        return pb.run(pol, int(mb))
    for key in keys:
        for _ in range(args.warmup):
            run(key)
    times = {key: [] for key in keys}
    for _ in range(args.steps):
        for key in keys:
            times[key].append(run(key))
    med = {key: statistics.median(v) for key, v in times.items()}
    parts = pb.run_parts()
    pb.close()
    best = min((k for k in keys if k.startswith("per_buffer")), key=lambda k: med[k])
    mb = best.split("@")[1]
    med["per_buffer"] = med[best]
    med["reverse_wait"] = med[f"reverse_wait@{mb}"]
    line = {
        "metric": "bucket pipeline: simulated backward time per policy", "unit": "ms",
        "value": round(med["per_buffer"] * 1e3, 3), "higher_is_better": False,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "config": {"workload": "bucket_pipeline_k8_16_buckets",
                   "buckets": "16, alternately 3*2^23 and 2^23 bf16 elements per rank, K=8",
                   "compute": "bf16 4096^3 matmuls on the compute stream, alternately 1 and 3 per bucket",
                   "buffers": 2},
        "ms": {k: round(v * 1e3, 3) for k, v in med.items()},
        "reduction_block_budget": int(mb),
        "alone_ms": {k: round(v * 1e3, 3) for k, v in parts.items()},
        "gather_reduce_gbs_serial": round(pb.bytes / parts["reduce"] / 1e9, 1),
        "per_buffer_vs_reverse_wait": round(med["reverse_wait"] / med["per_buffer"], 3),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_device(args, rank, world, local_rank):
    import torch
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    if args.workload == "zero3_per_param":
        wl = Zero3Workload(dev, stream, args.z3_layers)
        kernels = (args.only,) if args.only else Z3_KERNELS
    elif args.workload == "bf16_partition":
        wl = Bf16PartitionWorkload(dev, stream, args.n_per_rank)
        kernels = (args.only,) if args.only else BF16_KERNELS
    else:
        wl = Workload(dev, stream, args.n_per_rank)
        kernels = (args.only,) if args.only else STEP_KERNELS
    step_bytes = sum(wl.bytes[k] for k in kernels)
    for _ in range(args.warmup):
        wl.step(kernels)
    stream.synchronize()
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            wl.step(kernels)
        for _ in range(args.warmup):
            graph.replay()
        stream.synchronize()
    barrier(dev)
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank).start() if rank == 0 else None
    events = []
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            with torch.cuda.stream(stream):
                graph.replay()
        else:
            wl.step(kernels, events)
    t1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier(dev)
    clk = clocks.stop() if clocks else None
    elapsed = t0.elapsed_time(t1) / 1e3
    max_elapsed = max_over_ranks(elapsed, dev)
    launches = len(events)
    if graph is not None:
        # per-kernel times come from a short eager pass after the timed region
        launches = args.steps * len(kernels)
        for _ in range(min(args.steps, 20)):
            wl.step(kernels, events)
        stream.synchronize()
    per = {}
    for name, a, b in events:
        per.setdefault(name, []).append(a.elapsed_time(b) / 1e3)
    kernels_out = {}
    for name, ts in per.items():
        avg = sum(ts) / len(ts)
        kernels_out[name] = {"bytes_per_launch": wl.bytes[name], "avg_ms": avg * 1e3,
                             "gbs": wl.bytes[name] / avg / 1e9, "launches": len(ts),
                             "time_share": sum(ts) / sum(sum(v) for v in per.values())}
        if name in STEP_KERNELS:
            bb = ring_busbw(name, wl.K, wl.N, avg)
            if bb is not None:
                kernels_out[name]["busbw_ring_equivalent_gbs"] = bb
    headline = None
    if not args.only and args.workload == "zero_bucket":
        headline = time_headline_ops(wl, max(20, min(args.steps, 30)), 3)
    e2e = None
    if not args.no_e2e and not args.only and args.workload == "zero_bucket":
        e2e = run_e2e(wl, args, step_bytes)
    return {"elapsed": elapsed, "max_elapsed": max_elapsed, "step_bytes": step_bytes,
            "kernels": kernels_out, "clocks": clk, "e2e": e2e, "wl": wl,
            "launches": launches, "headline": headline}


NOMINAL_HBM_GBS = 7900.0    # GB300 HBM3e data-sheet bandwidth, for the second fraction


def time_headline_ops(wl, launches: int, warmup: int):
    """The metric's own operations at K=8, 1 GiB per rank, each timed alone
    after the step's timed region: the reduce-scatter of one micro-batch in
    both summation modes and the all-gather, `launches` back-to-back launches
    each between two CUDA events on the launching stream (inputs of 8 GiB, far
    larger than L2).  Each figure is given against the measured copy peak and
    against the data-sheet HBM bandwidth."""
    import torch
    dpr, K, N, s = wl.dpr, wl.K, wl.N, wl.stream
    peak, kind = load_peaks()
    ops = {
        "rs_ring_fp32_m1": (lambda: dpr.dpr_reduce_scatter(wl.ipg0, K, 1, N, wl.part_f32,
                                                           mode=dpr.RING_FP32, stream=s),
                            2 * K * N + 4 * N, "rs_fp32_m1"),
        "rs_hop_bf16_m1": (lambda: dpr.dpr_reduce_scatter(wl.ipg0, K, 1, N, wl.part_f32,
                                                          mode=dpr.HOP_BF16, stream=s),
                           2 * K * N + 4 * N, "rs_hop_m1"),
        "allgather": (lambda: dpr.dpr_allgather(wl.shards, K, N, wl.params, stream=s),
                      2 * N + 2 * K * N, "allgather"),
    }
    out = {}
    for name, (fn, nbytes, key) in ops.items():
        for _ in range(warmup):
            fn()
        s.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(launches):
            fn()
        b.record(s)
        s.synchronize()
        t = a.elapsed_time(b) / 1e3 / launches
        gbs = nbytes / t / 1e9
        tr = NCU_TRAFFIC.get(key)
        out[name] = {"bytes_per_launch": nbytes, "avg_ms": round(t * 1e3, 4),
                     "launches": launches, "gbs": round(gbs, 1),
                     "frac_of_measured_peak": round(gbs / peak, 4),
                     "frac_of_nominal_peak": round(gbs / NOMINAL_HBM_GBS, 4),
                     "traffic": tr["bytes"] if tr and tr["src_sha"] == kernel_src_sha(key)
                     and wl.N == 1 << 29 else None}
    out["peaks"] = {"measured_gbs": peak, "measured_kind": kind,
                    "nominal_gbs": NOMINAL_HBM_GBS,
                    "nominal_is": "GB300 HBM3e data-sheet bandwidth"}
    return out


def run_e2e(wl, args, step_bytes):
    """End-to-end steps through the public API from host memory.

    Every timed step copies its inputs (gradient fragments, the other micro-
    batch's bucket, the fp32 partition it accumulates into, the parameter
    shards) from pinned host buffers, runs the five launches, and reads every
    result (both fp32 partitions, the all-gathered parameters, the all-reduced
    bucket) back into pinned host buffers.  Copies in, kernels and copies out
    run on three streams over two device buffer sets, so step i+1's inputs
    and step i-1's results cross the host link while step i computes; each
    step still moves all of its own bytes inside the timed region."""
    import torch
    dev = wl.dev
    _, world, _ = dist_env()
    pinned = sum(t.numel() * t.element_size() for t in wl.inputs() + wl.outputs())
    local = int(os.environ.get("LOCAL_WORLD_SIZE", world))
    # every rank of this host pins its own copy: all ranks run the e2e steps,
    # or none does (they meet in a collective at the end)
    fits = host_available_bytes() >= local * pinned * 1.1 + (8 << 30)
    h_in = h_out = None
    if fits:
        try:
            h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in wl.inputs()]
            h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in wl.outputs()]
        except RuntimeError:
            fits = False
    if not all_ranks(fits, dev):
        h_in = h_out = None
        torch.cuda.empty_cache()
        return {"value": None, "unit": UNIT,
                "skipped": f"{local} rank(s) on this host need {local * pinned / 1e9:.0f} GB of "
                           "pinned host memory for the step's inputs and results"}
    # two buffer sets (a third one measured no faster on GB300: the host link,
    # not the set reuse, bounds the step)
    nsets = 2
    sets = [wl] + [Workload(dev, wl.stream, args.n_per_rank, fill=False) for _ in range(nsets - 1)]
    for h, d in zip(h_in, wl.inputs()):
        h.copy_(d)
    torch.cuda.synchronize()
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    s_in, s_out, s_comp = (torch.cuda.Stream(device=dev) for _ in range(3))
    for w in sets:
        w.stream = s_comp
    n = args.e2e_steps
    in_done = [torch.cuda.Event() for _ in range(nsets)]
    comp_done = [None] * nsets
    out_done = [None] * nsets

    def run(steps):
        for i in range(steps):
            b = i % nsets
            w = sets[b]
            # copies in: wait until step i-2 has finished with this set
            if comp_done[b] is not None:
                s_in.wait_event(comp_done[b])
            if out_done[b] is not None:
                s_in.wait_event(out_done[b])
            with torch.cuda.stream(s_in):
                for d, h in zip(w.inputs(), h_in):
                    d.copy_(h, non_blocking=True)
            in_done[b].record(s_in)
            s_comp.wait_event(in_done[b])
            w.step(STEP_KERNELS)
            ev = torch.cuda.Event()
            ev.record(s_comp)
            comp_done[b] = ev
            s_out.wait_event(ev)
            with torch.cuda.stream(s_out):
                for h, d in zip(h_out, w.outputs()):
                    h.copy_(d, non_blocking=True)
            ev2 = torch.cuda.Event()
            ev2.record(s_out)
            out_done[b] = ev2

    run(nsets)                               # warm-up of every buffer set
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    s_comp.wait_event(t0)
    s_out.wait_event(t0)
    run(n)
    s_in.wait_event(out_done[(n - 1) % nsets])
    t1.record(s_in)
    torch.cuda.synchronize()
    el = t0.elapsed_time(t1) / 1e3
    el = max_over_ranks(el, dev)
    for w in sets[1:]:
        w.plan.close()
    for w in sets:
        w.stream = wl.stream
    return {"value": round(job_value(step_bytes, n, world, el), 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "ms_per_step": round(el / n * 1e3, 3),
            "pipelining": "copies in / kernels / copies out on three streams, two buffer sets"}


# ---- CPU oracle baseline ---------------------------------------------------------

class OracleSample:
    """The bench workload scaled down for the CPU oracle: same K and fragment
    count, N_s elements per rank."""

    ARRAYS = ("frags", "ipg0", "part", "shards")

    def __init__(self, n_per_rank: int, arrays: dict | None = None):
        from workloads import configs as C
        w = C.BENCH
        self.K = K = w.K
        self.P = P = w.n_frag
        self.N = N = n_per_rank
        self.F = F = N // P
        self.S = S = N // K
        if arrays is None:
            from workloads import synthetic as syn
            bits = syn.bf16_bits
            import numpy as np
            arrays = {
                "frags": np.stack([np.stack([bits(w.dist.fill(0, F, w.frag_key(r, p)))
                                             for p in range(P)]) for r in range(K)]),
                "ipg0": np.stack([bits(w.dist.fill(0, N, w.micro0_key(r))) for r in range(K)]),
                "part": np.stack([syn.gauss_bf16(0, S, w.prev_grad_key(j), 1e-3).float().numpy()
                                  for j in range(K)]),
                "shards": np.stack([bits(w.param_dist.fill(j * S, S, w.param_key()))
                                    for j in range(K)]),
            }
        self.arrays = arrays
        self.frags = [list(arrays["frags"][r]) for r in range(K)]
        self.ipg0 = list(arrays["ipg0"])
        self.part = list(arrays["part"])
        self.shards = list(arrays["shards"])
        self.bytes = 4 * K * N + (4 * K * N + 4 * N) + (4 * K * N + 8 * N) + (2 * N + 2 * K * N) \
            + 4 * K * N

    def save(self, folder: str):
        import numpy as np
        for name in self.ARRAYS:
            np.save(os.path.join(folder, name + ".npy"), self.arrays[name])

    @classmethod
    def load(cls, folder: str, n_per_rank: int):
        import numpy as np
        return cls(n_per_rank, {name: np.load(os.path.join(folder, name + ".npy"))
                                for name in cls.ARRAYS})

    def step(self, impl: str = "numpy"):
        """The five steps through the numpy simulation (oracle/ring.py,
        oracle/flatten.py) or the C simulation (oracle/ring_sim.c)."""
        if impl == "c":
            from oracle import ring_c as ring
            flatten_bucket = ring.flatten_bucket
        else:
            from oracle import flatten as ofl
            from oracle import ring
            flatten_bucket = ofl.flatten_bucket
        K, P, F, N = self.K, self.P, self.F, self.N
        flat = flatten_bucket(self.frags, [F] * P, [p * F for p in range(P)], N)
        x = self.ipg0 + flat
        ring.reduce_scatter(x, K, 2, ring.RING_FP32, 1.0 / K)
        ring.reduce_scatter(x, K, 2, ring.HOP_BF16, 1.0 / K, out_init=self.part)
        ring.allgather(self.shards, K)
        ring.allreduce(flat, K, ring.RING_FP32, 1.0 / K)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _slab_worker(folder, n, barrier, cmds, impl):
    """One oracle process: every element position of the workload is
    independent, so each core runs the whole oracle on its own slab.  Waits at
    the barrier, runs the commanded number of passes, waits again."""
    smp = OracleSample.load(folder, n)
    smp.step(impl)                              # warm-up
    while True:
        passes = cmds.get()
        if passes is None:
            return
        barrier.wait()
        for _ in range(passes):
            smp.step(impl)
        barrier.wait()


class OracleSlabPool:
    """`cores` spawned processes, each holding one slab (a K=8 sample of n
    elements per rank) of the bench workload and running the oracle on it
    (impl "numpy" or "c", one thread each).  run(p) times p passes of every
    process, from a common start to the last one's end.  Processes are
    started with spawn: none inherits the parent's CUDA state."""

    def __init__(self, n: int, cores: int, impl: str = "numpy"):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.n, self.cores, self.impl = n, cores, impl
        if impl == "c":
            from oracle import ring_c
            ring_c.build()          # once, before the processes load it
        self.folder = tempfile.mkdtemp(prefix="oracle_slab_")
        smp = OracleSample(n)
        smp.save(self.folder)
        self.bytes = smp.bytes
        del smp
        self.barrier = ctx.Barrier(cores + 1)
        self.cmds = [ctx.Queue() for _ in range(cores)]
        env_before = os.environ.get("OMP_NUM_THREADS")
        os.environ["OMP_NUM_THREADS"] = "1"     # one thread per process
        try:
            self.procs = [ctx.Process(target=_slab_worker,
                                      args=(self.folder, n, self.barrier, q, impl),
                                      daemon=True)
                          for q in self.cmds]
            for pr in self.procs:
                pr.start()
        finally:
            if env_before is None:
                os.environ.pop("OMP_NUM_THREADS", None)
            else:
                os.environ["OMP_NUM_THREADS"] = env_before

    def run(self, passes: int) -> float:
        for q in self.cmds:
            q.put(passes)
        self.barrier.wait(timeout=600)
        t0 = time.perf_counter()
        self.barrier.wait(timeout=600)
        return time.perf_counter() - t0

    def close(self):
        import shutil
        for q in self.cmds:
            q.put(None)
        for pr in self.procs:
            pr.join(timeout=30)
            if pr.is_alive():
                pr.kill()
        shutil.rmtree(self.folder, ignore_errors=True)


def time_oracle(n_per_rank: int, min_seconds: float, min_steps: int = 1):
    smp = OracleSample(n_per_rank)
    smp.step()     # warm-up
    steps, t0 = 0, time.perf_counter()
    while steps < min_steps or time.perf_counter() - t0 < min_seconds:
        smp.step()
        steps += 1
    el = time.perf_counter() - t0
    return smp, steps, el


def time_pool(n: int, cores: int, impl: str, seconds: float):
    """GB/s of `cores` slab processes running the oracle `impl` for about
    `seconds`, with the passes and the time taken."""
    pool = OracleSlabPool(n, cores, impl)
    try:
        t1 = pool.run(1)
        passes = max(1, round(seconds / t1))
        el = pool.run(passes)
    finally:
        pool.close()
    return pool.bytes * cores * passes / el / 1e9, passes, el


def cpu_baseline(args):
    """The oracle on every host core, one slab per process: the C simulation
    (the line's value) and the numpy simulation, with the numpy single-process
    figure beside them."""
    n = 1 << 20
    smp, steps1, el1 = time_oracle(n, args.cpu_seconds / 4)
    one = smp.bytes * steps1 / el1 / 1e9
    del smp
    cores = host_cores()
    value, passes, el = time_pool(n, cores, "c", args.cpu_seconds / 4)
    c_one, c_passes1, c_el1 = time_pool(n, 1, "c", args.cpu_seconds / 4)
    np_value, np_passes, np_el = time_pool(n, cores, "numpy", args.cpu_seconds / 4)
    return {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "oracle": "C ring simulation (oracle/ring_sim.c, -O2, one thread per process)",
            "single_core_value": round(c_one, 4),
            "numpy_value": round(np_value, 4), "numpy_single_core_value": round(one, 4),
            "sample": f"K=8, the same five steps; {cores} processes, each running the oracle "
                      f"on its own slab of {n} elements per rank (32 fragments of {n // 32}): "
                      f"C simulation {passes} passes in {el:.1f} s, numpy simulation "
                      f"{np_passes} passes in {np_el:.1f} s; one process alone: C "
                      f"{c_passes1} passes in {c_el1:.1f} s, numpy {steps1} passes in "
                      f"{el1:.1f} s"}


def common_config(world):
    return {"workload": "zero_bucket_k8_1GiB", "K": 8, "elements_per_rank": 1 << 29,
            "bytes_per_rank": 1 << 30, "fragments_per_rank": "32 x (4096x4096)",
            "micro_batches": 2,
            "step": "flatten + RS(ring_fp32,M=2) + RS(hop_bf16,M=2,accumulate) + AG + AR",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU, 8 simulated ranks",
            "l2": "inputs (45 GiB resident) far larger than L2; no flush needed"}


def run_reference(args):
    """The reference arm: the oracle (the C simulation) on every host core,
    one slab per process, each step one pass of every process over its slab."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    n = 1 << 20          # per process, as in the CPU baseline of the bench line
    cores = host_cores()
    pool = OracleSlabPool(n, cores, "c")
    try:
        for _ in range(args.warmup):
            pool.run(1)
        el = sum(pool.run(1) for _ in range(args.steps))
    finally:
        pool.close()
    value = pool.bytes * cores * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage": "bf16 gradients and parameters, fp32 partitions",
        "data": "synthetic (seeded counter-hash generator; Box-Muller normals, uniform parameters)",
        "config": common_config(1),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "oracle": "C ring simulation (oracle/ring_sim.c, -O2, one thread "
                                   "per process)",
                         "sample": f"K=8, the same five steps per step; {cores} processes, each "
                                   f"running the oracle (C simulation, one thread) on its own "
                                   f"slab of {n} elements per rank (32 fragments of {n // 32})"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "bucket_pipeline":
        return run_pipeline_bench(args)
    if args.workload == "sweep":
        return run_sweep_bench(args)
    if args.workload == "configs":
        return run_configs_bench(args)
    if args.workload == "point":
        return run_point_bench(args)
    if args.workload == "fragments":
        return run_fragments_bench(args)
    if args.workload == "sequence":
        return run_sequence_bench(args)
    import torch
    rank, world, local_rank = dist_env()
    if world > 1:
        init_dist("nccl", torch.device("cuda", local_rank), args.pg_timeout)
    res = run_device(args, rank, world, local_rank)
    peak, peak_kind = load_peaks()
    kern = res["kernels"]
    dom = max(kern, key=lambda k: kern[k]["avg_ms"] * kern[k]["launches"])
    d = kern[dom]
    sha = kernel_src_sha()
    tr = NCU_TRAFFIC.get(dom)
    traffic = tr["bytes"] if tr and tr.get("src_sha") == kernel_src_sha(dom) \
        and not args.n_per_rank and not args.z3_layers else None
    value = job_value(res["step_bytes"], args.steps, world, res["max_elapsed"])
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(res["max_elapsed"] / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "storage": "bf16 gradients and parameters, fp32 partitions", "data": "synthetic (seeded counter-hash generator; Box-Muller normals, uniform parameters)",
        "config": common_config(world),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "pct_of_peak_is": f"of the {peak_kind} HBM copy peak ({peak} GB/s); the step's "
                          f"kernels read more than they write, so a read-dominated stream "
                          f"can exceed a copy",
        "pct_of_nominal_peak": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(d["gbs"], 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(d["gbs"] / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": d["bytes_per_launch"]},
        "kernels": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv)
                        for kk, vv in v.items()} for k, v in kern.items()},
        "headline_ops": res.get("headline"),
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "e2e": res["e2e"],
        "kernel_src_sha": sha,
    }
    if args.only:
        line["only"] = args.only
    if args.graph:
        line["graph"] = "one step captured in a CUDA graph and replayed; per-kernel figures from eager launches"
    if args.n_per_rank:
        line["config"]["elements_per_rank"] = wl_n = res["wl"].N
        line["config"]["bytes_per_rank"] = 2 * wl_n
        line["config"]["workload"] += f"_profile_case_{wl_n}"
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.only \
            and args.workload == "zero_bucket":
        line["cpu_baseline"] = cpu_baseline(args)
    if args.workload == "zero3_per_param":
        layers = args.z3_layers or 7
        line["config"] = {"workload": f"zero3_per_param_k8_h4096_{layers}layer", "K": 8,
                          "tensors_per_rank": 8 * layers, "elements_per_rank": res["wl"].N,
                          "step": "RS coalesced (ring_fp32, per-parameter shards) + AG coalesced",
                          "parallelism": "single GPU, 8 simulated ranks",
                          "l2": "inputs (42 GB resident) far larger than L2; no flush needed"}
        line["e2e"] = None
    if args.workload == "bf16_partition":
        line["config"] = {"workload": "zero3_bf16_partition_k8_1GiB" if not args.n_per_rank
                          else f"zero3_bf16_partition_k8_profile_case_{res['wl'].N}", "K": 8,
                          "elements_per_rank": res["wl"].N,
                          "step": "RS into bf16 partitions (copy_) + RS with bf16 add_ + "
                                  "step-time cast to fp32",
                          "parallelism": "single GPU, 8 simulated ranks",
                          "l2": "inputs (16 GiB resident) far larger than L2; no flush needed"}
        line["e2e"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if args.workload in ("zero3_per_param", "bf16_partition"):
        res["wl"].close()
    else:
        res["wl"].plan.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
