"""Benchmark of the fused chunked KL loss, forward + backward, on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one forward + backward of the loss (every kernel of the path) over one batch of
the named synthetic workload (default: the gpt-oss-20b-like student at 32K tokens, T=32768,
d=2880, V=201088, K=100).  Prints one JSON line.

* value: tokens/s over all ranks, inputs resident in HBM, timed with CUDA events on the
  launching stream over exactly K steps after W warm-up steps, barrier + synchronize on both
  sides, max over ranks.  Every input is larger than L2 (W alone is 1.16 GB), so no L2 flush
  is needed between steps.
* e2e: the same metric with the step's inputs (H, teacher cache, mask) copied host->device
  from pinned memory and the loss copied back inside the timed region; W stays resident as
  the model's LM-head weight.
* roofline: the tensor-core GEMM kind with the largest share of the step (forward
  projection, dS recompute, dW or dH); each of its launches is timed with a CUDA event pair
  that the library records on the launching stream during the timed steps (fkl_trace_*),
  and its algorithmic FLOPs (2*M*N*K) per launch are divided by the mean launch time, against
  the measured dense-bf16 tensor peak.  `tflops` / `tensor_frac_step` give the whole step's
  8*T*V*d against the same peak.
* cpu_baseline: the float64 oracle, timed as it stands on the host cores, on a bounded
  sample of the same workload (the first rows of the batch, full vocabulary).
* --impl reference: the oracle alone, on the host cores, as the comparison arm.

Under torchrun (N > 1) each rank holds one token shard of a global batch on its own GPU
(weak scaling: T tokens per rank), as a data-parallel trainer does: every step sums the
ranks' valid-token counts with an NCCL all-reduce before the loss (each rank divides by the
batch's count) and sums dW and the loss over the ranks after the backward
(lm_head_top_tcgen05_gb300.data_parallel.ShardedStep).  With one GPU the step is the plain
single-batch forward + backward.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd tokens/s & TFLOP/s (8TVd) at T=32K,V=201088,d=2880; peak GiB"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, busy_mhz_floor: float = 0.0):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


class EnergyMeter:
    """The GPU's total energy counter (NVML, millijoules) around the timed region, read through
    ctypes; None when NVML or the counter is not available."""

    def __init__(self, index: int):
        self.fn = None
        try:
            import ctypes

            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(handle)) != 0:
                return
            value = ctypes.c_ulonglong()

            def read():
                ok = nv.nvmlDeviceGetTotalEnergyConsumption(handle, ctypes.byref(value)) == 0
                return value.value if ok else None

            if read() is not None:
                self.fn = read
        except OSError:
            self.fn = None

    def read(self):
        return self.fn() if self.fn is not None else None


def cpu_oracle_rate(x, rows: int, divergence: str = "kl", div_param=None):
    """Tokens/s of the float64 oracle (forward + backward) on the first `rows` tokens."""
    import numpy as np

    import oracle

    W64 = oracle.to_f64(x.W)
    H64 = oracle.to_f64(x.H[:rows])
    idx, z, m = x.topk_idx[:rows], x.topk_logits[:rows], x.mask[:rows]
    t0 = time.perf_counter()
    if divergence == "kl":
        oracle.forward(H64, W64, idx, z, m, x.tau)
        oracle.backward(H64, W64, idx, z, m, x.tau)
    else:
        prm = {"jsd": 0.5, "skew_kl": 0.1, "skew_rkl": 0.1}.get(divergence, 0.0) if div_param is None else div_param
        oracle.divergences.forward(H64, W64, idx, z, m, x.tau, divergence, prm)
        oracle.divergences.backward(H64, W64, idx, z, m, x.tau, divergence, prm)
    dt = time.perf_counter() - t0
    del W64, H64
    cores = len(os.sched_getaffinity(0))
    return rows / dt, dt, cores, np.__version__


def loss_config(w, T, d, V, K, args, sharded: bool = False) -> dict:
    """The `config` of the loss's JSON line, the same for both arms."""
    world = args.gpus
    return {"workload": w.name, "T": T, "d": d, "V": V, "K": K, "tau": w.tau, "chunk": w.chunk,
            "divergence": args.divergence, "grad_dtype": args.grad_dtype,
            "l2": "inputs larger than L2 (W is 1.16 GB); no flush",
            "parallelism": "single GPU" if not sharded else
            f"token-sharded dp{world}: NCCL all-reduce of the valid-token count before the loss, of dW and "
            f"the loss after it; T={T} tokens per rank"}


def run_reference(args, rank):
    """The comparison arm: the float64 oracle on the host cores, bounded samples of the batch."""
    import workloads

    if rank != 0:
        return
    w = workloads.WORKLOADS[args.workload]
    x = workloads.make_inputs(w, rows=args.cpu_rows)
    cpu_oracle_rate(x, min(8, args.cpu_rows))  # warm-up: BLAS threads, page-in
    rates, secs = [], []
    for _ in range(args.steps):
        r, dt, cores, _ = cpu_oracle_rate(x, args.cpu_rows)
        rates.append(r)
        secs.append(dt)
    value = statistics.median(rates)
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * w.T / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": loss_config(w, w.T, w.d, w.V, w.K, args, sharded=args.gpus > 1 or args.sharded),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "blas_threads": blas_threads(),
                         "kind": "oracle",
                         "sample": f"first {args.cpu_rows} tokens of the batch per step, full "
                                   f"vocabulary, float64 forward+backward; ms_per_step extrapolates "
                                   f"to T={w.T}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over the ranks of the default process group (the value itself alone)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


KIND_NAMES = {0: "forward projection + logsumexp/top-K", 1: "dS recompute", 2: "dW", 3: "dH"}
FIXUP_KIND = 4
KERNEL_NAMES = {0: "gemm2_kernel<256,0,0,EpiFwd> (two-SM)", 1: "gemm2_kernel<256,0,0,EpiDs> (two-SM)",
                2: "gemm2_kernel<256,1,1,EpiF32> (two-SM, dW)", 3: "gemm2_kernel<256,0,1,EpiF32> (two-SM, dH)"}
# Launches per step outside the GEMM trace: forward prep, 3 token-weight kernels, 2 combine;
# backward prep, 3 token-weight kernels, gradient scale, poison check.  A divergence other
# than KL adds one per-row kernel to each pass.
UNTRACED_LAUNCHES_PER_STEP = 12
# Token-sharded data parallelism (N > 1) adds the local count's two kernels per step.
LOCAL_COUNT_LAUNCHES = 2

# Dense bf16 tensor-core rate of one Blackwell SM: 4096 FMA = 8192 FLOP per clock (NVIDIA's
# nominal 2.25 PFLOP/s for GB300 is 152 SMs x 8192 x 1.807 GHz).  The nominal roofline of a
# run is this rate x the device's SM count x the SM clock sampled during the timed region.
BF16_FLOP_PER_CLK_PER_SM = 8192


def blas_threads():
    """Threads of the BLAS that NumPy uses (the oracle's matrix products), or None."""
    try:
        from threadpoolctl import threadpool_info

        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    import ctypes
    import glob

    import numpy as np

    libs = glob.glob(os.path.join(os.path.dirname(np.__file__), os.pardir, "numpy.libs", "*openblas*"))
    for path in libs:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for name in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_", "openblas_get_num_threads"):
            fn = getattr(lib, name, None)
            if fn is not None:
                return int(fn())
    return None

# DRAM bytes (read + write) per launch of each GEMM kind on the 32K workload (T=32768,
# d=2880, V=201088), valid only for the CUDA sources they were taken on: one ncu capture of
# every launch of five full-size steps (dram__bytes_read.sum + dram__bytes_write.sum, one
# pass), averaged over the launches of each kind; TRAFFIC_FLOPS is that kind's mean work per
# launch, so the bench's own launches take the figures as they are.
TRAFFIC_SOURCES_SHA = "d536741306180354"
TRAFFIC_BYTES = {0: 9.214e9, 1: 1.610e9, 2: 2.439e9, 3: 3.129e9}
TRAFFIC_FLOPS = {0: 2.0 * 32768 * 201088 * 2880, 1: 2.0 * 32768 * 201088 * 2880 / 18,
                 2: 2.0 * 32768 * 201088 * 2880 / 18, 3: 2.0 * 32768 * 201088 * 2880 / 18}


# The sources that define the loss's tensor-core GEMMs and how they are launched (tiles,
# ring, epilogues, unit order, block planning): the measured traffic above is valid while
# their code (comments aside) is unchanged.  The light kernels (prep, combine, weights), the teacher cache and the
# trace do not enter.
GEMM_SOURCES = ("fkl_api.cu", "fkl_gemm.cuh", "fkl_gemm2.cu", "fkl_gemm2.cuh", "fkl_internal.h", "fkl_ptx.cuh")


def csrc_sha() -> str:
    """Hash of the GEMM sources' code: comments and whitespace do not enter."""
    import hashlib
    import re

    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "lm_head_top_tcgen05_gb300", "csrc", name), encoding="utf-8") as fh:
            code = fh.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        h.update(name.encode())
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


def traffic_per_launch(kind, flops_per_launch, d):
    """Measured bytes per launch, scaled to the mean launch by the work it does (traffic of
    these products grows in proportion to the slab width), or None when no capture applies."""
    if kind not in TRAFFIC_BYTES or d != 2880 or csrc_sha() != TRAFFIC_SOURCES_SHA:
        return None
    return TRAFFIC_BYTES[kind] * flops_per_launch / TRAFFIC_FLOPS[kind]


def trace_summary(L, cap):
    import ctypes

    ms = (ctypes.c_float * cap)()
    kind = (ctypes.c_int32 * cap)()
    flops = (ctypes.c_double * cap)()
    n = L.fkl_trace_read(ms, kind, flops, cap)
    if n < 0:
        raise RuntimeError("fkl_trace_read failed")
    if n >= cap:
        raise RuntimeError(f"the trace filled its {cap} entries: launches of the timed steps were not recorded")
    # kind 4 is the fixup of the K-split units of the dW or dH launch just before it: its time
    # belongs to that product and its launch is counted as the product's fixup launch
    per = {}
    prev = None
    for i in range(n):
        k = kind[i]
        if k == FIXUP_KIND and prev is not None:
            a = per[prev]
            a[1] += ms[i]
            a[3] += 1
            continue
        a = per.setdefault(k, [0, 0.0, 0.0, 0])
        a[0] += 1
        a[1] += ms[i]
        a[2] += flops[i]
        prev = k
    return {k: {"launches": c, "fixup_launches": fx, "ms_total": t, "ms_per_launch": t / c,
                "flops_per_launch": f / c, "tflops": f / (t / 1e3) / 1e12}
            for k, (c, t, f, fx) in sorted(per.items())}


def run_teacher_topk(args, world, rank, local_rank):
    """Times the offline teacher cache producer: the workload's H and W stand in for the
    teacher's final hidden states and LM head; K as in the workload."""
    import torch

    import lm_head_top_tcgen05_gb300 as fkl
    import workloads

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workloads.WORKLOADS[args.workload]
    if args.vocab is not None or args.tokens is not None:
        w = dataclasses.replace(w, name=f"{w.name}_V{args.vocab or w.V}_T{args.tokens or w.T}",
                                V=args.vocab or w.V, T=args.tokens or w.T)
    x = workloads.make_inputs(w)
    T, d, V, K = w.T, w.d, w.V, w.K
    Ht, Wt = x.H.to(dev), x.W.to(dev)
    ws = fkl.Workspace(dev)
    for _ in range(args.warmup):
        fkl.teacher_topk(Ht, Wt, K, workspace=ws, max_bound_stride=args.bound_stride)
    torch.cuda.synchronize()
    assert fkl.read_status(ws) == 0
    L = fkl.lib()
    cap = 2 * args.steps + 1
    fkl.check(L.fkl_trace_start(cap), "fkl_trace_start")
    stream = torch.cuda.current_stream(dev)
    with ClockSampler(local_rank) as clocks:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fkl.teacher_topk(Ht, Wt, K, workspace=ws, max_bound_stride=args.bound_stride)
        e1.record(stream)
        torch.cuda.synchronize()
    L.fkl_trace_stop()
    elapsed = e0.elapsed_time(e1) / 1e3
    kernels = trace_summary(L, cap)
    status = fkl.read_status(ws)
    peaks, peak_kind = load_peaks()
    sustained = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    dom = max(kernels, key=lambda k: kernels[k]["ms_total"])
    names = {5: "gemm2_kernel<256,0,0,EpiTopR> (bound pass)", 6: "gemm2_kernel<256,0,0,EpiCand> (candidate pass)"}
    out = {
        "metric": "teacher top-K cache tokens/s", "value": T * args.steps / elapsed,
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "T": T, "d": d, "V": V, "K": K, "max_bound_stride": args.bound_stride},
        # executed work: the bound pass over the sampled vocabulary rows + the full candidate pass
        "tflops": sum(v["flops_per_launch"] * v["launches"] for v in kernels.values()) / elapsed / 1e12,
        "projection_tflops": 2.0 * T * V * d * args.steps / elapsed / 1e12, "status": status,
        "roofline": {"bound": "tensor", "kernel": names.get(dom, str(dom)), "achieved": kernels[dom]["tflops"],
                     "peak": sustained, "unit": "TFLOP/s", "frac": kernels[dom]["tflops"] / sustained,
                     "peak_source": f"{peak_kind} bf16_tflops_sustained", "traffic": None},
        "kernels": {names.get(k, str(k)): v for k, v in kernels.items()},
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle

        rows = min(args.cpu_rows, T)
        W64, H64 = oracle.to_f64(x.W), oracle.to_f64(x.H[:rows])
        t0 = time.perf_counter()
        oracle.teacher_topk(H64, W64, K)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": rows / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                               "blas_threads": blas_threads(), "kind": "oracle",
                               "sample": f"first {rows} tokens, full vocabulary, float64, {dt:.1f} s"}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="gptoss20b_32k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=128, help="tokens in the CPU oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--vocab", type=int, default=None,
                    help="override V (profiling case with the full workload's per-launch GEMM shapes)")
    ap.add_argument("--chunk", type=int, default=None, help="override chunk")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (the memory / time sweep over sequence length)")
    ap.add_argument("--divergence", default="kl", choices=["kl", "jsd", "skew_kl", "skew_rkl", "tv"],
                    help="the loss's divergence (default: KL, the headline)")
    ap.add_argument("--div-param", type=float, default=None, help="b for jsd, a for the skew forms")
    ap.add_argument("--grad-dtype", default="fp32", choices=["fp32", "bf16"],
                    help="dtype of the dH / dW outputs (default fp32; bf16: fp32 sums rounded once)")
    ap.add_argument("--bound-stride", type=int, default=0,
                    help="teacher_topk: largest vocabulary sampling stride of the bound pass (0: default)")
    ap.add_argument("--sharded", action="store_true",
                    help="run the token-sharded data-parallel step (ShardedStep) even on one GPU, where "
                         "its all-reduces are no-ops (under torchrun with N > 1 it always runs)")
    ap.add_argument("--mode", default="loss", choices=["loss", "teacher_topk"],
                    help="loss: the fused KL fwd+bwd step (the headline); teacher_topk: the offline "
                         "teacher cache producer on the same shapes")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import torch.distributed as dist

    import lm_head_top_tcgen05_gb300 as fkl
    import workloads

    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if args.mode == "teacher_topk":
        run_teacher_topk(args, world, rank, local_rank)
        return
    w = workloads.WORKLOADS[args.workload]
    if args.vocab is not None or args.chunk is not None:
        w = dataclasses.replace(w, name=f"{w.name}_V{args.vocab or w.V}_chunk{args.chunk or w.chunk}",
                                V=args.vocab or w.V, chunk=args.chunk or w.chunk)
    if args.tokens is not None:
        w = dataclasses.replace(w, name=f"{w.name}_T{args.tokens}", T=args.tokens)
    x = workloads.make_inputs(w)
    T, d, V, K = w.T, w.d, w.V, w.K

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---------------------------------------------------------------- device-resident run
    H, Wt = x.H.to(dev), x.W.to(dev)
    idx, z, m = x.topk_idx.to(dev), x.topk_logits.to(dev), x.mask.to(dev)
    ws = fkl.Workspace(dev)
    gdt = torch.bfloat16 if args.grad_dtype == "bf16" else torch.float32
    dH = torch.empty((T, d), dtype=gdt, device=dev)
    dW = torch.empty((V, d), dtype=gdt, device=dev)
    torch.cuda.synchronize()
    inputs_bytes = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)

    # divergences other than KL hand the student logits at the cached ids to the backward
    div = dict(divergence=args.divergence, div_param=args.div_param)
    s_ids = torch.empty((T, K), dtype=torch.float32, device=dev) if args.divergence != "kl" else None

    # N > 1: token-sharded data parallelism (count all-reduce before the loss, dW and loss
    # all-reduce after it); one GPU: the plain step
    dp = None
    if world > 1 or args.sharded:
        from lm_head_top_tcgen05_gb300.data_parallel import ShardedStep

        dp = ShardedStep()

    def run_step(Hd, idd, zd, md, ev=None):
        """One step over the given device inputs; returns the loss (a device scalar)."""
        if dp is not None:
            loss, _, _ = dp(Hd, Wt, idd, zd, md, w.tau, w.chunk, workspace=ws, out=(dH, dW), grad_dtype=gdt,
                            student_topk_logits=s_ids, **div)
            return loss
        loss, lse = fkl.forward(Hd, Wt, idd, zd, md, w.tau, w.chunk, workspace=ws, student_topk_logits=s_ids, **div)
        if ev is not None:
            ev.record(stream)
        fkl.backward(Hd, Wt, idd, zd, md, lse, None, w.tau, w.chunk, workspace=ws, out=(dH, dW),
                     student_topk_logits=s_ids, grad_dtype=gdt, **div)
        return loss

    stream = torch.cuda.current_stream(dev)

    def step():
        return run_step(H, idx, z, m)

    for _ in range(args.warmup):
        step()
    barrier()
    assert fkl.read_status(ws) == 0, "device status not ok after warm-up"
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    nslabs = int(fkl.lib().fkl_backward_slabs(T, d, V, K, w.chunk))
    # per step: the forward, three products per backward block and at most one K-split
    # fixup each for dW and dH; one more entry so that a full trace is detected
    trace_cap = args.steps * (1 + 5 * nslabs) + 1
    fkl.check(fkl.lib().fkl_trace_start(trace_cap), "fkl_trace_start")
    energy = EnergyMeter(local_rank)
    with ClockSampler(local_rank) as clocks:
        barrier()
        mj0 = energy.read()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            loss = run_step(H, idx, z, m, ev=ev[i][1])
            ev[i][2].record(stream)
        end.record(stream)
        barrier()
        mj1 = energy.read()
    fkl.lib().fkl_trace_stop()
    elapsed = max_over_ranks(start.elapsed_time(end) / 1e3, dev)
    kernels = trace_summary(fkl.lib(), trace_cap)
    status = fkl.read_status(ws)
    peak_bytes = torch.cuda.max_memory_allocated(dev)
    fwd_ms = bwd_ms = None
    if dp is None:
        fwd_ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps))
        bwd_ms = statistics.mean(ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps))
    step_ms_median = statistics.median(ev[i][0].elapsed_time(ev[i][2]) for i in range(args.steps))
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    loss_val = loss.item()

    # ---------------------------------------------------------------- end to end (host buffers)
    e2e = None
    if not args.no_e2e:
        hH = x.H.pin_memory()
        hidx, hz, hm = x.topk_idx.pin_memory(), x.topk_logits.pin_memory(), x.mask.pin_memory()
        hloss = torch.empty((), dtype=torch.float32).pin_memory()
        h2d = hH.numel() * 2 + hidx.numel() * 4 + hz.numel() * 4 + hm.numel()

        # Inputs are double-buffered on the device: step i+1's host-to-device copies run on a
        # copy stream while step i computes, as a training loop that prefetches its next batch
        # does.  Every step's copies are inside the timed region (the first copy starts after
        # the start event), and each step's loss is read back to pinned host memory.
        hosts = (hH, hidx, hz, hm)
        bufs = [[torch.empty_like(t, device=dev) for t in hosts] for _ in range(2)]
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        free = [torch.cuda.Event() for _ in range(2)]
        for e in free:
            e.record(stream)

        def e2e_copy(b, after=None):
            with torch.cuda.stream(copy_stream):
                if after is not None:
                    copy_stream.wait_event(after)
                copy_stream.wait_event(free[b])
                for dst, src in zip(bufs[b], hosts):
                    dst.copy_(src, non_blocking=True)
                copied[b].record(copy_stream)

        def e2e_compute(b):
            stream.wait_event(copied[b])
            Hd, idd, zd, md = bufs[b]
            l = run_step(Hd, idd, zd, md)
            free[b].record(stream)
            hloss.copy_(l, non_blocking=True)

        def e2e_run(n, start=None):
            e2e_copy(0, after=start)
            for k in range(n):
                if k + 1 < n:
                    e2e_copy((k + 1) % 2)
                e2e_compute(k % 2)

        e2e_run(args.warmup)
        torch.cuda.synchronize(dev)
        barrier()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        e2e_run(args.steps, start=s0)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_t = max_over_ranks(s0.elapsed_time(s1) / 1e3, dev)
        e2e = {"value": world * T * args.steps / e2e_t, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": 4,
               "d2h": "loss read back each step; dH and dW stay resident on the device, as in a training loop"}

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return

    peaks, peak_kind = load_peaks()
    ms_per_step = 1e3 * elapsed / args.steps
    tokens_s = world * T * args.steps / elapsed
    tflops = world * w.flops_fwd_bwd * args.steps / elapsed / 1e12
    sustained = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    burst = float(peaks["bf16_tflops"])
    traced = sum(v["launches"] + v["fixup_launches"] for v in kernels.values())
    launches_per_step = (UNTRACED_LAUNCHES_PER_STEP + (2 if args.divergence != "kl" else 0)
                         + (LOCAL_COUNT_LAUNCHES if dp is not None else 0) + traced / args.steps)
    clk = clocks.summary()
    dom = max(kernels, key=lambda k: kernels[k]["ms_total"])  # largest share of the step
    nominal = None
    if clk and clk.get("sm_mhz"):
        at_clk = sms * BF16_FLOP_PER_CLK_PER_SM * clk["sm_mhz"] * 1e6 / 1e12
        at_max = sms * BF16_FLOP_PER_CLK_PER_SM * clk["sm_max_mhz"] * 1e6 / 1e12
        nominal = {"sms": sms, "flop_per_clk_per_sm": BF16_FLOP_PER_CLK_PER_SM,
                   "tflops_at_median_clock": at_clk, "frac": kernels[dom]["tflops"] / at_clk,
                   "step_frac": tflops / world / at_clk,
                   "tflops_at_max_clock": at_max, "frac_of_max_clock": kernels[dom]["tflops"] / at_max}
    out = {
        "metric": METRIC, "value": tokens_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": loss_config(w, T, d, V, K, args, sharded=dp is not None),
        "ms_per_step_median": step_ms_median,
        "tflops": tflops,
        "tensor_frac_step": tflops / sustained,
        "peak_gib": peak_bytes / 2**30,
        "peak_gib_above_inputs": (peak_bytes - inputs_bytes) / 2**30,
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "loss": loss_val, "status": status,
        "roofline": {"bound": "tensor", "kernel": KERNEL_NAMES[dom],
                     "achieved": kernels[dom]["tflops"], "peak": sustained, "unit": "TFLOP/s",
                     "frac": kernels[dom]["tflops"] / sustained,
                     "frac_of_burst": kernels[dom]["tflops"] / burst,
                     "peak_source": f"{peak_kind} bf16_tflops_sustained (timed inside a seconds-long loop)",
                     "flops_per_launch": kernels[dom]["flops_per_launch"],
                     "ms_per_launch": kernels[dom]["ms_per_launch"],
                     "traffic": traffic_per_launch(dom, kernels[dom]["flops_per_launch"], d)
                     if (T, V) == (32768, 201088) and args.grad_dtype == "fp32" else None,
                     "nominal": nominal},
        "kernels": {KIND_NAMES[k]: {kk: round(vv, 4) if isinstance(vv, float) else vv for kk, vv in v.items()}
                    for k, v in kernels.items()},
        "clocks": clk,
        # this GPU's energy over the timed steps (NVML counter; rank 0's GPU under torchrun)
        "energy_j_per_step": (mj1 - mj0) / 1e3 / args.steps if mj0 is not None and mj1 is not None else None,
        "gpu_launches": int(round(launches_per_step * args.steps)),
    }
    if e2e is not None:
        out["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        rate, dt, cores, _ = cpu_oracle_rate(x, args.cpu_rows, args.divergence, args.div_param)
        out["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores, "blas_threads": blas_threads(),
                               "kind": "oracle",
                               "sample": f"first {args.cpu_rows} tokens, full vocabulary, float64 "
                                         f"forward+backward, {dt:.1f} s"}
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
