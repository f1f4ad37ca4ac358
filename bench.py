#!/usr/bin/env python
"""Benchmark of the fused top-K KL distillation loss, forward + backward.

One step = one kd_topk_kl_forward_backward call over one synthetic batch (the
single-sweep training step: teacher prep, then per row chunk the row offsets, the
logit GEMM with online lse + gather that also stores the valid rows' logits as
bf16 values relative to their offsets, the combine, the cached-column pass, the
dh and dW contractions); `--api split` times
kd_topk_kl_forward + kd_topk_kl_backward instead (the backward recomputes the
logits).  Default workload: ctx_32k (T=32768, V=201088, d=2880,
K=100, tau=1, 10% rows masked), inputs resident in HBM and larger than L2.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line (rank 0).  With N > 1 (torchrun), every rank runs its own
batch (replicas, weak scaling, no collective on the data path); the timed
region is bracketed by barriers and the max over ranks is reported.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload instead.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused top-K KL fwd+bwd tokens/s (T=32k,V=201k,d=2880); % bf16 TC peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ---------------------------------------------------------------- ranks

def rank_info():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def dist_setup(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device="cpu") -> float:
    """Max of a per-rank scalar (the slowest rank sets the job time)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job units/s: all ranks' units over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ---------------------------------------------------------------- clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling (200 ms) while the timed region runs."""

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="kd_clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return parse_clock_csv(open(self.path).read())


def parse_clock_csv(text: str) -> dict:
    sm, smax, power, reasons = [], [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.strip().splitlines():
        f = [c.strip() for c in line.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            smax.append(float(f[2]))
            power.append(float(f[3]))
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    return {"sm_mhz": float(statistics.median(sm)), "sm_max_mhz": float(max(smax)),
            "power_w_max": float(max(power)), "reasons": sorted(reasons), "samples": len(sm)}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


DEVICE_SOURCES = ("kd_kernels.cuh", "kd_ptx.cuh", "kd_topk_producer.cuh")


def device_source_sha256() -> str:
    """Hash of the device-code files the profiled kernels are compiled from."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunked_top_kl_logit_b300", "csrc")
    for name in DEVICE_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def load_traffic(kernel: str, workload: str, chunk: int):
    """DRAM bytes per launch of `kernel` from a committed ncu summary, only if
    it was captured on this workload and chunk size and the device code still
    hashes to what was profiled (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("device_sha256") != device_source_sha256():
        return None
    if d.get("workload") != workload or d.get("chunk") not in (None, chunk):
        return None
    return d.get("bytes_per_launch")


# ---------------------------------------------------------------- CPU oracle

def blas_threads() -> int:
    try:
        import threadpoolctl
        n = [i.get("num_threads", 0) for i in threadpoolctl.threadpool_info()
             if i.get("internal_api") in ("openblas", "mkl", "blis")]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample(w, rows: int, seed: int = 0):
    """A `rows`-row sample of workload `w` (full V, d), as the oracle sees it."""
    from synth import make_inputs
    x = make_inputs(w.replace(T=rows), seed=seed)
    return dict(h=x["h"].to(torch.bfloat16).double().numpy(),
                W=x["W"].to(torch.bfloat16).double().numpy(),
                idx=x["teacher_idx"].numpy(), tl=x["teacher_logits"].double().numpy(),
                valid=x["valid"].numpy(), tau=w.tau)


def oracle_step_seconds(s) -> float:
    """Wall time of the fp64 oracle's forward + backward on sample `s`."""
    from oracle import kd_oracle as O
    t0 = time.perf_counter()
    f = O.forward(s["h"], s["W"], s["idx"], s["tl"], s["valid"], s["tau"])
    O.backward(s["h"], s["W"], s["idx"], s["tl"], s["valid"], s["tau"], 1.0, lse=f["lse"])
    return time.perf_counter() - t0


def run_reference(args, w, world, rank):
    if rank != 0:
        return None
    rows = args.ref_rows
    s = oracle_sample(w, rows)
    times = []
    for i in range(args.warmup + args.steps):
        dt = oracle_step_seconds(s)
        if i >= args.warmup:
            times.append(dt)
    sec = statistics.mean(times)
    value = rows / sec
    sample = (f"fp64 oracle fwd+bwd on a {rows}-row sample of {w.name} "
              f"(full V={w.V}, d={w.d}) per step")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, args.chunk or w.chunk),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def workload_config(w, chunk):
    return {"workload": w.name, "T": w.T, "V": w.V, "d": w.d, "K": w.K, "tau": w.tau,
            "chunk": chunk, "mask": w.mask_kind, "teacher_idx": w.idx_kind,
            "l2": "inputs larger than L2 (W alone is V*d*2 B)"}


# ---------------------------------------------------------------- GPU run
KERNEL_DESC = {
    "logits_fwd": "forward logit GEMM + online lse + gather",
    "logits_fwd_sweep": "forward logit GEMM + online lse + gather + bf16 logits relative "
                        "to the row offsets stored into the chunk's G buffer",
    "logits_bwd": "backward logit recompute + bf16 gradient tile",
    "dh": "dh^T = W^T G^T over the chunk's valid rows",
    "dW": "dW = G^T h_c, accumulated over chunks",
}


def kernel_table(kstats: dict, steps: int, T: int, n_valid: int, d: int, V: int,
                 K: int, sweep: bool = False) -> dict:
    """Per timed kernel: launches, time and achieved rate over the timed steps.
    Contractions (TFLOP/s), algorithmic FLOPs: 2 T d V for the forward logits,
    2 Nv d V for each backward contraction (masked rows are skipped).  The
    single sweep's cached-column pass (GB/s): 14 K bytes per valid row (the
    sorted index, the teacher probability and the gathered logit read, one
    bf16 value written per slot); the zero rows it writes after a chunk's
    valid rows are not counted.  In the single sweep the backward recompute
    launch runs only for a chunk whose stored values would leave their range
    (it returns at once otherwise), so it gets a time but no rate."""
    out = {}
    for name, (cnt, ms) in kstats.items():
        if cnt == 0:
            continue
        row = {"launches": cnt, "ms_total": ms, "ms_per_step": ms / steps,
               "ms_per_launch": ms / cnt}
        if sweep and name == "logits_bwd":
            row["note"] = "recompute of a flagged chunk's G (returns at once otherwise)"
        elif name == "sweep_fix":
            nbytes = 14.0 * K * n_valid * steps
            row.update(bytes_per_launch=nbytes / cnt,
                       gbs=nbytes / (ms / 1e3) / 1e9 if ms > 0 else None)
        else:
            rows = T if name == "logits_fwd" else n_valid
            flops = 2.0 * rows * d * V * steps
            row.update(flops_per_launch=flops / cnt,
                       tflops=flops / (ms / 1e3) / 1e12 if ms > 0 else None)
        out[name] = row
    return out



def run_e2e_pipelined(kd, args, m0, x, dev_inputs, T, V, d, K, chunk, tau, n, world, dev,
                      fused):
    """End-to-end throughput through the public API with host transfers inside
    the timed region, pipelined over two buffer sets (see run_ours)."""
    names = ("h", "W", "idx", "tl", "valid")
    host_src = (x["h"], x["W"], x["teacher_idx"], x["teacher_logits"], x["valid"])
    hin = {k: v.pin_memory() for k, v in zip(names, host_src)}
    sets = [dict(zip(names, dev_inputs), m=m0),
            dict({k: torch.empty_like(v) for k, v in zip(names, dev_inputs)},
                 m=kd.TopKKL(T, V, d, K, chunk, device=dev, fused=fused))]
    hout = {"loss": torch.empty(1, pin_memory=True), "lse": torch.empty(T, pin_memory=True),
            "dh": torch.empty(T, d, pin_memory=True), "dW": torch.empty(V, d, pin_memory=True)}
    s_comp = torch.cuda.current_stream(dev)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def launch(i):
        j = i % 2
        b = sets[j]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_done[j])      # step i-2 has finished with these inputs
            for k in names:
                b[k].copy_(hin[k], non_blocking=True)
            ev_in[j].record(s_in)
        s_comp.wait_event(ev_in[j])
        if i >= 2:
            s_comp.wait_event(ev_out[j])         # step i-2's outputs have been copied out
        mm = b["m"]
        if fused:
            mm.forward_backward(b["h"], b["W"], b["idx"], b["tl"], b["valid"], tau, 1.0,
                                valid_rows_only=args.valid_rows_only,
                                stream=s_comp)
        else:
            mm.forward(b["h"], b["W"], b["idx"], b["tl"], b["valid"], tau, stream=s_comp)
            mm.backward(b["h"], b["W"], b["idx"], b["tl"], b["valid"], tau, 1.0, stream=s_comp)
        ev_done[j].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[j])
            for k, t in (("loss", mm.loss), ("lse", mm.lse), ("dh", mm.dh), ("dW", mm.dW)):
                hout[k].copy_(t, non_blocking=True)
            ev_out[j].record(s_out)

    for i in range(2):                             # warm the second buffer set
        launch(i)
    torch.cuda.synchronize()
    ne = max(2, n)  # as many steps as the device-timed region: the pipeline's fill (the
    # first step's inputs) and drain (the last step's outputs) are in the timed region
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(s_comp)
    s_in.wait_stream(s_comp)
    s_out.wait_stream(s_comp)
    for i in range(ne):
        launch(i)
    s_comp.wait_stream(s_out)
    s_comp.wait_stream(s_in)
    t1.record(s_comp)
    torch.cuda.synchronize()
    barrier(world)
    for b in sets:
        kd.check_device_status(b["m"].status, "e2e steps")
    sec = max_over_ranks(t0.elapsed_time(t1) / 1e3, world, device=dev)
    return {"value": job_throughput(T * ne, world, sec), "unit": "tokens/s",
            "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in hin.values())),
            "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in hout.values())),
            "ms_per_step": sec * 1e3 / ne, "steps": ne,
            "pipelined": "2 buffer sets, 3 streams: H2D / compute / D2H overlap across steps"}


def run_ours(args, w, world, rank, local_rank):
    import chunked_top_kl_logit_b300 as kd
    from synth import make_inputs
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    chunk = args.chunk or w.chunk
    x = make_inputs(w, seed=args.seed + rank, device=dev)
    T, V, d, K, tau = w.T, w.V, w.d, w.K, w.tau
    h = x["h"].to(dev)
    W = x["W"].to(dev)
    idx = x["teacher_idx"].to(dev)
    tl = x["teacher_logits"].to(dev)
    valid = x["valid"].to(dev)
    n_valid = int(x["valid"].sum())

    torch.cuda.synchronize()
    base_alloc = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    free_before = torch.cuda.mem_get_info(dev)[0]  # cross-check with the CUDA device's free-memory count
    residual = args.variant == "residual"
    fused = args.api == "fused"
    m = kd.TopKKL(T, V, d, K, chunk, device=dev, fused=fused)
    if residual:
        from synth import teacher_full_lse
        tlse = teacher_full_lse(x["teacher_logits"].cpu(), tau, seed=args.seed + rank).to(dev)
        outside_mass = torch.empty(T, dtype=torch.float32, device=dev)

    def fwd_part():
        if residual and fused:
            m.forward_backward_residual(h, W, idx, tl, tlse, valid, tau, 1.0,
                                        valid_rows_only=args.valid_rows_only)
        elif residual:
            kd.kd_topk_kl_forward_residual(h, W, idx, tl, tlse, valid, tau, chunk, m.loss, m.lse,
                                           m.row_kl, outside_mass, ws=m.ws, dev_status=m.status)
        elif fused:
            m.forward_backward(h, W, idx, tl, valid, tau, 1.0,
                               valid_rows_only=args.valid_rows_only)
        else:
            m.forward(h, W, idx, tl, valid, tau)

    def bwd_part():
        if residual and not fused:
            kd.kd_topk_kl_backward_residual(h, W, idx, tl, tlse, valid, tau, chunk, m.lse,
                                            outside_mass, 1.0, m.dh, m.dW, ws=m.ws,
                                            dev_status=m.status)
        elif not fused:
            m.backward(h, W, idx, tl, valid, tau, 1.0)

    def step():
        fwd_part()
        bwd_part()

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize()
    kd.check_device_status(m.status, "warm-up step")
    peak = torch.cuda.max_memory_allocated(dev)
    free_after = torch.cuda.mem_get_info(dev)[0]

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_id).start()
    time.sleep(0.3)
    n = args.steps
    fl, bl = kd.kd_topk_kl_launch_count(T, V, d, K, chunk)
    sweep_launches = kd.kd_topk_kl_forward_backward_workspace_size(T, V, d, K, chunk)[1]
    step_launches = sweep_launches if fused else fl + bl
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    barrier(world)
    torch.cuda.synchronize()
    # every contraction launch of the timed steps is bracketed by CUDA events
    # on its own stream (the library records them; diagnostic interface)
    kd.kd_timing_start(step_launches * n + 8)
    for i in range(n):
        ev[i][0].record()
        fwd_part()
        ev[i][1].record()
        bwd_part()
        ev[i][2].record()
    torch.cuda.synchronize()
    kd.kd_timing_stop()
    barrier(world)
    clocks = sampler.stop()
    kd.check_device_status(m.status, "timed steps")
    kstats = {name: kd.kd_timing_query(kid)
              for name, kid in {**kd.KERNELS, **kd.SWEEP_KERNELS}.items()}
    kd.kd_timing_release()
    total_ms = ev[0][0].elapsed_time(ev[n - 1][2])
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    max_sec = max_over_ranks(total_ms / 1e3, world, device=dev)
    ms_per_step = max_sec * 1e3 / n
    value = job_throughput(T * n, world, max_sec)

    # end to end through the public API: every step copies its inputs from
    # pinned host memory to the device, runs forward + backward and copies its
    # outputs (loss, lse, dh, dW) back to pinned host memory.  The steps are
    # pipelined over two device buffer sets on three streams: step i+1's inputs
    # go up and step i-1's outputs come down while step i computes.
    e2e = None
    if not args.no_e2e and not residual:
        e2e = run_e2e_pipelined(kd, args, m, x, (h, W, idx, tl, valid), T, V, d, K, chunk, tau,
                                n, world, dev, fused)


    peaks, peak_src = load_peaks()
    sweep = fused
    flops_nominal = 8.0 * T * d * V
    # the single sweep forms each row's logits once: no recompute GEMM
    fwd_rows = n_valid if (sweep and args.valid_rows_only) else T
    flops_alg = (2.0 * fwd_rows + (4.0 if sweep else 6.0) * n_valid) * d * V
    tf_nominal = flops_nominal / (ms_per_step / 1e3) / 1e12 * world
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    kernels = kernel_table(kstats, n, fwd_rows, n_valid, d, V, K, sweep)
    contractions = [k for k, v in kernels.items() if "tflops" in v]
    dom = max(contractions, key=lambda k: kernels[k]["ms_per_step"])
    kd_dom = kernels[dom]
    dom_desc = KERNEL_DESC["logits_fwd_sweep" if (sweep and dom == "logits_fwd") else dom]
    if dom == "logits_fwd":  # the forward's epilogue mode: single sweep / residual variant
        dom_id = (8 if residual else 7) if sweep else (6 if residual else 0)
    else:
        dom_id = kd.KERNELS[dom]
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": n,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(w, chunk), parallelism=f"replicas x{world}",
                       masked_rows=("logits not formed (KD_VALID_ROWS_ONLY), lse NaN"
                                    if (sweep and args.valid_rows_only)
                                    else "logits formed, lse of every row")),
        "tflops_nominal": tf_nominal / world,
        "tflops_algorithmic": flops_alg / (ms_per_step / 1e3) / 1e12,
        "flop_counts": ("nominal: the metric's 8 T d V (forward, recompute, dh, dW); "
                        "algorithmic: the FLOPs performed, (2 T + 4 Nv) d V for the single sweep "
                        "(no recompute) and (2 T + 6 Nv) d V for the split calls"),
        "frac_bf16_peak_burst": tf_nominal / world / burst,
        "frac_bf16_peak_sustained": tf_nominal / world / sustained,
        "api": "fused" if fused else "split", "variant": args.variant,
        "fwd_ms": None if fused else fwd_ms, "bwd_ms": None if fused else bwd_ms,
        "kernels": kernels,
        "roofline": {"kernel": f"kd_gemm_kernel<{dom_id}> ({dom_desc})",
                     "bound": "tensor", "achieved": kd_dom["tflops"],
                     "peak": sustained, "unit": "TFLOP/s", "frac": kd_dom["tflops"] / sustained,
                     "peak_kind": f"bf16 sustained (kernel timed inside the step), {peak_src}",
                     "frac_of_burst": kd_dom["tflops"] / burst,
                     "flops_per_launch": kd_dom["flops_per_launch"],
                     "traffic": load_traffic("logits_fwd_sweep"
                                             if (sweep and dom == "logits_fwd") else dom,
                                             w.name, chunk)},
        "memory": {"peak_allocated_bytes": int(peak),
                   "peak_minus_inputs_bytes": int(peak - base_alloc),
                   "device_free_drop_bytes": int(free_before - free_after),
                   "dense_TxV_bf16_bytes": int(T) * int(V) * 2},
        "gpu_launches": int(step_launches * n),
        "clocks": clocks,
        "e2e": e2e,
    }
    return out


def run_teacher_topk(args, w, world, rank, local_rank):
    """The teacher-side top-K cache producer on the workload's shape (h, W of a
    synthetic teacher): one step = one kd_teacher_topk call over all T rows
    (per row chunk: one logit pass that also stores the chunk's fp32 logits,
    the threshold, a candidate scan of the stored logits, the selection).
    Roofline of the logit pass: tensor, 2 d V FLOPs per row; the scan is
    reported against HBM, 4 V bytes read per row (from the library's launch
    events)."""
    import chunked_top_kl_logit_b300 as kd
    from synth import make_inputs
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    x = make_inputs(w.replace(idx_kind="uniform"), seed=args.seed + rank, device=dev)
    h, W = x["h"].to(dev), x["W"].to(dev)
    T, d, V, K = w.T, w.d, w.V, w.K
    chunk = args.chunk or 4096
    ws = torch.empty(kd.kd_teacher_topk_workspace_size(T, V, d, K, chunk), dtype=torch.uint8,
                     device=dev)
    idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    val = torch.empty(T, K, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        kd.kd_teacher_topk(h, W, K, w.tau, chunk, idx, val, lse, ws=ws, dev_status=st)

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize()
    kd.check_device_status(st, "teacher_topk warm-up")
    n = args.steps
    chunks = (T + chunk - 1) // chunk
    sampler = ClockSampler(None).start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    kd.kd_timing_start(2 * chunks * n + 4)
    e0.record()
    for _ in range(n):
        step()
    e1.record()
    torch.cuda.synchronize()
    kd.kd_timing_stop()
    barrier(world)
    clocks = sampler.stop()
    kd.check_device_status(st, "teacher_topk")
    passes = {name: kd.kd_timing_query(kid) for name, kid in kd.PRODUCER_KERNELS.items()}
    kd.kd_timing_release()
    ms = e0.elapsed_time(e1)
    max_sec = max_over_ranks(ms / 1e3, world, device=dev)
    peaks, src = load_peaks()
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    cnt, kms = passes["topk_pass1"]
    kern = {"topk_pass1": {"launches": cnt, "ms_per_step": kms / n,
                           "tflops": 2.0 * T * d * V * n / (kms / 1e3) / 1e12 if kms > 0 else None}}
    cnt, kms = passes["topk_scan"]
    scan_gbs = 4.0 * T * V * n / (kms / 1e3) / 1e9 if kms > 0 else None
    kern["topk_scan"] = {"launches": cnt, "ms_per_step": kms / n, "gbs": scan_gbs,
                         "hbm_frac": scan_gbs / hbm if scan_gbs else None}
    return {
        "metric": "teacher top-K cache producer rows/s", "op": "teacher_topk",
        "value": job_throughput(T * n, world, max_sec), "unit": "rows/s", "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": max_sec * 1e3 / n,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "T": T, "V": V, "d": d, "K": K, "tau": w.tau,
                   "chunk": chunk, "l2": "inputs larger than L2 (W alone is V*d*2 B)"},
        "tflops_logits": 2.0 * T * d * V / (max_sec / n) / 1e12,
        "memory": {"workspace_bytes": int(ws.numel())},
        "kernels": kern,
        "roofline": {"kernel": "kd_gemm_kernel<5> (topk_pass1)",
                     "bound": "tensor", "achieved": kern["topk_pass1"]["tflops"],
                     "peak": sustained, "unit": "TFLOP/s",
                     "frac": kern["topk_pass1"]["tflops"] / sustained,
                     "peak_kind": f"bf16 sustained, {src}",
                     "traffic": load_traffic("topk_pass1", w.name, chunk)},
        "clocks": clocks,
        "gpu_launches": 4 * chunks * n,
    }


def run_entropy_filter(args, w, world, rank, local_rank):
    """The teacher-entropy token filter on the workload's teacher cache: one
    step = one kd_entropy_filter call (entropy of every row + exact selection),
    inputs resident in HBM.  Roofline: HBM, algorithmic bytes = the teacher
    logits read once + valid_in read + valid_out written."""
    import chunked_top_kl_logit_b300 as kd
    from synth import make_inputs
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    x = make_inputs(w.replace(idx_kind="uniform"), seed=args.seed + rank, device=dev)
    tl = x["teacher_logits"].to(dev)
    valid = x["valid"].to(dev)
    T, K = tl.shape
    out = torch.empty(T, dtype=torch.uint8, device=dev)
    ent = torch.empty(T, dtype=torch.float32, device=dev)
    ws = torch.empty(kd.kd_entropy_filter_workspace_size(T), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # 256 MB > L2

    def step():
        kd.kd_entropy_filter(tl, valid, w.tau, 7, 10, out, ent, ws=ws, dev_status=st)

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize()
    n = args.steps
    e = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    barrier(world)
    for i in range(n):
        flush.zero_()
        e[i][0].record()
        step()
        e[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    ms = statistics.mean(a.elapsed_time(b) for a, b in e)
    max_sec = max_over_ranks(ms / 1e3 * n, world, device=dev)
    alg_bytes = T * K * 4 + 2 * T
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = alg_bytes / (ms / 1e3) / 1e9
    return {
        "metric": "teacher-entropy token filter rows/s", "op": "entropy_filter",
        "value": job_throughput(T * n, world, max_sec), "unit": "rows/s", "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": max_sec * 1e3 / n,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "T": T, "K": K, "tau": w.tau, "keep": "7/10",
                   "l2": "256 MB buffer written between timed calls"},
        "roofline": {"kernel": "kd_entropy_kernel + kd_entropy_select_kernel", "bound": "hbm",
                     "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "peak_kind": f"HBM copy bandwidth, {src}", "traffic": None,
                     "bytes_per_launch": alg_bytes},
        "gpu_launches": 2 * n,
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="b300", choices=["b300", "reference"])
    ap.add_argument("--workload", default="ctx_32k")
    ap.add_argument("--chunk", type=int, default=0)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--op", default="loss", choices=["loss", "entropy_filter", "teacher_topk"],
                    help="loss: the fused top-K KL forward + backward (headline); "
                         "entropy_filter: the mask producer alone; "
                         "teacher_topk: the teacher-side top-K cache producer")
    ap.add_argument("--variant", default="main", choices=["main", "residual"],
                    help="main: teacher renormalised over its top-K; residual: the teacher's "
                         "full-vocabulary normaliser and an 'everything else' outcome")
    ap.add_argument("--api", default="fused", choices=["split", "fused"],
                    help="fused: one kd_topk_kl_forward_backward call per step (the single "
                         "sweep, each row's logits formed once); split: kd_topk_kl_forward + "
                         "kd_topk_kl_backward per step (the backward recomputes the logits)")
    ap.add_argument("--valid-rows-only", action="store_true",
                    help="fused API only: pass KD_VALID_ROWS_ONLY, so that the logits of "
                         "masked rows are not formed (their lse is NaN)")
    ap.add_argument("--cpu-rows", type=int, default=1024)
    ap.add_argument("--ref-rows", type=int, default=256)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    from synth import workload
    w = workload(args.workload)
    rank, world, local_rank = rank_info()

    if args.impl == "reference":
        out = run_reference(args, w, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0

    dist_setup(world, "nccl")
    if args.op in ("entropy_filter", "teacher_topk"):
        run = run_entropy_filter if args.op == "entropy_filter" else run_teacher_topk
        out = run(args, w, world, rank, local_rank)
        if rank == 0:
            print(json.dumps(out), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    out = run_ours(args, w, world, rank, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu:
            rows = args.cpu_rows
            sec = oracle_step_seconds(oracle_sample(w, rows))
            out["cpu_baseline"] = {"value": rows / sec, "unit": "tokens/s", "cores": blas_threads(),
                                   "kind": "oracle",
                                   "sample": f"fp64 oracle fwd+bwd on a {rows}-row sample of "
                                             f"{w.name} (full V, d), {sec:.1f} s"}
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
