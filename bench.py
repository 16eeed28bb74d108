"""Benchmark: fused Adam/AdamW shard step on GB300, capturable vs regular.

Default workload: 201 fp32 tensors x 20,971,520 elements (the tensor list of
the TE issue's adam_bench.py), AdamW, lr 1.6e-3, betas (0.9, 0.95),
eps 1e-8, wd 0.1, no param-out copy: 28 algorithmic bytes per element,
118.03 GB per step, far larger than the 129 MB L2, so no flush is needed
between steps.

One step = one fadam_step launch over the whole shard (a single persistent
kernel).  Timed with CUDA events on the launching stream, per launch, after
warm-up; the headline value is the capturable path's achieved HBM GB/s
(algorithmic bytes / mean launch time).  Also measured: the regular path,
a CUDA-graph replay of the capturable step, the in-kernel inf/nan screen,
and an end-to-end number through fadam_step_host_grads (host gradients
copied in from pinned memory, the step, the step counter read back).

`--impl reference` times the CPU oracle instead (the reference arm): each
step is a bounded sample of the same workload on the host cores.

Multi-GPU (torchrun): every rank updates its own shard of the same size
(weak scaling, no data-path collective); rank 0 prints the line with the
maximum time over ranks.
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
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "Adam step achieved HBM GB/s (fraction of GB300 peak) + Gparams/s, capturable vs regular"


# ---- distributed plumbing (timing only) ---------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value over ranks (timing reduction; not on the data path)."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate(bytes_per_rank: float, elems_per_rank: float, world: int, seconds: float) -> dict:
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return {"gbs": world * bytes_per_rank / seconds / 1e9,
            "gparams_per_s": world * elems_per_rank / seconds / 1e9}


# ---- clocks -------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (200 ms) of the benchmark's GPU during timed work."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        self.thread = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = ["-i", str(device_index)]
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}",
                    "--format=csv,noheader,nounits", "-lms", "200"]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, pw, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
                pw.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "power_w_max": max(pw), "reasons": sorted(reasons)}


# ---- timing helpers -----------------------------------------------------------

def time_launches(fn, steps: int, warmup: int, world: int):
    """Per-launch CUDA-event times (ms) of `fn` on the current stream, plus
    the bracketed wall time of the K timed steps (s)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        starts[i].record()
        fn()
        ends[i].record()
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return per, wall


def summarise(per_ms, bytes_per_step, elems, world, device):
    mean_ms = statistics.mean(per_ms)
    mean_ms = max_over_ranks(mean_ms, world, device)
    agg = aggregate(bytes_per_step, elems, world, mean_ms / 1e3)
    return {"ms_per_step": mean_ms, "min_ms": min(per_ms), "max_ms": max(per_ms),
            "gbs": agg["gbs"], "gparams_per_s": agg["gparams_per_s"]}


# ncu counters of the headline kernel (one capture of the large_uniform launch,
# with the hash of the kernel sources it was taken on)
PROFILE = os.path.join(ROOT, "profiles", "fadam_update_kernel_large_uniform_traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "include", "fadam.h")] + sorted(
    os.path.join(ROOT, "adamw_optimizer_step_persistent_gb300", "csrc", f)
    for f in os.listdir(os.path.join(ROOT, "adamw_optimizer_step_persistent_gb300", "csrc"))
    if f.endswith((".cu", ".cuh", ".h")))


def _code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace runs collapsed, so
    that edits to comments alone keep the hash (string literals in these
    sources hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """sha256 over the code of the CUDA library's sources, comments left out
    (decides whether a stored ncu traffic figure still describes the kernel
    that runs)."""
    import hashlib
    h = hashlib.sha256()
    for path in KERNEL_SOURCES:
        with open(path, encoding="utf-8") as fh:
            h.update(os.path.relpath(path, ROOT).encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()


def profiled_traffic(elements: int):
    """DRAM bytes (read + written) per launch from the committed ncu counters
    of the headline kernel, per element of the captured launch times the
    elements of this one, or None when the kernel sources changed since the
    capture (or there is none)."""
    try:
        with open(PROFILE) as fh:
            d = json.load(fh)
        if d.get("source_sha256") != kernel_source_hash():
            return None
        per_elem = (float(d["dram_bytes_read"]) + float(d["dram_bytes_write"])) / float(d["elements"])
    except (OSError, KeyError, ValueError, TypeError, ZeroDivisionError):
        return None
    return per_elem * elements


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "source": "fallback"}


def host_memory_allows(nbytes: int) -> bool:
    """True when nbytes of page-locked host memory stay within half of the
    memory the host has available now (unknown: assume it does)."""
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        return True
    return nbytes <= avail // 2


def e2e_fits(node_bytes: int, world: int, device=None) -> bool:
    """Whether the end-to-end leg can pin its host gradients on every node,
    as one decision for all ranks (the leg has barriers and a reduction, so
    no rank may skip it alone)."""
    veto = 0.0 if host_memory_allows(node_bytes) else 1.0
    return max_over_ranks(veto, world, device) == 0.0


# ---- CPU baseline (the oracle, as it stands) ----------------------------------

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _np_view(t: torch.Tensor) -> np.ndarray:
    """Zero-copy numpy view of a CPU tensor (16-bit floats as uint16 bits)."""
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


# bounded CPU samples of the four timed workloads: (name, spec factory,
# bytes per element), each about 0.15-0.35e9 elements
CPU_SAMPLES = [
    ("capturable_l2", lambda: workloads.capturable_l2(layers=1), 28),
    ("large_uniform", lambda: workloads.large_uniform(n_tensors=8), 28),
    ("remainder_shard", lambda: workloads.remainder_shard(total=150_000_000, n_views=64), 26),
    ("many_small", lambda: workloads.many_small(n_tensors=2500), 28),
]


def cpu_oracle_steps(spec, steps: int):
    """Time `steps` steps of the oracle's timed OpenMP build (-O3 -fopenmp;
    each tensor split across the host cores) on a CPU copy of `spec`.
    Returns (seconds per step, elements)."""
    import oracle

    shard = workloads.materialize(spec, "cpu")
    gdt = {torch.float32: oracle.DT_F32, torch.bfloat16: oracle.DT_BF16,
           torch.float16: oracle.DT_F16}
    groups = [oracle.Group(mode=oracle.MODE_ADAMW if g.adam_w_mode else oracle.MODE_L2,
                           bias_correction=1 if g.bias_correction else 0, beta1=g.betas[0],
                           beta2=g.betas[1], eps=g.eps, weight_decay=g.weight_decay, lr=g.lr,
                           grad_scale=spec.grad_scale) for g in spec.groups]
    work = []
    for i in shard.plan_order():
        if spec.sizes[i] == 0:
            continue
        grp = groups[spec.group_of[i]]
        g = _np_view(shard.grads[i])
        m, v = _np_view(shard.exp_avgs[i]), _np_view(shard.exp_avg_sqs[i])
        if spec.remainders:
            hi, rem = _np_view(shard.params[i]), shard.remainders[i].numpy()
            work.append(lambda k, a=(hi, rem, m, v, g), grp=grp: oracle.adam_rem(
                grp, k, a[0], a[1], a[2], a[3], a[4], gdt[spec.g_dtype], a[0], timed=True))
        else:
            p = _np_view(shard.params[i])
            out = _np_view(shard.params_out[i]) if shard.params_out[i] is not None else None
            odt = gdt[spec.out_dtype] if spec.out_dtype is not None else oracle.DT_NONE
            work.append(lambda k, a=(p, m, v, g, out), grp=grp, odt=odt: oracle.adam_f32(
                grp, k, a[0], a[1], a[2], a[3], gdt[spec.g_dtype], a[4], odt, timed=True))
    per_step = []
    for k in range(1, steps + 1):
        t0 = time.perf_counter()
        for w in work:
            w(k)
        per_step.append(time.perf_counter() - t0)
    return per_step, spec.n_elements


def cpu_baseline(steps: int = 3):
    """The oracle on the host cores: one bounded sample of each of the four
    timed workloads, a few steps each; the line's value is the large-uniform
    sample's (its workload)."""
    import oracle

    threads = oracle.timed_lib().oracle_omp_threads()
    per = {}
    for name, make_spec, bpe in CPU_SAMPLES:
        spec = make_spec()
        times, elems = cpu_oracle_steps(spec, steps)
        sec = statistics.median(times)
        per[name] = {"gbs": elems * bpe / sec / 1e9, "gparams_per_s": elems / sec / 1e9,
                     "s_per_step": sec, "elements": elems, "bytes_per_element": bpe,
                     "sample": f"{len(spec.sizes)} tensors of the {name} recipe"}
    head = per["large_uniform"]
    return {"value": head["gbs"], "unit": "GB/s", "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(), "gparams_per_s": head["gparams_per_s"],
            "build": "oracle C source, -O3 -fopenmp -ffp-contract=off -fno-math-errno "
                     "(vectorised; each tensor split across the OpenMP threads)",
            "sample": (f"8 of the 201 tensors x 20,971,520 fp32 elements "
                       f"({head['elements']} elements, {head['elements'] * 28 / 1e9:.2f} GB per "
                       f"step), median of {steps} steps; per-workload samples in 'workloads'"),
            "workloads": per}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle

    threads = oracle.timed_lib().oracle_omp_threads()
    spec = workloads.large_uniform(n_tensors=args.ref_tensors)
    per_step, elems = cpu_oracle_steps(spec, args.warmup + args.steps)
    timed = per_step[args.warmup:]
    sec = statistics.mean(timed)
    gbs = elems * 28 / sec / 1e9
    sample = (f"each step: {args.ref_tensors} of the 201 tensors x 20,971,520 fp32 elements "
              f"({elems} elements); the oracle's timed OpenMP build on {threads} threads "
              f"({cpu_model()})")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "large_uniform: 201 fp32 tensors x 20,971,520, AdamW "
                                   "(bounded sample per step)", "sample_elements": elems},
            "gparams_per_s": elems / sec / 1e9,
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- the GPU arm --------------------------------------------------------------

def run_gpu(args):
    from adamw_optimizer_step_persistent_gb300 import FusedAdamShard

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    device = torch.device("cuda", local)
    if args.workload == "large_uniform":
        spec = workloads.large_uniform(n_tensors=args.n_tensors or 201, numel=args.numel,
                                       seed=1237 + 1000 * rank)
    elif args.workload == "large_uniform_bf16_out":
        spec = workloads.large_uniform(n_tensors=args.n_tensors or 201, numel=args.numel,
                                       seed=1237 + 1000 * rank, out_dtype=torch.bfloat16)
    elif args.workload == "large_uniform_bf16_moments":
        spec = workloads.large_uniform(n_tensors=args.n_tensors or 201, numel=args.numel,
                                       seed=1237 + 1000 * rank, moment_dtype=torch.bfloat16)
    elif args.workload == "large_uniform_bf16_state" and args.n_tensors:
        spec = workloads.large_uniform(n_tensors=args.n_tensors, numel=args.numel,
                                       seed=1237 + 1000 * rank, state_dtype=torch.bfloat16,
                                       g_dtype=torch.bfloat16)
    elif args.workload == "scaled_state_shard":
        spec = workloads.scaled_state_shard(layers=args.layers or 8, seed=1241 + 1000 * rank)
    elif args.workload == "exchange_shard":
        spec = workloads.exchange_shard(layers=args.layers or 8, seed=1240 + 1000 * rank)
    elif args.workload == "remainder_shard" and args.total:
        spec = workloads.remainder_shard(total=args.total, seed=1238 + 1000 * rank)
    elif args.workload == "capturable_l2" and args.layers:
        spec = workloads.capturable_l2(layers=args.layers, seed=1236 + 1000 * rank)
    elif args.workload == "many_small" and args.n_tensors:
        spec = workloads.many_small(n_tensors=args.n_tensors, seed=1239 + 1000 * rank)
    else:
        spec = workloads.full_versions()[args.workload]
        spec.seed += 1000 * rank
    shard = workloads.materialize(spec, device)
    groups = shard.param_groups()
    kw = dict(remainders=spec.remainders, grad_scale=spec.grad_scale, recip_bc=args.recip_bc)

    # scaled state: every plan of the run steps the same p, m, v, so they
    # share one scales tensor too (a plan with a copy of its own would start
    # from scales that no longer match the state the previous plan left)
    scales = (shard.state_scales[shard.plan_order()].contiguous() if spec.scaled_state
              else None)

    def make(capturable, **more):
        if spec.scaled_state:
            more["state_scales"] = scales
        opt = FusedAdamShard(groups, capturable=capturable, **kw, **more)
        if args.start_step:  # a shard resumed this many steps into training
            opt.set_group_steps([args.start_step] * len(groups))
        if spec.exchange_ranks:  # the data-parallel exchange stand-in
            opt.set_exchange(shard.buckets["g"], list(shard.sources),
                             average=spec.exchange_average, out_shard=shard.buckets["p_out"],
                             dests=list(shard.dests))
        return opt

    cap = make(True)
    info = cap.info()
    bytes_step = info["bytes_per_step"]
    elems = info["n_elements"]
    if spec.scaled_state:
        # the rescale depends on every new value of a tensor: a second pass
        # reads p, m, v and g again (24 B per element for fp16 state, bf16 g)
        bytes_step += elems * (3 * shard.params[0].element_size() + shard.grads[0].element_size())
    if spec.exchange_ranks:
        gsz = shard.buckets["g"].element_size()
        # every step also writes the param-out copy to each destination
        bytes_step += elems * spec.exchange_dests * shard.buckets["p_out"].element_size()
        # fused: the R sources are read and the shard's g written, instead of g read
        exchange_bytes = bytes_step + elems * spec.exchange_ranks * gsz
        reduce_bytes = elems * (spec.exchange_ranks + 1) * gsz
    res = {}
    variants = args.variants.split(",")
    sampler = ClockSampler(local)
    sampler.start()
    if spec.exchange_ranks and "exchange" in variants:
        per, _ = time_launches(cap.step_reduce, args.steps, args.warmup, world)
        r = summarise(per, exchange_bytes, elems, world, device)
        r["bytes_per_step"] = exchange_bytes
        res["exchange"] = r
    if spec.exchange_ranks and "reduce" in variants:
        per, _ = time_launches(cap.grad_reduce, args.steps, args.warmup, world)
        r = summarise(per, reduce_bytes, elems, world, device)
        r["bytes_per_step"] = reduce_bytes
        res["reduce"] = r
    if spec.exchange_ranks and "accumulate" in variants:
        # a later micro-batch's reduce-scatter: the R sources read, the
        # shard's g read, added to and written back
        cap.set_accumulate(True)
        per, _ = time_launches(cap.grad_reduce, args.steps, args.warmup, world)
        cap.set_accumulate(False)
        acc_bytes = elems * (spec.exchange_ranks + 2) * gsz
        r = summarise(per, acc_bytes, elems, world, device)
        r["bytes_per_step"] = acc_bytes
        res["reduce_accumulate"] = r
    if spec.exchange_ranks and "clip_pipeline" in variants:
        # the data-parallel step with gradient clipping, captured as one
        # graph: the grad scale reset (the loss scaler's value), the
        # reduce-scatter stand-in, the shard's squared norm, the clip folded
        # into the grad scale, the step writing every destination
        gs0 = float(spec.grad_scale)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())

        def pipeline():
            cap.set_grad_scale(gs0)
            cap.grad_reduce()
            cap.clip_apply(cap.grad_norm_sq(), 1.0)
            cap.step()

        with torch.cuda.stream(s):
            pipeline()
        torch.cuda.current_stream().wait_stream(s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            pipeline()
        per, _ = time_launches(graph.replay, args.steps, args.warmup, world)
        pipe_bytes = reduce_bytes + elems * gsz + bytes_step
        r = summarise(per, pipe_bytes, elems, world, device)
        r["bytes_per_step"] = pipe_bytes
        r["launches"] = "grad scale fill, fadam_grad_reduce, fadam_grad_sumsq, fadam_clip_apply, fadam_step"
        res["clip_pipeline"] = r
        del graph
    if "capturable" in variants:
        per, _ = time_launches(cap.step, args.steps, args.warmup, world)
        res["capturable"] = summarise(per, bytes_step, elems, world, device)
    if "regular" in variants:
        reg = make(False)
        per, _ = time_launches(reg.step, args.steps, args.warmup, world)
        res["regular"] = summarise(per, bytes_step, elems, world, device)
        reg.close()
    if "graph" in variants:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            cap.step()
        torch.cuda.current_stream().wait_stream(s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cap.step()
        per, _ = time_launches(graph.replay, args.steps, args.warmup, world)
        res["graph_replay"] = summarise(per, bytes_step, elems, world, device)
        del graph
    if "check_finite" in variants:
        chk = make(True, check_finite=True)
        per, _ = time_launches(chk.step, args.steps, args.warmup, world)
        r = summarise(per, bytes_step, elems, world, device)
        r["gbs_including_screen"] = r["gbs"] * (bytes_step + chk.info()["check_bytes_per_step"]) / bytes_step
        res["check_finite"] = r
        chk.close()
    if "norm" in variants:
        per, _ = time_launches(cap.grad_norm_sq, args.steps, args.warmup, world)
        gbytes = elems * shard.grads[0].element_size()
        r = summarise(per, gbytes, elems, world, device)
        r["bytes_per_step"] = gbytes
        res["grad_norm"] = r
    clocks = sampler.stop()

    e2e = None
    host_bytes = sum(g.numel() * g.element_size() for g in shard.grads)
    ranks_here = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    fits = e2e_fits(ranks_here * host_bytes, world, device)
    if "e2e" in variants and not fits:
        # every rank of the node pins its own copy of the gradients: leave
        # the leg out rather than exhaust the host
        e2e = {"value": None, "unit": "GB/s", "h2d_bytes_per_step": host_bytes,
               "d2h_bytes_per_step": 4 * len(groups),
               "skipped": f"{ranks_here} ranks x {host_bytes / 1e9:.1f} GB of pinned host "
                          "gradients exceed half of the node's available memory"}
    elif "e2e" in variants:
        host = [shard.grads[i].cpu().pin_memory() for i in shard.plan_order()]
        for _ in range(max(1, args.warmup // 2)):
            cap.step_from_host(host)
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            cap.step_from_host(host)
        barrier(world)
        sec = max_over_ranks((time.perf_counter() - t0) / args.steps, world, device)
        agg = aggregate(bytes_step, elems, world, sec)
        e2e = {"value": agg["gbs"], "unit": "GB/s", "ms_per_step": sec * 1e3,
               "h2d_bytes_per_step": int(sum(g.numel() * g.element_size() for g in host)),
               "d2h_bytes_per_step": 4 * len(groups),
               "path": "fadam_step_host_grads: pinned host grads read in place by the update "
                       "(zero copy over the host link, overlapping the p/m/v traffic), one "
                       "launch, step counter -> host, stream sync"}
        del host

    head = (res.get("exchange") or res.get("capturable") or res.get("regular")
            or next(iter(res.values())))
    head_bytes = head.get("bytes_per_step", bytes_step)
    peaks = measured_peaks()
    achieved = head_bytes / (head["ms_per_step"] / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": head["gbs"], "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": (f"large_uniform: {args.n_tensors or 201} fp32 tensors x {args.numel}, "
                                "AdamW lr 1.6e-3 betas (0.9,0.95) eps 1e-8 wd 0.1, no param-out"
                                if args.workload == "large_uniform" else
                                f"{spec.name}: {len(spec.sizes)} tensors, {spec.n_elements} elements"
                                + (f", fp32 state, bf16 g and param-out, {spec.exchange_ranks} ranks "
                                   f"averaged into the shard, {spec.exchange_dests} destinations"
                                   if spec.exchange_ranks else "")),
                   "elements_per_step": elems, "bytes_per_step": head_bytes,
                   "bytes_per_element": head_bytes / elems, "grid": info["grid"],
                   "block": info["block"], "items": info["n_items"],
                   "l2": "inputs larger than L2 (no flush needed)",
                   "start_step": args.start_step,
                   "recip_bc": args.recip_bc,
                   "parallelism": f"weak: one shard per GPU x {world}"},
        "fraction_of_peak": head["gbs"] / world / peaks["hbm_gbs"],
        "gparams_per_s": head["gparams_per_s"],
        "variants": res,
        "capturable_vs_regular": (res["capturable"]["ms_per_step"] / res["regular"]["ms_per_step"]
                                  if "capturable" in res and "regular" in res else None),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "peak_source": peaks["source"],
                     "traffic": (profiled_traffic(elems) if args.workload == "large_uniform" else None),
                     "kernel": "fadam_update_kernel (bulk-copy pipeline)"},
        "clocks": clocks,
        "gpu_launches": args.steps,
    }
    if e2e:
        line["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == "large_uniform":
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    cap.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large_uniform",
                    choices=["large_uniform", "capturable_l2", "remainder_shard", "many_small",
                             "large_uniform_bf16_state", "large_uniform_bf16_moments",
                             "large_uniform_bf16_out",
                             "exchange_shard", "scaled_state_shard"])
    ap.add_argument("--n-tensors", type=int, default=None,
                    help="tensor count of large_uniform[_bf16_state|_bf16_moments|_bf16_out] (201) or "
                         "many_small (20000)")
    ap.add_argument("--numel", type=int, default=320 * 65536)
    ap.add_argument("--total", type=int, default=None,
                    help="elements of the remainder_shard bucket (1,200,000,000)")
    ap.add_argument("--layers", type=int, default=None,
                    help="layers of the capturable_l2 / exchange_shard / scaled_state_shard "
                         "layer list (8)")
    ap.add_argument("--variants", default="capturable,regular,graph,check_finite,norm,e2e",
                    help="also exchange,reduce,accumulate,clip_pipeline on the exchange_shard "
                         "workload")
    ap.add_argument("--start-step", type=int, default=0,
                    help="steps already taken by every group when timing starts (0: a fresh "
                         "shard; from 165 / 338 / 17,321 the bias corrections of beta 0.9 / "
                         "0.95 / 0.999 are 1 in float)")
    ap.add_argument("--recip-bc", action="store_true",
                    help="FADAM_RECIP_BC: the 16-bit state forms multiply by reciprocal bias "
                         "corrections (within the tolerance, not bit-identical)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-tensors", type=int, default=4)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
