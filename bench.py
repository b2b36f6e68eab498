#!/usr/bin/env python3
"""Throughput of the fused partitioned mixed-precision ZeRO step on GB300.

Default workload: flat psi = 1.5e9 parameters, N = 8 simulated ranks, stage 1
(P_os), fp16 gradients N(0, 1e-3^2) x loss scale 2^16, warm m/v, four grad
sets cycled (the third carries one +inf in rank 5, so every fourth step is
the overflow-skip path).  One bench step = one zero_step call over one set:
reduce-scatter + unscale + overflow flag + global norm + AdamW + cast +
all-gather into 8 replicas, all inputs resident in HBM (84 GB per step, far
larger than L2).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
a bounded slab of the same workload instead (it needs no GPU).
Other workloads (``--workload toy|gpt2|llama7b|sweep``) print lines of the
same form for the tables in the docs.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "params/sec of fused ZeRO step at N ranks; achieved HBM GB/s vs GB300 peak"
RESULT_BYTES = 56   # sizeof(zero_result_t)


# ---------------------------------------------------------------- environment
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("zero_kernels.cu", "zero_internal.h", "zero_device.cuh"):
        with open(os.path.join(ROOT, "zero_partitioned_mixed_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(summary: str):
    """DRAM bytes per launch from a committed ncu figure (JSON), if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    val = d.get("dram_bytes_per_launch_full_size")
    return float(val) if val is not None else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [float(p[1]) for p in self.samples if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for p in self.samples if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in self.samples for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The slowest rank's value (timings are max-reduced across ranks)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world_size: int, seconds: float) -> float:
    """Whole-job throughput: every rank processed units_per_rank in the max-over-ranks time."""
    return units_per_rank * world_size / seconds


# ---------------------------------------------------------------- CPU oracle timing
def oracle_case(psi_sample: int, n: int, stage: int, dtype: str, seed: int = 0):
    """The oracle's state, 16-bit gradients and hyper-parameters for a slab of
    the flat workload (its distributions: master N(0, 0.02^2), warm m/v,
    gradients N(0, 1e-3^2) x 2^16)."""
    import numpy as np
    import oracle as O
    rng = np.random.default_rng(seed)
    part = O.partition(psi_sample, n, 8)
    master = rng.normal(0, 0.02, psi_sample).astype(np.float32)
    m = rng.normal(0, 1e-4, psi_sample).astype(np.float32)
    v = np.abs(rng.normal(0, 1e-6, psi_sample)).astype(np.float32)
    st = O.init_state(stage, dtype, part, master, m, v, loss_scale=65536.0)
    g = np.zeros((n, part.psi_pad), np.float32)
    g[:, :psi_sample] = rng.normal(0, 1e-3, (n, psi_sample)) * 65536.0
    gb = O.rne16(g, dtype)
    return st, gb, O.Hyper()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_worker(conn, psi_sample, n, stage, dtype, seed):
    """One process of OraclePool: builds its own slab, then runs one oracle
    step per request and replies with the step's duration."""
    import oracle as O
    st, gb, h = oracle_case(psi_sample, n, stage, dtype, seed)
    conn.send("ready")
    while conn.recv():
        t0 = time.perf_counter()
        st, _ = O.step(st, gb, h)
        conn.send(time.perf_counter() - t0)
    conn.close()


class OraclePool:
    """The unmodified oracle in P processes (spawned: no process is forked
    from one that has used the GPU), each on its own slab of the workload.
    A pool step sends every process one step at once and lasts until the
    slowest replies, so P slabs are processed per pool step."""

    def __init__(self, procs: int, psi_sample: int, n: int, stage: int, dtype: str):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        for i in range(procs):
            parent, child = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(child, psi_sample, n, stage, dtype, i), daemon=True)
            p.start()
            self.conns.append(parent)
            self.procs.append(p)
        for c in self.conns:
            if c.recv() != "ready":
                raise RuntimeError("oracle worker failed to start")

    def step(self) -> float:
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(True)
        for c in self.conns:
            c.recv()
        return time.perf_counter() - t0

    def close(self):
        for c in self.conns:
            try:
                c.send(False)
            except OSError:
                pass
        for p in self.procs:
            p.join(timeout=10)
            if p.is_alive():
                p.terminate()


def oracle_timing_all_cores(psi_sample: int, n: int, stage: int, dtype: str, steps: int, warmup: int,
                            budget_s: float = None, procs: int = None):
    """Aggregate oracle throughput with one process per host core (see OraclePool)."""
    procs = procs or host_cores()
    pool = OraclePool(procs, psi_sample, n, stage, dtype)
    try:
        for _ in range(warmup):
            pool.step()
        times = []
        t_start = time.perf_counter()
        for i in range(steps):
            times.append(pool.step())
            if budget_s is not None and time.perf_counter() - t_start > budget_s and i >= 2:
                break
    finally:
        pool.close()
    total = sum(times)
    return {"value": procs * psi_sample * len(times) / total, "steps": len(times), "seconds": total,
            "ms_per_step": 1e3 * total / len(times), "cores": procs}


def oracle_timing(psi_sample: int, n: int, stage: int, dtype: str, steps: int, warmup: int,
                  budget_s: float = None):
    """Time the oracle's step on a slab of psi_sample elements (numpy, one core)."""
    import oracle as O
    st, gb, h = oracle_case(psi_sample, n, stage, dtype)
    for _ in range(warmup):
        st, _ = O.step(st, gb, h)
    times = []
    t_start = time.perf_counter()
    for i in range(steps):
        t0 = time.perf_counter()
        st, _ = O.step(st, gb, h)
        times.append(time.perf_counter() - t0)
        if budget_s is not None and time.perf_counter() - t_start > budget_s and i >= 2:
            break
    total = sum(times)
    return {"value": psi_sample * len(times) / total, "steps": len(times), "seconds": total,
            "ms_per_step": 1e3 * total / len(times)}


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    psi_s = 1 << 20
    r = oracle_timing_all_cores(psi_s, 8, 1, "fp16", args.steps, args.warmup)
    line = {
        "impl": "reference", "metric": METRIC, "value": r["value"], "unit": "params/s",
        "n_gpus": ws, "steps": r["steps"], "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "flat_psi1.5e9_n8_stage1_fp16_ls65536", "n_ranks": 8, "stage": 1,
                   "parallelism": "replicas only"},
        "cpu_baseline": {"value": r["value"], "unit": "params/s", "cores": r["cores"], "kind": "oracle",
                         "sample": f"{r['cores']} processes, each an oracle stage-1 step per bench step on "
                                   f"its own slab of {psi_s} parameters x 8 ranks (numpy, one thread "
                                   "each), same distributions as the workload"},
        "e2e": {"value": r["value"], "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU workloads
def setup_flat15b(Z, S, torch, psi=None):
    """Buffers and four resident gradient sets of the 1.5B stage-1 workload
    (psi overrides the size for small profiling runs)."""
    import dataclasses
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    w = S.FLAT15B
    if psi is not None and psi != w.psi:
        w = dataclasses.replace(w, psi=psi, name=f"flat_psi{psi}_n8_stage1_fp16_ls65536")
    buf = RankBuffers(w.psi, w.n_ranks, w.stage, w.dtype, double_buffer=True, alloc_grads=False)
    P = buf.psi_pad
    mv, mm, vv = buf.state(0)
    S.draw_master(w, mv, w.psi)
    S.draw_moments(w, mm, vv, w.psi)
    buf.params[:, :P].copy_(mv.to(S.torch_dtype(w.dtype)).unsqueeze(0).expand(w.n_ranks, P))
    td = S.torch_dtype(w.dtype)
    sets = torch.empty((w.steps, w.n_ranks, buf.stride), dtype=td, device="cuda")
    scale = w.loss_scale
    for k in range(w.steps):
        for r in range(w.n_ranks):
            S.draw_grads(w, sets[k, r], w.psi, k + 1, r, scale)
        if k + 1 == w.inject_step:
            S.inject_inf(w, sets[k, w.inject_rank], w.psi)
            scale = max(scale / 2, 1.0)   # the step after the skip is drawn at the halved scale
    buf.set_scaler(w.loss_scale, 0, 0)
    torch.cuda.synchronize()
    return w, buf, sets


def run_ours(args, ws, rank, local):
    import torch
    import zero_partitioned_mixed_gb300 as Z
    from zero_partitioned_mixed_gb300 import synth as S
    from zero_partitioned_mixed_gb300.build import build_library

    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or ws > 1:
        build_library()
    if ws > 1:
        dist.barrier()

    w, buf, sets = setup_flat15b(Z, S, torch, args.psi)
    N, P = w.n_ranks, buf.psi_pad
    step_mode = Z.ZERO_MODE_SPECULATIVE_STAGED if args.mode == "staged" else Z.ZERO_MODE_AUTO
    hyp = Z.hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm, step_mode)
    stream = torch.cuda.current_stream()
    nsets = sets.shape[0]

    def rows(k):
        return [sets[k, r] for r in range(N)]

    for i in range(args.warmup):
        buf.step(hyp, rows(i % nsets))
    torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kinds = []
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(K):
            k = (args.warmup + i) % nsets
            kinds.append(k)
            ev[i][0].record(stream)
            buf.step(hyp, rows(k))
            ev[i][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    if ws > 1:
        total_ms = max_over_ranks(total_ms, dist, "cuda")
    status = buf.status()

    inject_set = w.inject_step - 1
    applied_ms = [t for t, k in zip(step_ms, kinds) if k != inject_set]
    skipped_ms = [t for t, k in zip(step_ms, kinds) if k == inject_set]
    alg_bytes = (4 * N + 24) * P                 # per applied step: 2N + 12 read, 12 + 2N write
    kernel_ms = statistics.mean(applied_ms) if applied_ms else statistics.mean(step_ms)
    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9
    # the committed full-size traffic figure is the plain-load kernel's
    traffic = ncu_traffic("step_spec_flat1.5b_n8.json") if args.mode != "staged" else None

    value = job_throughput(w.psi * K, ws, total_ms * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage_dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "psi": w.psi, "n_ranks": N, "stage": w.stage,
                   "mode": "speculative, staged through shared memory" if args.mode == "staged" else "speculative",
                   "grad_sets": nsets, "overflow_every": f"set {inject_set + 1} of {nsets} (+inf in rank 5)",
                   "l2": f"inputs larger than L2: {alg_bytes / 1e9:.1f} GB per step, no flush needed",
                   "parallelism": "replicas only" if ws > 1 else "1 GPU"},
        "hbm_gbs_applied_step": achieved,
        "ms_per_applied_step": kernel_ms,
        "ms_per_skipped_step": statistics.mean(skipped_ms) if skipped_ms else None,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "k_step_tma (fp16, 8-wide)" if args.mode == "staged" else "k_step_spec (fp16, 8-wide)",
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "peak_source": f"{peak_src} hbm_gbs (copy)"},
        "gpu_launches": 3 * K,   # per step: the step kernel, the fixup, the commit
        "status_after": {k: status[k] for k in ("steps_applied", "steps_skipped", "loss_scale")},
    }
    c = clocks.summary()
    line["clocks"] = c

    if not args.no_e2e:
        line["e2e"] = e2e_flat(args, w, buf, sets, hyp, stream, torch, ws, dist)
    del sets
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline and ws >= 1:
        one = oracle_timing(1 << 21, 8, 1, "fp16", 200, 1, budget_s=10.0)
        r = oracle_timing_all_cores(1 << 21, 8, 1, "fp16", 200, 1, budget_s=10.0)
        line["cpu_baseline"] = {"value": r["value"], "unit": "params/s", "cores": r["cores"], "kind": "oracle",
                                "sample": f"{r['steps']} steps of {r['cores']} processes, each running the "
                                          "oracle's stage-1 step on its own slab of 2^21 parameters x 8 "
                                          "ranks (numpy, one thread each)",
                                "one_core": {"value": one["value"], "unit": "params/s", "cores": 1,
                                             "sample": f"{one['steps']} oracle stage-1 steps on one slab of "
                                                       "2^21 parameters x 8 ranks, one process"}}
    buf.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def e2e_flat(args, w, buf, sets, hyp, stream, torch, ws, dist):
    """Same step through the public API with the gradients coming from pinned host memory.

    Three ways to bring a step's 24 GB of gradients in, each timed with the
    step and the device->host read of its result:
      copy     one cudaMemcpyAsync of all N rank rows, then zero_step;
      streams  one copy per rank row spread over four side streams, then zero_step;
      direct   zero_step reads the pinned host rows itself (unified addresses,
               over NVLink-C2C), so the transfer overlaps the HBM stream.
    The line's value is the fastest; every mode is reported.
    """
    N = w.n_ranks
    try:
        host = torch.empty((N, buf.stride), dtype=sets.dtype, pin_memory=True)
    except Exception as e:  # not enough pinnable host memory
        return {"value": None, "unit": "params/s", "error": f"pinned host buffer: {e}"[:200]}
    host.copy_(sets[0])
    dev = sets[0]
    K = max(3, min(args.steps, 10))
    side = [torch.cuda.Stream() for _ in range(4)]

    def step_copy():
        dev.copy_(host, non_blocking=True)
        buf.step(hyp, [dev[r] for r in range(N)])

    def step_streams():
        ev = torch.cuda.Event()
        ev.record(stream)
        done = []
        for r in range(N):
            s = side[r % len(side)]
            s.wait_event(ev)
            with torch.cuda.stream(s):
                dev[r].copy_(host[r], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s)
                done.append(e)
        for e in done:
            stream.wait_event(e)
        buf.step(hyp, [dev[r] for r in range(N)])

    def step_direct():
        buf.step(hyp, [host[r] for r in range(N)])

    out = {}
    for name, fn in (("copy", step_copy), ("streams", step_streams), ("direct", step_direct)):
        fn()
        buf.status(stream)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(K):
            fn()
            buf.status(stream)          # device->host read of the step's result, synchronises
        t = time.perf_counter() - t0
        if ws > 1:
            t = max_over_ranks(t, dist, "cuda")
        out[name] = job_throughput(w.psi * K, ws, t)
    del host
    best = max(out, key=out.get)
    return {"value": out[best], "unit": "params/s", "mode": best, "modes": out,
            "h2d_bytes_per_step": N * buf.stride * 2, "d2h_bytes_per_step": RESULT_BYTES, "steps": K}


# ---------------------------------------------------------------- other workloads
class CallTimer:
    """Sums the CUDA-event durations of library calls made on the current stream."""

    def __init__(self, torch):
        self.torch = torch
        self.pairs = []

    def __enter__(self):
        a = self.torch.cuda.Event(enable_timing=True)
        b = self.torch.cuda.Event(enable_timing=True)
        a.record()
        self.cur = (a, b)
        return self

    def __exit__(self, *exc):
        self.cur[1].record()
        self.pairs.append(self.cur)
        return False

    def total_ms(self):
        self.torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in self.pairs)


def _step_ms(parts: dict, wall: CallTimer, steps: int, flushed: bool) -> float:
    """ms per step of a multi-call step: the device time from the step's first
    call to its last (gaps between calls included), or, when an L2 flush runs
    between the calls, the sum of the calls' own durations.  Records which
    into `parts`, with the per-call sum beside it."""
    calls = sum(v for k, v in parts.items() if k.endswith("_ms"))
    parts["calls_ms"] = calls
    if flushed:
        parts["timing"] = "sum of the calls' durations (L2 flush between calls excluded)"
        return calls
    parts["timing"] = "first call to last call of each step, gaps included"
    return wall.total_ms() / steps


def _line(workload, value, ms, steps, warmup, bytes_per_step, dtype, extra=None):
    peaks, src = measured_peaks()
    gbs = bytes_per_step / (ms * 1e-3) / 1e9
    out = {"metric": METRIC, "value": value, "unit": "params/s", "n_gpus": 1, "steps": steps,
           "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f32", "storage_dtype": dtype, "data": "synthetic",
           "config": {"workload": workload}, "hbm_gbs": gbs,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes_per_step": bytes_per_step,
                        "peak_source": f"{src} hbm_gbs (copy)"}}
    if extra:
        out["config"].update(extra)
    return out


def _bytes_delta(buf, before):
    b = buf.bytes_moved()
    return (b["hbm_read_total"] + b["hbm_write_total"]) - before


def _bytes_total(buf):
    b = buf.bytes_moved()
    return b["hbm_read_total"] + b["hbm_write_total"]


def bench_dense(w, stage, steps, warmup, torch, S, Z, flush_l2=False, sets_max=5, mode=None):
    """Stages 0-2: resident gradient sets, one zero_step per bench step
    (mode: a ZERO_MODE_*, default AUTO)."""
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    buf = RankBuffers(w.psi, w.n_ranks, stage, w.dtype, double_buffer=stage != 0, alloc_grads=False)
    P, N = buf.psi_pad, w.n_ranks
    td = S.torch_dtype(w.dtype)
    mv, mm, vv = buf.state(0)
    if stage == 0:
        S.draw_master(w, mv[0], w.psi)
        S.draw_moments(w, mm[0], vv[0], w.psi)
        mv[1:].copy_(mv[0].expand(N - 1, P)); mm[1:].copy_(mm[0].expand(N - 1, P)); vv[1:].copy_(vv[0].expand(N - 1, P))
        buf.params[:, :P].copy_(mv.to(td))
    else:
        S.draw_master(w, mv, w.psi)
        S.draw_moments(w, mm, vv, w.psi)
        buf.params[:, :P].copy_(mv.to(td).unsqueeze(0).expand(N, P))
    shapes = S.shapes_of(w)
    sv = S.fan_in_scale(shapes, "cuda") if (w.fan_in_scaled and shapes) else None
    nsets = max(1, min(w.steps, sets_max))
    sets = torch.empty((nsets, N, buf.stride), dtype=td, device="cuda")
    for k in range(nsets):
        for r in range(N):
            S.draw_grads(w, sets[k, r], w.psi, k + 1, r, w.loss_scale, sv)
    del sv
    buf.set_scaler(w.loss_scale, 0, 0)
    hyp = Z.hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm,
                  Z.ZERO_MODE_AUTO if mode is None else mode)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if flush_l2 else None
    rows = lambda k: [sets[k, r] for r in range(N)]
    for i in range(warmup):
        buf.step(hyp, rows(i % nsets))
    timer = CallTimer(torch)
    before = _bytes_total(buf)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        with timer:
            buf.step(hyp, rows((warmup + i) % nsets))
    ms = timer.total_ms() / steps
    per_step = _bytes_delta(buf, before) / steps
    st = buf.status()
    buf.close()
    del sets
    torch.cuda.empty_cache()
    return ms, per_step, st


def bench_stage3(w, buckets, steps, warmup, torch, S, Z, flush_l2=False, fused=True):
    """ZeRO-3: per step, gather every bucket (forward), then per bucket in reverse
    gather again and reduce-scatter, then finish the step.  One drawn gradient
    buffer of the largest bucket is reused for every bucket (timing only).
    fused: in backward each reduce-scatter carries the next bucket's gather
    (zero_reduce_scatter_gather_bucket), into two alternating output sets."""
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    buf = RankBuffers(w.psi, w.n_ranks, 3, w.dtype, double_buffer=(w.max_norm == 0))
    P, N = buf.psi_pad, w.n_ranks
    td = S.torch_dtype(w.dtype)
    mv, mm, vv = buf.state(0)
    S.draw_master(w, mv, w.psi)
    S.draw_moments(w, mm, vv, w.psi)
    buf.params[:P].copy_(mv.to(td))
    lmax = max(b - a for a, b in buckets)
    lpad = (lmax + 7) // 8 * 8
    gbuf = torch.empty((N, lpad), dtype=td, device="cuda")
    for r in range(N):
        S.draw_grads(w, gbuf[r], lmax, 1, r, w.loss_scale)
    outs = torch.empty((2 if fused else 1, N, lpad), dtype=td, device="cuda")
    buf.set_scaler(w.loss_scale, 0, 0)
    hyp = Z.hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm,
                  Z.ZERO_MODE_AUTO)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if flush_l2 else None
    grows = Z.pointer_array([gbuf[r] for r in range(N)])
    orows = [Z.pointer_array([o[r] for r in range(N)]) for o in outs]
    back = list(reversed(buckets))

    def one_step(tg, tr, tf):
        for (a, b) in buckets:
            if flush is not None:
                flush.zero_()
            with tg:
                buf.gather(a, b, orows[0])
        if fused:
            with tg:
                buf.gather(back[0][0], back[0][1], orows[0])
            for k, (a, b) in enumerate(back):
                if flush is not None:
                    flush.zero_()
                with tr:
                    if k + 1 < len(back):
                        buf.reduce_scatter_gather(a, b, grows, hyp, back[k + 1][0], back[k + 1][1],
                                                  orows[(k + 1) % 2])
                    else:
                        buf.reduce_scatter(a, b, grows, hyp)
        else:
            for (a, b) in back:
                if flush is not None:
                    flush.zero_()
                with tg:
                    buf.gather(a, b, orows[0])
                with tr:
                    buf.reduce_scatter(a, b, grows, hyp)
        with tf:
            buf.step(hyp)

    for _ in range(warmup):
        one_step(CallTimer(torch), CallTimer(torch), CallTimer(torch))
    torch.cuda.synchronize()
    tg, tr, tf, wall = CallTimer(torch), CallTimer(torch), CallTimer(torch), CallTimer(torch)
    before = _bytes_total(buf)
    for _ in range(steps):
        with wall:
            one_step(tg, tr, tf)
    parts = {"gather_ms": tg.total_ms() / steps, "reduce_scatter_ms": tr.total_ms() / steps,
             "finish_ms": tf.total_ms() / steps}
    if fused:
        parts["reduce_scatter_ms_note"] = "backward reduce-scatters with the next bucket's gather fused in"
    ms = _step_ms(parts, wall, steps, flush is not None)
    bench_stage3.parts = parts
    per_step = _bytes_delta(buf, before) / steps
    st = buf.status()
    buf.close()
    del gbuf, outs
    torch.cuda.empty_cache()
    return ms, per_step, st


def bench_stage2_buckets(w, bucket, steps, warmup, torch, S, Z):
    """ZeRO-2 reduced during backward: per step, every bucket (in reverse order)
    arrives in one constant-size buffer per rank and is reduce-scattered with
    the fused AdamW + all-gather; then the step is finished."""
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    buf = RankBuffers(w.psi, w.n_ranks, 2, w.dtype, double_buffer=True, alloc_grads=False)
    P, N = buf.psi_pad, w.n_ranks
    td = S.torch_dtype(w.dtype)
    mv, mm, vv = buf.state(0)
    S.draw_master(w, mv, w.psi)
    S.draw_moments(w, mm, vv, w.psi)
    buf.params[:, :P].copy_(mv.to(td).unsqueeze(0).expand(N, P))
    buckets = S.flat_buckets(P, N, bucket)
    lmax = max(b - a for a, b in buckets)
    cb = torch.empty((N, (lmax + 7) // 8 * 8), dtype=td, device="cuda")
    for r in range(N):
        S.draw_grads(w, cb[r], lmax, 1, r, w.loss_scale)
    buf.set_scaler(w.loss_scale, 0, 0)
    hyp = Z.hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm, Z.ZERO_MODE_AUTO)
    rows = [cb[r] for r in range(N)]

    def one_step(timer):
        for (a, b) in reversed(buckets):
            with timer:
                buf.reduce_scatter(a, b, rows, hyp)
        with timer:
            buf.finish_bucketed_step(hyp)

    for _ in range(warmup):
        one_step(CallTimer(torch))
    timer, wall = CallTimer(torch), CallTimer(torch)
    before = _bytes_total(buf)
    for _ in range(steps):
        with wall:
            one_step(timer)
    ms = _step_ms({"calls_ms": timer.total_ms() / steps}, wall, steps, False)
    per_step = _bytes_delta(buf, before) / steps
    st = buf.status()
    buf.close()
    del cb
    torch.cuda.empty_cache()
    return ms, per_step, st, len(buckets)


def bench_stage3_zeropp(w, buckets, steps, warmup, torch, S, Z, bits):
    """ZeRO-3 with the ZeRO++ exchanges: INT8 block-quantized parameter gathers
    (forward and backward) and a reduce-scatter of the ranks' INT8/INT4
    block-quantized gradients, then the step.  The ranks' gradient codes are
    produced once before timing (the producer-side quantization belongs to
    backward); its own time is measured separately on one bucket."""
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    buf = RankBuffers(w.psi, w.n_ranks, 3, w.dtype, double_buffer=True)
    P, N = buf.psi_pad, w.n_ranks
    td = S.torch_dtype(w.dtype)
    zdt = Z.ZERO_BF16 if w.dtype == "bf16" else Z.ZERO_FP16
    mv, mm, vv = buf.state(0)
    S.draw_master(w, mv, w.psi)
    S.draw_moments(w, mm, vv, w.psi)
    buf.params[:P].copy_(mv.to(td))
    lmax = max(b - a for a, b in buckets)
    lpad = (lmax + 7) // 8 * 8
    nb = (lmax + 255) // 256
    gbuf = torch.empty((N, lpad), dtype=td, device="cuda")
    for r in range(N):
        S.draw_grads(w, gbuf[r], lmax, 1, r, w.loss_scale)
    cbytes = (lpad if bits == 8 else lpad // 2 + 16)
    gcodes = torch.empty((N, (cbytes + 15) // 16 * 16), dtype=torch.uint8, device="cuda")
    gscales = torch.empty((N, 2 * nb + 2), dtype=torch.float32, device="cuda")
    qt = CallTimer(torch)
    for r in range(N):
        with qt:
            Z.zero_quantize_blocks(zdt, bits, gbuf[r], lmax, gcodes[r], gscales[r])
    quant_ms = qt.total_ms() / N
    ocodes = torch.empty((N, (lpad + 15) // 16 * 16), dtype=torch.uint8, device="cuda")
    oscales = torch.empty((N, 2 * nb + 2), dtype=torch.float32, device="cuda")
    buf.set_scaler(w.loss_scale, 0, 0)
    hyp = Z.hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm, Z.ZERO_MODE_AUTO)
    cr, sr = [gcodes[r] for r in range(N)], [gscales[r] for r in range(N)]
    ocr, osr = [ocodes[r] for r in range(N)], [oscales[r] for r in range(N)]

    def one_step(tg, tr, tf):
        for (a, b) in buckets:
            with tg:
                Z.zero_gather_bucket_q8(buf.h, a, b, buf.params, ocr, osr)
        for (a, b) in reversed(buckets):
            with tg:
                Z.zero_gather_bucket_q8(buf.h, a, b, buf.params, ocr, osr)
            with tr:
                Z.zero_reduce_scatter_bucket_q(buf.h, a, b, bits, cr, sr, buf.master, buf.m, buf.v,
                                               buf.params, hyp)
        with tf:
            buf.step(hyp)

    for _ in range(warmup):
        one_step(CallTimer(torch), CallTimer(torch), CallTimer(torch))
    tg, tr, tf, wall = CallTimer(torch), CallTimer(torch), CallTimer(torch), CallTimer(torch)
    before = _bytes_total(buf)
    for _ in range(steps):
        with wall:
            one_step(tg, tr, tf)
    parts = {"gather_ms": tg.total_ms() / steps, "reduce_scatter_ms": tr.total_ms() / steps,
             "finish_ms": tf.total_ms() / steps}
    ms = _step_ms(parts, wall, steps, False)
    per_step = _bytes_delta(buf, before) / steps
    st = buf.status()
    buf.close()
    del gbuf, gcodes, gscales, ocodes, oscales
    torch.cuda.empty_cache()
    return ms, per_step, st, quant_ms, lmax, parts


def bench_schedule(w, buckets, steps, warmup, torch, S, Z, prefetch, graph, fuse=True):
    """Whole ZeRO-3 steps through Zero3Schedule (gathers one bucket ahead on a
    side stream when `prefetch`; backward gathers carried by the reduce-scatters
    when `fuse`; the step replayed from a CUDA graph when `graph`), timed with
    events on the main stream around each step."""
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    from zero_partitioned_mixed_gb300.schedule import Zero3Schedule
    buf = RankBuffers(w.psi, w.n_ranks, 3, w.dtype, double_buffer=True)
    P, N = buf.psi_pad, w.n_ranks
    td = S.torch_dtype(w.dtype)
    mv, mm, vv = buf.state(0)
    S.draw_master(w, mv, w.psi)
    S.draw_moments(w, mm, vv, w.psi)
    buf.params[:P].copy_(mv.to(td))
    lmax = max(b - a for a, b in buckets)
    gbuf = torch.empty((N, (lmax + 7) // 8 * 8), dtype=td, device="cuda")
    for r in range(N):
        S.draw_grads(w, gbuf[r], lmax, 1, r, w.loss_scale)
    rows = Z.pointer_array([gbuf[r] for r in range(N)])
    buf.set_scaler(w.loss_scale, 0, 0)
    hyp = Z.hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm, Z.ZERO_MODE_AUTO)
    sched = Zero3Schedule(buf, buckets, prefetch=prefetch, fuse=fuse)
    grads = lambda i: rows
    for _ in range(warmup):
        sched.step(hyp, grads)
    g = sched.capture(hyp, grads) if graph else None
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        if g is not None:
            g.replay()
        else:
            sched.step(hyp, grads)
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    buf.close()
    del gbuf, sched, g
    torch.cuda.empty_cache()
    return ms


def bench_persist(shapes, name, threshold, steps, warmup, torch, S, Z, graph):
    """GPT-2-small ZeRO-3 steps with one bucket per tensor through
    Zero3Schedule (prefetch on), with tensors below `threshold` kept resident
    (param_persistence_threshold); eager or replayed from a CUDA graph.
    Returns (ms per step, algorithmic bytes per step from the library's
    counters, gathered buckets, all buckets, launches per step)."""
    from zero_partitioned_mixed_gb300.buffers import RankBuffers
    from zero_partitioned_mixed_gb300.persistence import persistent_layout, tensor_buckets
    from zero_partitioned_mixed_gb300.schedule import Zero3Schedule
    lay = persistent_layout(shapes, threshold)
    w = S.Workload(name, lay.psi, 8, 3, "bf16", 1, grad_sigma=1e-3)
    buf = RankBuffers(w.psi, w.n_ranks, 3, w.dtype, double_buffer=True)
    P, N = buf.psi_pad, w.n_ranks
    buckets = tensor_buckets(lay, P)
    td = S.torch_dtype(w.dtype)
    mv, mm, vv = buf.state(0)
    S.draw_master(w, mv, w.psi)
    S.draw_moments(w, mm, vv, w.psi)
    buf.params[:P].copy_(mv.to(td))
    lmax = max(b - a for a, b in buckets)
    gbuf = torch.empty((N, (lmax + 7) // 8 * 8), dtype=td, device="cuda")
    for r in range(N):
        S.draw_grads(w, gbuf[r], lmax, 1, r, w.loss_scale)
    rows = Z.pointer_array([gbuf[r] for r in range(N)])
    buf.set_scaler(w.loss_scale, 0, 0)
    hyp = Z.hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_norm, Z.ZERO_MODE_AUTO)
    sched = Zero3Schedule(buf, buckets, prefetch=True, persistent_from=lay.persistent_from(P))
    grads = lambda i: rows
    for _ in range(warmup):
        sched.step(hyp, grads)
    b0 = _bytes_total(buf)
    sched.step(hyp, grads)
    bps = _bytes_total(buf) - b0
    g = sched.capture(hyp, grads) if graph else None
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        if g is not None:
            g.replay()
        else:
            sched.step(hyp, grads)
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    ng = len(sched.gathered)
    # two gathers per gathered bucket, one reduce-scatter per bucket, finalise +
    # rollback, and the resident refresh
    launches = 2 * ng + len(buckets) + 2 + (1 if sched.resident is not None else 0)
    buf.close()
    del gbuf, sched, g
    torch.cuda.empty_cache()
    return ms, bps, ng, len(buckets), launches, lay


def run_other(args, ws, rank, local):
    import dataclasses

    import torch
    import zero_partitioned_mixed_gb300 as Z
    from zero_partitioned_mixed_gb300 import synth as S
    from zero_partitioned_mixed_gb300.build import build_library

    torch.cuda.set_device(local)
    build_library()
    lines = []
    if args.workload == "toy":
        base = S.TOY
        for stage in (0, 1, 2, 3):
            w = dataclasses.replace(base, stage=stage)
            if stage == 3:
                pp = S.flat_buckets(((w.psi + 255) // 256) * 256, w.n_ranks, 50_000)
                ms, bps, st = bench_stage3(w, pp, args.steps, args.warmup, torch, S, Z, flush_l2=True)
            else:
                ms, bps, st = bench_dense(w, stage, args.steps, args.warmup, torch, S, Z, flush_l2=True)
            lines.append(_line(f"{base.name}_stage{stage}", w.psi / (ms * 1e-3), ms, args.steps, args.warmup,
                               bps, w.dtype, {"stage": stage, "l2": "256 MiB written between timed calls",
                                              "note": "L2-resident size: latency-bound, not a roofline point"}))
    elif args.workload == "zero2-buckets":
        w = dataclasses.replace(S.FLAT15B, name="flat_psi1.5e9_n8_stage2_buckets5e7_fp16", stage=2,
                                inject_step=0)
        ms, bps, st, nb = bench_stage2_buckets(w, 50_000_000, args.steps, args.warmup, torch, S, Z)
        lines.append(_line(w.name, w.psi / (ms * 1e-3), ms, args.steps, args.warmup, bps, w.dtype,
                           {"stage": 2, "buckets": nb, "mode": "speculative, fused per bucket, one "
                            "constant-size gradient buffer per rank", "l2": "inputs larger than L2"}))
    elif args.workload == "llama7b-zeropp":
        w = S.LLAMA7B
        buckets = S.layer_buckets(S.llama7b_shapes(), w.psi)
        for bits in (8, 4):
            ms, bps, st, qms, lmax, parts = bench_stage3_zeropp(w, buckets, args.steps, args.warmup, torch, S, Z,
                                                                bits)
            lines.append(_line(f"{w.name}_zeropp_int8gather_int{bits}rs", w.psi / (ms * 1e-3), ms, args.steps,
                               args.warmup, bps, w.dtype,
                               {"stage": 3, "buckets": len(buckets), "gather": "int8 blocks of 256 (qwZ)",
                                "reduce_scatter": f"int{bits} blocks of 256 (qgZ)",
                                "producer_quantize_ms_per_rank_per_layer": qms, "layer_elems": lmax,
                                "l2": "inputs larger than L2", **parts}))
    elif args.workload in ("flat-zero3", "flat-zeropp"):
        psi = args.psi or (1 << 25)
        n = args.n_ranks or 8
        w = S.Workload(f"flat_psi{psi}_n{n}_stage3_bf16", psi, n, 3, "bf16", 1, grad_sigma=1e-3)
        pp = ((psi + n * 8 - 1) // (n * 8)) * (n * 8)
        buckets = S.flat_buckets(pp, n, args.bucket or max(64, psi // 4))
        if args.workload == "flat-zero3" and args.prefetch:
            # whole steps through Zero3Schedule: each gather one bucket ahead on a side stream
            ms = bench_schedule(w, buckets, args.steps, args.warmup, torch, S, Z, True, False)
            bps = (6 * n + 30) * pp
            parts = {"schedule": "Zero3Schedule, gathers one bucket ahead on a side stream"}
        elif args.workload == "flat-zero3":
            ms, bps, st = bench_stage3(w, buckets, args.steps, args.warmup, torch, S, Z, fused=not args.separate)
            parts = dict(bench_stage3.parts, fused=not args.separate)
        else:
            ms, bps, st, _, _, parts = bench_stage3_zeropp(w, buckets, args.steps, args.warmup, torch, S, Z,
                                                           args.rs_bits)
        extra = {"stage": 3, "buckets": len(buckets), **parts}
        if args.workload == "flat-zeropp":
            extra.update({"gather": "int8 blocks of 256", "reduce_scatter": f"int{args.rs_bits} blocks of 256"})
        lines.append(_line(w.name + (f"_zeropp_int{args.rs_bits}rs" if args.workload == "flat-zeropp" else ""),
                           psi / (ms * 1e-3), ms, args.steps, args.warmup, bps, "bf16", extra))
    elif args.workload == "schedule":
        # ZeRO-3 step scheduling: sequential vs one-ahead prefetch on a side
        # stream (Llama-7B), and eager vs CUDA-graph replay (toy buffer, launch-bound)
        w = S.LLAMA7B
        buckets = S.layer_buckets(S.llama7b_shapes(), w.psi)
        for prefetch, fuse in ((False, False), (True, False), (False, True), (True, True)):
            ms = bench_schedule(w, buckets, args.steps, args.warmup, torch, S, Z, prefetch, False, fuse)
            lines.append(_line(f"{w.name}_{'prefetch' if prefetch else 'sequential'}{'_fused' if fuse else ''}",
                               w.psi / (ms * 1e-3), ms, args.steps, args.warmup, (6 * 8 + 30) * w.psi, w.dtype,
                               {"stage": 3, "buckets": len(buckets), "prefetch": prefetch,
                                "fused_backward_gathers": fuse}))
        toy = dataclasses.replace(S.TOY, stage=3)
        tb = S.flat_buckets(637_952, 32, 50_000)
        for graph in (False, True):
            ms = bench_schedule(toy, tb, max(args.steps, 20), args.warmup, torch, S, Z, True, graph)
            lines.append(_line(f"{toy.name}_stage3_{'graph' if graph else 'eager'}", toy.psi / (ms * 1e-3), ms,
                               max(args.steps, 20), args.warmup, (6 * 32 + 30) * 637_952, toy.dtype,
                               {"stage": 3, "buckets": len(tb), "cuda_graph": graph,
                                "l2": "L2-resident, back-to-back replays"}))
    elif args.workload == "gpt2-zero3-persist":
        # ZeRO-3 with one bucket per tensor: every tensor gathered (threshold 0)
        # against the guide's param_persistence_threshold of 1e5 (biases and
        # layer norms resident), eager and graph-replayed
        shapes = S.gpt2_small_shapes()
        for thr in (0, 100_000):
            for graph in (False, True):
                name = f"gpt2_small_zero3_n8_tensor_buckets_persist{thr}"
                ms, bps, ng, nb, launches, lay = bench_persist(shapes, name, thr, args.steps, args.warmup,
                                                               torch, S, Z, graph)
                lines.append(_line(f"{name}_{'graph' if graph else 'eager'}", lay.psi / (ms * 1e-3), ms,
                                   args.steps, args.warmup, bps, "bf16",
                                   {"stage": 3, "param_persistence_threshold": thr, "buckets": nb,
                                    "gathered_buckets": ng, "persistent_tensors": lay.n_persistent,
                                    "persistent_elems": lay.psi_persistent, "cuda_graph": graph,
                                    "launches_per_step": launches, "prefetch": True,
                                    "l2": "inputs larger than L2"}))
    elif args.workload == "gpt2":
        w = S.GPT2
        ms, bps, st = bench_dense(w, 2, args.steps, args.warmup, torch, S, Z)
        lines.append(_line(w.name, w.psi / (ms * 1e-3), ms, args.steps, args.warmup, bps, w.dtype,
                           {"stage": 2, "mode": "speculative one pass; a step whose norm exceeds 1.0 is redone",
                            "l2": "inputs larger than L2"}))
        ms, bps, st = bench_dense(w, 2, args.steps, args.warmup, torch, S, Z, mode=Z.ZERO_MODE_TWO_PASS_WS)
        lines.append(_line(w.name + "_two_pass", w.psi / (ms * 1e-3), ms, args.steps, args.warmup, bps, w.dtype,
                           {"stage": 2, "mode": "two-pass: fp32 g_hat to the workspace, clip decided before the update",
                            "l2": "inputs larger than L2"}))
    elif args.workload == "llama7b":
        w = S.LLAMA7B
        buckets = S.layer_buckets(S.llama7b_shapes(), w.psi)
        ms, bps, st = bench_stage3(w, buckets, args.steps, args.warmup, torch, S, Z, fused=not args.separate)
        lines.append(_line(w.name, w.psi / (ms * 1e-3), ms, args.steps, args.warmup, bps, w.dtype,
                           {"stage": 3, "buckets": len(buckets), "mode": "speculative, fused per bucket",
                            "l2": "inputs larger than L2", "fused_backward_gathers": not args.separate,
                            **bench_stage3.parts}))
    elif args.workload == "sweep":
        stages = [int(x) for x in args.stages.split(",")]
        for psi, n in S.sweep_points():
            if (args.psi and psi != args.psi) or (args.n_ranks and n != args.n_ranks):
                continue
            for stage in stages:
                w = S.Workload(f"sweep_psi{psi}_n{n}_stage{stage}", psi, n, stage, "bf16", 1, grad_sigma=1e-3)
                flush = psi * (4 * n + 24) < (512 << 20)
                if stage == 3:
                    pp = ((psi + n * 8 - 1) // (n * 8)) * (n * 8)
                    ms, bps, st = bench_stage3(w, S.flat_buckets(pp, n, 50_000_000), args.steps, args.warmup,
                                               torch, S, Z, flush_l2=flush, fused=not args.separate)
                else:
                    mode = Z.ZERO_MODE_SPECULATIVE_STAGED if args.mode == "staged" else None
                    ms, bps, st = bench_dense(w, stage, args.steps, args.warmup, torch, S, Z, flush_l2=flush,
                                              sets_max=1, mode=mode)
                extra = {"psi": psi, "n_ranks": n, "stage": stage,
                         "l2": "256 MiB written between timed calls" if flush else "inputs larger than L2"}
                if stage == 3:
                    extra.update(bench_stage3.parts)
                lines.append(_line(w.name, psi / (ms * 1e-3), ms, args.steps, args.warmup, bps, "bf16", extra))
                print(json.dumps(lines[-1]), flush=True)
        return 0
    for ln in lines:
        print(json.dumps(ln), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["flat1.5b", "toy", "gpt2", "llama7b", "sweep", "zero2-buckets", "llama7b-zeropp",
                                      "flat-zero3", "flat-zeropp", "schedule", "gpt2-zero3-persist"],
                    default="flat1.5b")
    ap.add_argument("--mode", choices=["auto", "staged"], default="auto",
                    help="flat workload and the sweep's stages 1/2: the step kernel (staged = inputs through "
                         "shared memory by bulk copies)")
    ap.add_argument("--rs-bits", type=int, choices=[8, 4], default=8,
                    help="flat-zeropp: code width of the quantized gradient reduce-scatter")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--psi", type=int, default=None,
                    help="override psi of the flat workloads (profiling); sweep: run only this psi")
    ap.add_argument("--n-ranks", type=int, default=None,
                    help="flat-zero3 / flat-zeropp: simulated ranks (default 8); sweep: run only this N")
    ap.add_argument("--bucket", type=int, default=None,
                    help="flat-zero3 / flat-zeropp: elements per bucket (default psi / 4)")
    ap.add_argument("--stages", default="1,2,3", help="sweep: stages to run")
    ap.add_argument("--prefetch", action="store_true",
                    help="flat-zero3: run whole steps through the ZeRO-3 schedule with side-stream prefetch")
    ap.add_argument("--separate", action="store_true",
                    help="stage-3 workloads (flat-zero3, llama7b, sweep): backward gathers as calls of their own "
                         "(default: each backward reduce-scatter carries the next bucket's gather)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    if args.workload != "flat1.5b":
        return run_other(args, ws, rank, local)
    return run_ours(args, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
