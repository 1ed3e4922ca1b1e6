"""Benchmark of the single-pass flash-attention backward on GB300.

One step = the whole hot path on one batch: fa_bwd_preprocess (D and the
zeroed dQ accumulator) -> fa_bwd (the tcgen05 kernel) -> fa_bwd_dq_finalize.
Default workload: B=4, H=16, s1=s2=4096, head_dim=128, non-causal, the
shape the throughput target is stated on.  FLOPs per step = 10*s1*s2*d*H*B
(halved when causal).  Inputs are synthetic (seeded N(0,1) bf16); O, m, l
come from the library's forward-statistics kernel before timing.

  python bench.py [--gpus N --steps K --warmup W] [--workload cfg3nc|cfg2|...]
  python bench.py --impl reference     # the fp64 CPU oracle on the same workload

Variant workloads (--workload gqa|swa|br) exercise grouped-query attention,
the causal sliding window and the bottom-right causal alignment; their FLOPs
count 10*d per visible (query, key) pair.  --stats lse feeds the backward
the single statistic lse = m + ln l instead of (m, l).

Under torchrun every rank runs its own copy of the workload (the path
shards over independent (sequence, head) units with no collective: weak
scaling); rank 0 prints one JSON line with the max time over ranks.
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
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "FA-backward TFLOP/s (bf16, device-timed) and % of GB300 dense BF16 peak"
L2_BYTES = 129 * 1024 * 1024


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(values, pg=None, device=None):
    """Element-wise max of a list of floats over all ranks (timing only; the
    data path has no collective)."""
    if pg is None:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


COMMON_SOURCES = ("sm103.cuh", "api.cu", "internal.h")


def kernel_sources(head_dim: int, dq_mode: int):
    """The sources that decide what fa_bwd launches for this head_dim and
    dQ mode: the kernels, their PTX wrappers, the grid set-up and launch
    order."""
    if head_dim == 256:
        return ("bwd_d256.cu",) + COMMON_SOURCES
    return ("bwd_main.cu",) + (("dq_main.cu",) if dq_mode else ()) + COMMON_SOURCES


def kernel_source_hash(head_dim: int = 128, dq_mode: int = 0):
    h = hashlib.sha256()
    for f in kernel_sources(head_dim, dq_mode):
        with open(os.path.join(ROOT, "attention_backward_sm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, head_dim: int, dq_mode: int):
    """DRAM bytes per fa_bwd call (all its kernels) from the committed ncu
    summary of this workload and dQ mode, if it was taken on the current
    sources; otherwise None."""
    name = f"fa_bwd_det_{workload}.md" if dq_mode else f"fa_bwd_{workload}.md"
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    mh = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    mt = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not mh or not mt or mh.group(1) != kernel_source_hash(head_dim, dq_mode):
        return None
    return float(mt.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed
    region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        # raw samples: $FA_CLOCKS_DIR if set, else the system temporary directory
        out_dir = os.environ.get("FA_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_gpu{gpu_index}.csv")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_index)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower() in ("active", "0x1", "1"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


WORKLOADS = {**si.CONFIGS, **si.VARIANTS}


def make_case(name: str) -> si.Case:
    return WORKLOADS[name]()


def visible_pairs(s1: int, s2: int, causal: bool, window: int = 0, bottom_right: bool = False,
                  rows: int | None = None) -> int:
    """Number of (query, key) pairs the mask admits among the first `rows`
    queries: query i sees keys max(0, i+off-W+1) .. min(s2-1, i+off)
    (causal; off = s2 - s1 bottom-right, else 0; W = window > 0)."""
    n = s1 if rows is None else min(rows, s1)
    if not causal:
        return n * s2
    i = np.arange(n, dtype=np.int64)
    off = s2 - s1 if bottom_right else 0
    hi = np.minimum(s2 - 1, i + off)
    lo = np.maximum(0, i + off - window + 1) if window > 0 else np.zeros_like(i)
    return int(np.maximum(0, hi - lo + 1).sum())


def useful_flops(case: si.Case) -> float:
    """FLOPs of one backward: 10*s1*s2*d per (sequence, query head), halved
    under the plain causal mask (the counting rule of the target metric);
    for a sliding window or the bottom-right alignment, 10*d per visible
    (query, key) pair, the same rule counted exactly."""
    if case.window == 0 and not case.bottom_right:
        return case.flops()
    pairs = sum(visible_pairs(a, b, case.causal, case.window, case.bottom_right)
                for a, b in zip(case.q_lens, case.kv_lens))
    return 10.0 * pairs * case.head_dim * case.heads


_TENSORS = {}


def case_tensors(case: si.Case):
    """CPU inputs of a case, generated once per process."""
    if case.name not in _TENSORS:
        _TENSORS[case.name] = case.tensors()
    return _TENSORS[case.name]


def workload_desc(case: si.Case) -> str:
    mask = "non-causal"
    if case.causal:
        mask = "causal bottom-right" if case.bottom_right else "causal"
        if case.window:
            mask += f" window={case.window}"
    heads = f"H={case.heads}" + (f" Hkv={case.kv_heads}" if case.kv_heads != case.heads else "")
    if len(set(case.q_lens)) == 1 and len(set(case.kv_lens)) == 1:
        return (f"B={case.batch} {heads} s1={case.q_lens[0]} s2={case.kv_lens[0]} d={case.head_dim} {mask}")
    return (f"varlen B={case.batch} {heads} d={case.head_dim} q_lens={case.q_lens} "
            f"kv_lens={case.kv_lens} {mask}")


def mask_kw(case: si.Case) -> dict:
    return dict(window=case.window, bottom_right=case.bottom_right)


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(case: si.Case, budget_s: float, max_units: int | None = None):
    """Times the fp64 oracle backward on whole (sequence, head) units of the
    workload until about budget_s seconds of CPU work.  Returns
    (flops, seconds, units)."""
    import oracle
    q, k, v, do = case_tensors(case)
    flops, secs, units = 0.0, 0.0, 0
    order = [(b, h) for b in range(case.batch) for h in range(case.heads)]
    G = case.heads // case.kv_heads
    for b, h in order:
        qs, qe = int(case.cu_q[b]), int(case.cu_q[b + 1])
        ks, ke = int(case.cu_kv[b]), int(case.cu_kv[b + 1])
        qq, kk, vv, dd = q[qs:qe, h], k[ks:ke, h // G], v[ks:ke, h // G], do[qs:qe, h]
        o, m, l = oracle.forward_head(qq, kk, vv, case.softmax_scale, case.causal, **mask_kw(case))   # untimed
        t0 = time.perf_counter()
        oracle.backward_head(qq, kk, vv, o, dd, m, l, case.softmax_scale, case.causal, **mask_kw(case))
        secs += time.perf_counter() - t0
        if case.window == 0 and not case.bottom_right:
            f = 10.0 * (qe - qs) * (ke - ks) * case.head_dim
            flops += f / 2 if case.causal else f
        else:
            flops += 10.0 * case.head_dim * visible_pairs(qe - qs, ke - ks, True, case.window, case.bottom_right)
        units += 1
        if secs >= budget_s or (max_units and units >= max_units):
            break
    return flops, secs, units


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def blas_threads():
    """Threads numpy's BLAS uses in this process: threadpoolctl when it is
    installed, else the OpenBLAS library numpy loaded, asked directly."""
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    import ctypes
    paths = set()
    try:
        for line in open("/proc/self/maps"):
            parts = line.split()
            if len(parts) >= 6 and "openblas" in parts[-1].lower():
                paths.add(parts[-1])
    except OSError:
        return None
    for path in sorted(paths):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads",
                    "openblas_get_num_threads64_", "openblas_get_num_threads"):
            fn = getattr(lib, sym, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn())
    return None


def single_thread_probe():
    """Runs in a child process whose BLAS is limited to one thread: the
    fp64 oracle backward on cfg1 (whole) and on whole units of cfg2 for up
    to ~5 s.  Prints one JSON object."""
    out = {"blas_threads": blas_threads()}
    for name, budget in (("cfg1", 5.0), ("cfg2", 5.0)):
        f, s, u = oracle_sample(make_case(name), budget)
        out[name] = {"value": f / s / 1e12, "unit": "TFLOP/s", "units": u, "flop": f, "seconds": s}
    print(json.dumps(out), flush=True)


def single_thread_baseline():
    """Oracle times at one BLAS thread on cfg1 and cfg2 (a child process, so
    that this process keeps its full thread count)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--single-thread-probe"], env=env,
                           capture_output=True, text=True, timeout=120)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal: this is a context number
        return {"error": f"{type(e).__name__}: {e}"}


def oracle_rows(case: si.Case, rows: int, b: int = 0, h: int = 0):
    """Times the fp64 oracle backward of the first `rows` query rows of one
    (sequence, head) unit against all of its keys: dQ of those rows and
    their share of dK and dV.  Returns (flops, seconds)."""
    import oracle
    q, k, v, do = case_tensors(case)
    qs = int(case.cu_q[b])
    ks, ke = int(case.cu_kv[b]), int(case.cu_kv[b + 1])
    s1, s2 = int(case.cu_q[b + 1]) - qs, ke - ks
    rows = max(1, min(rows, s1))
    hk = h // (case.heads // case.kv_heads)
    if case.bottom_right:
        # keys past what the first `rows` queries can see are dropped; the
        # kept s2' = s2 - s1 + rows keys give the same bottom-right offset
        ke = ks + max(0, min(s2, s2 - s1 + rows))
    qq, kk, vv, dd = q[qs:qs + rows, h], k[ks:ke, hk], v[ks:ke, hk], do[qs:qs + rows, h]
    o, m, l = oracle.forward_head(qq, kk, vv, case.softmax_scale, case.causal, **mask_kw(case))   # untimed
    t0 = time.perf_counter()
    oracle.backward_head(qq, kk, vv, o, dd, m, l, case.softmax_scale, case.causal, **mask_kw(case))
    secs = time.perf_counter() - t0
    pairs = visible_pairs(s1, s2, case.causal, case.window, case.bottom_right, rows)
    return 10.0 * pairs * case.head_dim, secs


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    case = make_case(args.workload)
    # Size each step's sample so that warm-up plus timed steps stay near
    # three minutes of CPU time: calibrate on 256 query rows first.
    f0, s0 = oracle_rows(case, 256)
    rate = f0 / max(s0, 1e-9)
    per_step_s = min(20.0, 180.0 / max(1, args.steps + args.warmup))
    unit_pairs = case.q_lens[0] * case.kv_lens[0]
    rows = int(max(64, min(case.q_lens[0], per_step_s * rate / (10.0 * case.head_dim * case.kv_lens[0]))))
    for _ in range(args.warmup):
        oracle_rows(case, rows)
    total_f, total_s = 0.0, 0.0
    for _ in range(args.steps):
        f, s = oracle_rows(case, rows)
        total_f += f
        total_s += s
    value = total_f / total_s / 1e12
    sample = (f"fp64 backward of query rows [0, {rows}) of (sequence 0, head 0) against all "
              f"{case.kv_lens[0]} keys per step ({total_f / args.steps:.3e} FLOP; a full unit has "
              f"{unit_pairs} score entries)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {workload_desc(case)}", "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample, "blas_threads": blas_threads()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def run_gpu(args):
    import attention_backward_sm_gb300 as fab
    from attention_backward_sm_gb300 import build as fab_build

    rank, world, local = dist_env()
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        fab_build.build()
    if pg is not None:
        pg.barrier()
    fab.lib()

    case = make_case(args.workload)
    cu_q_host, cu_kv_host = case.cu_q, case.cu_kv      # host offsets, computed once
    q, k, v, do = (t.to(dev) for t in case_tensors(case))
    cu_q = torch.from_numpy(case.cu_q).to(dev)
    cu_kv = torch.from_numpy(case.cu_kv).to(dev)
    scale = case.softmax_scale
    mask = fab.mask_kind(case.causal, case.bottom_right)
    lse_stats = args.stats == "lse"
    if lse_stats:
        o, lse = fab.forward_lse(q, k, v, cu_q, cu_kv, cu_q_host, cu_kv_host, case.causal, scale, **mask_kw(case))
        stats = (lse,)
    else:
        o, m, l = fab.forward_stats(q, k, v, cu_q, cu_kv, cu_q_host, cu_kv_host, case.causal, scale, **mask_kw(case))
        stats = (m, l)
    work = fab.Workspace(q, cu_q_host, cu_kv_host, case.causal, args.dq_mode)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream(dev)
    flops = useful_flops(case)
    launches_per_step = 3 + (1 if args.dq_mode == 1 else 0) + (2 if case.total_kv > int(case.cu_kv[-1]) else 0)
    input_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, do, o, *stats, work.dq_acc))

    def bwd():
        if lse_stats:
            fab.fa_bwd_lse(q, k, v, do, stats[0], work.D, work.dq_acc, dk, dv, cu_q, cu_kv, cu_q_host, cu_kv_host,
                           mask, case.window, scale, args.dq_mode, work.ws)
        else:
            fab.fa_bwd_ex(q, k, v, do, *stats, work.D, work.dq_acc, dk, dv, cu_q, cu_kv, cu_q_host, cu_kv_host,
                          mask, case.window, scale, args.dq_mode, work.ws)

    def step(ev=None):
        fab.fa_bwd_preprocess(o, do, work.D, work.dq_acc)
        if ev is not None:
            ev[0].record(stream)
        bwd()
        if ev is not None:
            ev[1].record(stream)
        fab.fa_bwd_dq_finalize(work.dq_acc, dq, scale)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    fab.fa_check_device_status()

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    # Inputs that fit in L2 would stay cached from one step to the next: every
    # timed step is then preceded by writing a buffer four times the L2, and
    # timed by its own events.  While that write runs the host enqueues the
    # whole step, so no host-side gap falls inside the timed interval.
    # Otherwise events at every step boundary time the steps back to back.
    small = input_bytes <= L2_BYTES
    flush = torch.empty(4 * L2_BYTES, dtype=torch.uint8, device=dev) if small else None
    step_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)] if small else None
    bounds = None if small else [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize(dev)
    if not small:
        bounds[0].record(stream)
    for i in range(args.steps):
        if small:
            flush.zero_()
            step_evs[i][0].record(stream)
        step(evs[i])
        if small:
            step_evs[i][1].record(stream)
        else:
            bounds[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    if pg is not None:
        pg.barrier()
    clk = clocks.stop() if clocks else None
    fab.fa_check_device_status()
    if small:
        step_ms = [a.elapsed_time(b) for a, b in step_evs]
    else:
        step_ms = [bounds[i].elapsed_time(bounds[i + 1]) for i in range(args.steps)]
    step_bwd_ms = [a.elapsed_time(b) for a, b in evs]
    med_ms, mean_ms = statistics.median(step_ms), statistics.mean(step_ms)
    med_ms, mean_ms = max_over_ranks([med_ms, mean_ms], pg, dev)
    ms_per_step = med_ms
    value = world * flops / (med_ms * 1e-3) / 1e12

    # Roofline leg: fa_bwd alone.  Small inputs: the L2-flushed steps above.
    # Otherwise a back-to-back loop of fa_bwd launches lasting at least half
    # a second, each launch timed by its own events, with its own clock
    # samples (a step loop of a few tens of milliseconds is too short for
    # the nvidia-smi sampler).
    if small:
        bwd_times, roof_clk = step_bwd_ms, clk
    else:
        n_roof = max(20, int(0.5 / max(statistics.median(step_bwd_ms) * 1e-3, 1e-6)) + 1)
        roof_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(n_roof)]
        roof_clocks = ClockSampler(local) if rank == 0 else None
        time.sleep(0.3 if roof_clocks else 0)
        torch.cuda.synchronize(dev)
        for ea, eb in roof_evs:
            ea.record(stream)
            bwd()
            eb.record(stream)
        torch.cuda.synchronize(dev)
        roof_clk = roof_clocks.stop() if roof_clocks else None
        fab.fa_check_device_status()
        bwd_times = [ea.elapsed_time(eb) for ea, eb in roof_evs]
    bwd_ms, bwd_mean_ms = statistics.median(bwd_times), statistics.mean(bwd_times)
    bwd_ms, bwd_mean_ms = max_over_ranks([bwd_ms, bwd_mean_ms], pg, dev)

    # End to end through the public API from pinned host buffers.  Every step
    # copies all of its inputs host -> device, runs the backward and copies
    # dQ, dK, dV device -> host.  The copies run on their own streams with
    # two sets of device buffers, as a training loop would run them: step
    # i+1's inputs arrive and step i-1's gradients leave while step i
    # computes.  The timed region spans the first input copy to the last
    # output copy.
    e2e = None
    if not args.no_e2e:
        host_in = [t.cpu().pin_memory() for t in (q, k, v, o, do, *stats)]
        host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)] for _ in range(2)]
        dev_in = [[torch.empty_like(t) for t in (q, k, v, o, do, *stats)] for _ in range(2)]
        dev_out = [(torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out[0])
        n_e2e = max(3, min(args.steps, 20))
        # (several input copy streams were measured no faster than one: the
        # host link, not a copy engine, is the limit)
        n_in = 1
        s_ins = [torch.cuda.Stream(dev) for _ in range(n_in)]
        s_in, s_out = s_ins[0], torch.cuda.Stream(dev)
        s_comp = stream
        ev = lambda: torch.cuda.Event()
        in_ready = [[ev() for _ in range(n_in)], [ev() for _ in range(n_in)]]
        comp_done = [ev(), ev()]
        out_done = [ev(), ev()]
        api = fab.backward_lse if lse_stats else fab.backward

        def run_steps(n):
            for i in range(n):
                b = i & 1
                for j, sj in enumerate(s_ins):
                    with torch.cuda.stream(sj):
                        if i >= 2:
                            sj.wait_event(comp_done[b])        # step i-2 has finished reading dev_in[b]
                        for d_, h_ in list(zip(dev_in[b], host_in))[j::n_in]:
                            d_.copy_(h_, non_blocking=True)
                        in_ready[b][j].record(sj)
                for e_ in in_ready[b]:
                    s_comp.wait_event(e_)
                if i >= 2:
                    s_comp.wait_event(out_done[b])             # step i-2's gradients have left dev_out[b]
                outs = api(*dev_in[b], cu_q, cu_kv, cu_q_host, cu_kv_host, case.causal, scale, args.dq_mode,
                           out=dev_out[b], work=work, stream=s_comp, check=False, **mask_kw(case))
                comp_done[b].record(s_comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[b])
                    for h_, d_ in zip(host_out[b], outs):
                        h_.copy_(d_, non_blocking=True)
                    out_done[b].record(s_out)

        run_steps(2)
        torch.cuda.synchronize(dev)
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(s_in)
        run_steps(n_e2e)
        for sj in s_ins[1:] + [s_out, s_comp]:
            s_in.wait_stream(sj)
        e2.record(s_in)
        torch.cuda.synchronize(dev)
        fab.fa_check_device_status()
        e2e_ms = s2.elapsed_time(e2) / n_e2e
        e2e_ms = max_over_ranks([e2e_ms], pg, dev)[0]
        e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "copies": "overlapped with compute on separate streams (two sets of device buffers)"}

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return

    peak, hbm, peak_src = peaks()
    achieved = flops / (bwd_ms * 1e-3) / 1e12
    traffic = None if lse_stats else profiled_traffic(args.workload, case.head_dim, args.dq_mode)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "hbm_gbs": None if traffic is None else traffic / (bwd_ms * 1e-3) / 1e9,
                "hbm_frac": None if traffic is None else traffic / (bwd_ms * 1e-3) / 1e9 / hbm,
                "kernel": ("fa_bwd (bwd256_kernel)" if case.head_dim == 256 else
                           "fa_bwd (bwd_kernel<%d> + dq_kernel<%d>)" % (case.head_dim, case.head_dim)
                           if args.dq_mode else "fa_bwd (bwd_kernel<%d>)" % case.head_dim),
                "fa_bwd_ms": bwd_ms, "fa_bwd_ms_mean": bwd_mean_ms, "launches_timed": len(bwd_times),
                "timing": "median of per-launch CUDA events on the launching stream; " +
                ("the L2-flushed steps" if small else
                 f"{len(bwd_times)} back-to-back launches ({sum(bwd_times) / 1e3:.2f} s)"),
                "clocks": roof_clk,
                "peak_source": f"bf16_tflops (burst) of {peak_src}; hbm_gbs of {peak_src}"}

    cpu = None
    if not args.no_cpu_baseline:
        f, s, u = oracle_sample(case, args.cpu_budget)
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "blas_threads": blas_threads(),
               "sample": f"fp64 backward of {u} (sequence, head) unit(s) of the workload, {f:.3e} FLOP in {s:.2f} s",
               "single_thread": single_thread_baseline()}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "ms_per_step_mean": mean_ms,
        "value_mean": world * flops / (mean_ms * 1e-3) / 1e12, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {workload_desc(case)}", "dq_mode": args.dq_mode,
                   "statistics": "lse" if lse_stats else "m, l",
                   "l2": f"inputs larger than L2 ({input_bytes / 2**20:.0f} MiB resident per step)"
                   if input_bytes > L2_BYTES else
                   f"L2 flushed before every timed step ({4 * L2_BYTES / 2**20:.0f} MiB written; inputs "
                   f"{input_bytes / 2**20:.0f} MiB)",
                   "flops_per_step": flops},
        "frac_of_peak_step": value / world / peak,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="cfg3nc", choices=sorted(WORKLOADS))
    ap.add_argument("--stats", choices=["ml", "lse"], default="ml",
                    help="softmax statistics the backward consumes: (m, l) or lse = m + ln l")
    ap.add_argument("--dq-mode", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--single-thread-probe", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.single_thread_probe:
        single_thread_probe()
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
