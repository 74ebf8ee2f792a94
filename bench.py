#!/usr/bin/env python
"""Benchmark of the decode-step KV path on GB300.

One step = one decode step of a 4-layer IndexShare group for B requests:
top-k over the indexer scores, one shared plan, and per layer a gather of the
k selected latent rows (pool hits from HBM, misses read in place from pinned
host memory) plus sparse MLA decode attention, with the pool refill on a side
stream. Metric: selected KV rows per second (B x layers x k rows per step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on host cores

Prints one JSON line (rank 0). Multi-GPU (torchrun): every rank serves its own
B requests (weak scaling, no data-path collective); value = rows of all ranks
/ max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workload as wl  # noqa: E402

METRIC = "selected KV rows/s per decode step (plan+gather+SFA); % of HBM/link roofline"
UNIT = "rows/s"
KERNELS = ("topk", "plan", "gather", "sfa", "refill")
# our kernels per step: top-k (1: one cluster per request, or 2: histogram + select)
# + plan 1 + gather 1 (every layer) + layers x (sfa 1 or 2 + refill 1; the
# reuse policy has no refill)
LAUNCHES_PLAN, LAUNCHES_GATHER = 1, 1


def topk_launches(w) -> int:
    """One cluster launch up to 262,144 positions (up to 8 CTAs a request),
    else histogram, select and output launches."""
    return 1 if w.ctx <= 262144 else 3


def sfa_launches(w) -> int:
    """The chunk kernel and the merge kernel of a layer's attention."""
    return 2


# after each layer's attention a one-thread kernel writes the layer's words
LAUNCHES_POST = 1


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--workload", default="large_batch", choices=sorted(wl.BY_NAME))
    ap.add_argument("--settle-steps", type=int, default=64,
                    help="most untimed steps before the warm-up, run in chunks of 16 until "
                         "two chunks agree (0: none, for profiler runs)")
    ap.add_argument("--query-slots", type=int, default=4,
                    help="distinct query tensors, cycled (queries do not change the work)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--e2e-settle-steps", type=int, default=16)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=6.0,
                    help="CPU seconds of oracle work per leg of the CPU baseline")
    ap.add_argument("--only", choices=KERNELS, default=None,
                    help="after the warm-up steps, launch only this kernel --steps times "
                         "(on the state the warm-up left) and report its time per launch")
    ap.add_argument("--B", type=int, default=None, help="override the workload's request count")
    ap.add_argument("--sets", type=int, default=None,
                    help="override the pool's sets (16 ways each): 512 = 8K entries, 1024 = 16K")
    ap.add_argument("--policy", choices=("fifo", "lru", "reuse"), default="fifo",
                    help="device pool: the set-associative FIFO pool (default), a fully "
                         "associative LRU pool of the same size, or the base design's "
                         "adjacent-step reuse of the previous selection")
    ap.add_argument("--layout", choices=("staged", "selection"), default="staged",
                    help="staged: the attention reads its rows straight from the pool (only "
                         "the misses are staged in HBM); selection: every row is gathered "
                         "into a selection buffer first")
    ap.add_argument("--layer-waits", action="store_true",
                    help="staged layout: each layer's attention waits for the whole layer's "
                         "rows (default: streamed, each attention CTA waits for its own "
                         "request's rows while the gather runs)")
    ap.add_argument("--mtp", type=int, default=0, choices=(0, 1, 2, 3),
                    help="MTP draft steps whose queries are folded into the heads "
                         "(the step attends (1 + N) x H query rows over one selection)")
    ap.add_argument("--profile-steps", type=int, default=10,
                    help="steps after the timed region with every launch's timing events "
                         "(the per-kernel figures other than the gather's)")
    ap.add_argument("--no-kernel-events", action="store_true",
                    help="time the steps without per-kernel events (no per-kernel roofline)")
    ap.add_argument("--oracle-worker", default=None, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over ranks (timing only; not on the data path)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def first_request(rank: int, w: wl.Workload) -> int:
    """Rank r serves requests r*B .. r*B+B-1 of the workload's request stream."""
    return rank * w.B


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((ts, float(f[1]), float(f[2]), f))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1] or \
            sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for i, n in enumerate(names):
                if r[3][5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": sorted(reasons),
                "samples": len(inside)}


# ---------------------------------------------------------------------------
# peaks
# ---------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def link_peak_gbs(torch, buf, reps=5):
    """Host-to-device bandwidth of the machine's host link: DMA copy of pinned
    (registered) host memory `buf` (a PinnedHost; best of `reps`, CUDA
    events)."""
    buf.array[:] = 1
    src = buf.tensor()
    nbytes = buf.array.nbytes
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    del src, dst
    return best


def settle(torch, g, step, max_steps, chunk=16, tol=0.03):
    """Run untimed steps in chunks until the step time is steady: on this
    platform, zero-copy reads of host memory run slow for a while after host
    memory is registered, copied by DMA or first touched. Stops when two
    consecutive chunks agree within `tol` and are within `tol` of the fastest
    chunk seen, or before more than `max_steps` steps; returns the steps run.
    `step()` takes the next step of the forward input stream."""
    times, n = [], 0
    while n + chunk <= max_steps:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(g.main)
        for _ in range(chunk):
            step()
        n += chunk
        g.join(g.main)
        b.record(g.main)
        b.synchronize()
        times.append(a.elapsed_time(b))
        if len(times) >= 2:
            lo = min(times)
            if abs(times[-1] - times[-2]) <= tol * lo and times[-1] <= (1 + tol) * lo:
                break
    return n


def device_digest_of(source_text: str, common_text: str) -> str:
    """Digest of the device code in a kernel source and common.cuh: every
    __global__ / __device__ definition and every constexpr line. Host-only
    edits leave it unchanged; any device edit changes it."""
    text = common_text + "\n" + source_text
    parts = []
    for m in re.finditer(r"(__global__|__device__)[^;{]*\{", text):
        depth, i = 0, m.end() - 1
        while i < len(text):
            if text[i] == "{":
                depth += 1
            elif text[i] == "}":
                depth -= 1
                if depth == 0:
                    break
            i += 1
        parts.append(text[m.start():i + 1])
    parts += re.findall(r"^\s*constexpr[^\n]*", text, flags=re.M)
    return hashlib.sha256("\n".join(parts).encode()).hexdigest()[:16]


def device_digest(source: str) -> str:
    """device_digest_of for a file of the package's csrc/ (by name)."""
    csrc = os.path.join(ROOT, "decode_dsa_kv_gb300", "csrc")
    return device_digest_of(open(os.path.join(csrc, source)).read(),
                            open(os.path.join(csrc, "common.cuh")).read())


def traffic_record(kernel: str, workload: str, layout: str = None):
    """DRAM bytes per launch (and host-link bytes, where counted) from a
    committed ncu summary, if it was taken on the current device code of that
    kernel's source file: (dram, link), each None when unknown. A record for
    the layout (`kernel/workload/layout`) is preferred to one for any layout."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None, None
    recs = json.load(open(p))
    rec = (recs.get(f"{kernel}/{workload}/{layout}") if layout else None) \
        or recs.get(f"{kernel}/{workload}")
    if not rec:
        return None, None
    src = os.path.join(ROOT, "decode_dsa_kv_gb300", "csrc", rec["source"])
    if not os.path.exists(src) or device_digest(rec["source"]) != rec.get("device_digest"):
        return None, None
    return rec["bytes_per_launch"], rec.get("link_bytes_per_launch")


# ---------------------------------------------------------------------------
# algorithmic bytes / flops per launch
# ---------------------------------------------------------------------------

def algorithmic(w: wl.Workload, lens, hit_frac: float, install_frac: float,
                deferred_frac: float = None, staged: bool = False):
    """Per-launch algorithmic work of every kernel, with the measured hit and
    install fractions (per selected row). The gather writes the installs
    whose victim slots no hit of the step reads; the refill copies the rest
    (`deferred_frac`; all installs when None, as in the per-layer calls).
    Staged layout: the gather moves only the misses (staged in HBM, plus the
    installs on arrival); the attention reads every row where it lies."""
    direct = 0.0 if deferred_frac is None else install_frac - deferred_frac
    deferred = install_frac if deferred_frac is None else deferred_frac
    rows = w.B * w.k
    row = 1152
    miss = 1 - hit_frac
    out = {}
    out["topk"] = {"hbm_bytes": float(np.sum(lens)) * 4 + rows * 4, "link_bytes": 0.0}
    out["plan"] = {"hbm_bytes": rows * (4 + 4) + w.B * (w.P * 4 + 2 * w.S * 4)
                   + rows * miss * (4 * 3 + 1), "link_bytes": 0.0}
    # one launch gathers every layer
    if staged:
        out["gather"] = {"hbm_bytes": w.layers * rows * (miss * (row + 13) + direct * row),
                         "link_bytes": w.layers * rows * miss * row}
    else:
        out["gather"] = {"hbm_bytes": w.layers * rows * (hit_frac * row + row + direct * row + 4),
                         "link_bytes": w.layers * rows * miss * row}
    out["refill"] = {"hbm_bytes": rows * (deferred * 2 * row + install_frac * 13),
                     "link_bytes": 0.0}
    out["sfa"] = {"hbm_bytes": rows * row + w.B * w.H * (1152 + 1024),
                  "link_bytes": 0.0, "flops": 2.0 * w.B * w.H * w.k * (576 + 512)}
    return out


def roofline_of(name, alg, ms, peaks, link_gbs):
    t = ms * 1e-3
    t_hbm = alg["hbm_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_link = alg["link_bytes"] / (link_gbs * 1e9) if link_gbs else 0.0
    t_tc = alg.get("flops", 0.0) / (peaks["bf16_tflops"] * 1e12)
    bound = max((t_hbm, "hbm"), (t_link, "host_link"), (t_tc, "tensor"))[1]
    if bound == "hbm":
        achieved, peak, unit = alg["hbm_bytes"] / t / 1e9, peaks["hbm_gbs"], "GB/s"
    elif bound == "host_link":
        achieved, peak, unit = alg["link_bytes"] / t / 1e9, link_gbs, "GB/s"
    else:
        achieved, peak, unit = alg["flops"] / t / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "ms_per_launch": ms,
            "hbm_gbs": alg["hbm_bytes"] / t / 1e9,
            "link_gbs": alg["link_bytes"] / t / 1e9 if alg["link_bytes"] else 0.0}


def config_of(args, w: wl.Workload, world: int) -> dict:
    """The workload a line reports on; the same dict for both arms."""
    return {"workload": w.name, "B": w.B, "layers": w.layers, "k": w.k,
            "ctx": w.ctx, "sets": w.S, "ways": w.W, "heads": w.H,
            "mtp_draft_steps": args.mtp, "pool_policy": args.policy,
            "layout": args.layout,
            "attention_start": ("layer waits" if args.layer_waits or args.layout != "staged"
                                else "streamed per request"),
            "requests_per_gpu": w.B,
            "score_stream": "forward only: every step run (settle, warm-up, timed, end to end) "
                            "is the next step of the workload's score process; none is replayed",
            "l2": "inputs larger than L2 (host KV, pools and per-step inputs)",
            "parallelism": f"requests sharded over {world} GPU(s), no collective"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and the reference arm)
# ---------------------------------------------------------------------------

def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model Name", "CPU part"):
        m = re.search(rf"^{key}\s*:\s*(.+)$", text, flags=re.M)
        if m:
            return m.group(1).strip()
    return "unknown"


def oracle_worker(spec: dict) -> dict:
    """One worker of the CPU baseline (run in its own process): the oracle's
    whole decode step (top-k, plan, and per layer gather, float64 SFA over all
    heads, refill; metadata update) for requests spec["requests"] of the
    workload, one at a time on a cold pool, until spec["budget_s"] seconds of
    oracle work have run. Every context is full size; on a cold pool the step
    reads only the selected rows, so only those are generated (the rest of
    each host array is untouched zero pages). Only the decode step is timed."""
    import oracle
    import workload.gen as gen
    gen._threads = lambda: 1
    w = wl.scaled(wl.get(spec["workload"]), **spec.get("overrides", {}))
    L = w.layers
    lens = wl.ctx_lens(w)
    scale = 1 / math.sqrt(576)
    rows = secs = 0.0
    n = 0
    for b in spec["requests"]:
        scores = wl.ScoreStream(wl.scaled(w, B=1), b).next()[0]
        n_ctx = int(lens[b])
        ids = oracle.topk_ids(scores, n_ctx, w.k)
        host = np.zeros((L, w.ctx_stride, 576), np.uint16)
        for l in range(L):
            for t in ids:
                wl.normal_bf16(1, 576, w.seed, wl.gen.DOMAIN_KV, l, b, int(t), host[l, t:t + 1])
        q = np.empty((L, w.H, 576), np.uint16)
        for l in range(L):
            wl.normal_bf16(w.H, 576, w.seed, wl.gen.DOMAIN_Q, 0, (l << 32) | b, 0, q[l])
        st = oracle.init_state(L, w.S, w.W)
        t0 = time.perf_counter()
        oracle.decode_step(st, scores, n_ctx, w.k, w.S, w.W, host, q, scale)
        secs += time.perf_counter() - t0
        rows += L * w.k
        n += 1
        if secs >= spec["budget_s"]:
            break
    return {"rows": rows, "secs": secs, "requests": n}


def _spawn_workers(specs, threads_env):
    env = dict(os.environ, **threads_env)
    procs = [subprocess.Popen([sys.executable, os.path.abspath(__file__), "--oracle-worker",
                               json.dumps(sp)], stdout=subprocess.PIPE, text=True, env=env,
                              cwd=ROOT) for sp in specs]
    out = []
    for p in procs:
        o, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError("oracle worker failed")
        out.append(json.loads(o.strip().splitlines()[-1]))
    return out


def cpu_baseline_leg(args, w: wl.Workload, overrides: dict) -> dict:
    """The oracle as it stands, on the host cores, on a bounded sample of the
    workload (cold-pool decode steps of whole requests, all layers): once on
    one core (BLAS and OpenMP held to one thread) and once on every core (one
    single-threaded worker process per core, each on its own requests, all at
    once; the value is the sum of the workers' rates)."""
    one = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}
    cores = os.cpu_count() or 1
    nw = max(1, min(cores, w.B))
    single = _spawn_workers([{"workload": w.name, "overrides": overrides,
                              "requests": list(range(w.B)), "budget_s": args.cpu_seconds}], one)[0]
    per = max(args.cpu_seconds / 2, 1.0)
    par = _spawn_workers([{"workload": w.name, "overrides": overrides,
                           "requests": list(range(i, w.B, nw)), "budget_s": per}
                          for i in range(nw)], one)
    single_rate = single["rows"] / single["secs"]
    par_rate = sum(r["rows"] / r["secs"] for r in par)
    return {"value": par_rate, "unit": UNIT, "cores": nw, "kind": "oracle",
            "single_core_value": single_rate, "cpu_model": cpu_model(),
            "host_cores": cores,
            "sample": (f"cold-pool decode steps of whole {w.name} requests ({w.layers} layers, "
                       f"top-k, plan, gather, float64 SFA over {w.H} heads, refill), full "
                       f"contexts; one core: {single['requests']} request(s) in "
                       f"{single['secs']:.1f} s; all cores: {nw} single-threaded processes, "
                       f"{sum(r['requests'] for r in par)} request(s) in total")}


def oracle_hit_check(w: wl.Workload, scores_steps, lens, first_timed: int, timed: int,
                     gpu_miss_log, requests, policy: str = "fifo") -> dict:
    """The oracle's plan (the FIFO pool, or the LRU pool) followed step by step
    over every step the device ran up to the end of the timed region, for a
    few requests: its hit rate over the timed steps beside the device's for
    the same requests and steps (the plans are bit-exact, so the two must be
    equal)."""
    import oracle
    ora_hits = gpu_hits = 0
    for b in requests:
        st = oracle.init_state(1, w.S, w.W)
        lru = oracle.LruSlots(w.P)
        for t in range(first_timed + timed):
            ids = oracle.topk_ids(scores_steps[t, b], int(lens[b]), w.k)
            if policy == "lru":
                plan = lru.plan(ids, int(lens[b]))
            else:
                plan = oracle.dsa_plan(ids, int(lens[b]), st.tags, st.fifo_ptr, w.S, w.W)
                oracle.metadata_update(st.tags, st.fifo_ptr, plan)
            if t >= first_timed:
                ora_hits += w.k - plan.miss_rows
                gpu_hits += w.k - int(gpu_miss_log[t - first_timed, b])
    n = len(requests) * timed * w.k
    return {"requests": list(requests), "steps": timed, "oracle_hit_rate": ora_hits / n,
            "device_hit_rate": gpu_hits / n}


def run_reference(args, w, rank, world):
    """`--impl reference`: the CPU oracle, on the host cores, timed step by
    step: each step is the next step of request 0's score process through one
    layer of the group (top-k, plan, gather, float64 SFA over all heads,
    refill), on a pool that carries over from step to step (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    lens = wl.ctx_lens(w)
    stream = wl.ScoreStream(wl.scaled(w, B=1))   # request 0's scores
    b = 0
    host = np.zeros((1, w.ctx_stride, 576), np.uint16)
    n_ctx = int(lens[b])
    wl.normal_bf16(n_ctx, 576, w.seed, 1, 0, b, 0, host[0, :n_ctx])
    st = oracle.init_state(1, w.S, w.W)
    scale = 1 / math.sqrt(576)
    step_no = [0]

    def one():
        q = wl.queries(wl.scaled(w, B=1, layers=1), step_no[0])
        oracle.decode_step(st, stream.next()[0], n_ctx, w.k, w.S, w.W, host, q[:1, 0], scale)
        step_no[0] += 1

    for _ in range(args.warmup):
        one()
    dt = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        one()
        dt += time.perf_counter() - t0
    value = args.steps * w.k / dt
    sample = (f"each step: the next step of request 0 of {w.name} (ctx {n_ctx}, k {w.k}, "
              f"{w.H} heads) through 1 layer: top-k, plan, gather, float64 SFA, refill; the pool "
              f"carries over ({args.warmup} warm-up steps first); numpy with its default threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(args, w, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

def run_native(args, w, rank, world, local, overrides):
    import torch
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    import decode_dsa_kv_gb300 as dk
    from decode_dsa_kv_gb300 import _abi as abi

    first = first_request(rank, w)
    lens = wl.ctx_lens(w, first)
    host = dk.HostKV(w.layers, w.B, w.ctx_stride)
    wl.fill_host_kv(w, host.array, first_request=first)
    # the input stream runs forward only: settle, warm-up, timed and
    # end-to-end steps each take the next step of the score process
    n_e2e = 0 if args.no_e2e else min(args.e2e_steps, args.steps)
    n_prof = 0 if args.no_kernel_events else max(1, args.profile_steps)
    n_e2e_prof = min(3, n_prof) if n_e2e else 0
    e2e_steps = (args.e2e_settle_steps + args.warmup + n_e2e + n_e2e_prof) if n_e2e else 0
    T = args.settle_steps + args.warmup + args.steps + n_prof + e2e_steps
    QS = max(1, min(args.query_slots, T))
    stream = wl.ScoreStream(w, first)
    # every registered host buffer of the run is made here, before any timing
    # (registering host memory slows zero-copy reads for a while afterwards)
    scores_pin = dk.PinnedHost((T, w.B, w.ctx_stride), np.float32)
    q_pin = dk.PinnedHost((QS, w.layers, w.B, w.H, 576), np.int16)
    out_pin = dk.PinnedHost((w.layers, w.B, w.H, 512), np.int16)
    link_buf = dk.PinnedHost((1 << 30,), np.uint8, kind="register")  # a DMA source
    for t in range(T):
        scores_pin.array[t] = stream.next()
    for t in range(QS):
        wl.queries(w, t, out=q_pin.array[t].view(np.uint16), first_request=first)
    # device-resident copies of every input step, moved by the SMs (no DMA
    # from these buffers); then one read of every host KV page by the SMs
    # (the first zero-copy access of a host page is slow)
    scores_d = torch.empty(scores_pin.array.shape, dtype=torch.float32, device="cuda")
    q_d = torch.empty(q_pin.array.shape, dtype=torch.int16, device="cuda")
    abi.check(abi.ts_copy(scores_d, scores_pin.dev, scores_pin.array.nbytes, None), "ts_copy")
    abi.check(abi.ts_copy(q_d, q_pin.dev, q_pin.array.nbytes, None), "ts_copy")
    touch = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    host_bytes = host.array.nbytes
    for off in range(0, host_bytes, 1 << 30):
        abi.check(abi.ts_copy(touch, host.dev + off, min(1 << 30, host_bytes - off), None),
                  "ts_copy")
    torch.cuda.synchronize()
    del touch
    staged = args.layout == "staged" and args.policy != "reuse"
    g = dk.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host,
                       policy=args.policy, layout="staged" if staged else "selection",
                       streamed=not args.layer_waits)
    peaks = measured_peaks()
    link = link_peak_gbs(torch, link_buf)

    cursor = [0]  # the next step of the input stream

    def step(timing=None):
        i = cursor[0]
        cursor[0] += 1
        g.step(scores_d[i], q_d[i % QS], timing=timing)

    # the clock sampler starts before the settle steps: the GPU then never
    # idles between them, the warm-up and the timed region (after an idle
    # pause of a fraction of a second the first host reads of a step run
    # slowly, measured on GB300: after 20 s idle, 14.5 GB/s for the first
    # gigabyte read against 210 GB/s once busy)
    sampler = ClockSampler(local)
    if not args.only:
        sampler.start()
    settled = settle(torch, g, step, args.settle_steps) if args.settle_steps > 0 else 0
    for _ in range(args.warmup):
        step()
    g.join()
    torch.cuda.synchronize()
    if g.synchronize():
        raise RuntimeError("device error during warm-up")

    if args.only:
        i = cursor[0]
        return run_only(args, w, g, scores_d[i], q_d[i % QS], peaks, link, lens, host, rank)

    # timed region: K steps, per-kernel events on the launching streams
    first_timed = cursor[0]
    miss_log = torch.zeros((args.steps, w.B), dtype=torch.int32, device="cuda")
    # timing events of every timed step, created before the region: only the
    # step's first start, the gather's start and end (on its own stream) and
    # the last attention's end -- every recorded event costs the streams time
    # (measured: long_context 0.285 ms a step without any, 0.315 with every
    # launch's); the other launches are timed on the steps after the region
    timings = (None if args.no_kernel_events
               else [g.timing(light=True) for _ in range(args.steps)])
    # every launch's events on n_prof steps enqueued right behind the timed
    # region (the GPU does not idle in between; host reads after an idle
    # pause run slowly)
    prof = [g.timing() for _ in range(n_prof)]
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(g.main)
    t_enq0 = time.perf_counter()
    for s in range(args.steps):
        step(timings[s] if timings else None)
        with torch.cuda.stream(g.main):
            miss_log[s].copy_(g.miss_count, non_blocking=True)
    t_enq1 = time.perf_counter()
    g.join(g.main)
    e1.record(g.main)
    for t in prof:
        step(t)
    e1.synchronize()
    t_wall1 = time.time()
    g.join()
    torch.cuda.synchronize()
    barrier(world)
    time.sleep(0.2)
    sampler.stop()
    ms_total = e0.elapsed_time(e1)
    bits = g.synchronize()
    if bits:
        raise RuntimeError(f"device error bits {bits:#x} in the timed region or the steps "
                           "after it")
    # the link's peak measured again after the timed region; the higher of
    # the two is the denominator (one measurement alone has come out 25 % low)
    link = max(link, link_peak_gbs(torch, link_buf))
    ms_step = max_over_ranks(ms_total / args.steps, world, "cuda")
    rows_step = w.rows_per_step * world
    value = rows_step / (ms_step * 1e-3)

    # hit and install fractions over the timed region (plan outputs)
    miss_host = miss_log.cpu().numpy()
    misses = float(miss_host.astype(np.float64).sum())
    hit_frac = 1.0 - misses / (args.steps * w.B * w.k)
    install_frac = (1.0 - hit_frac)   # installs ~ misses (overflow sets install fewer)
    deferred_frac = None
    if args.policy == "fifo":
        # installs into slots read as hits in the same step (the last step's plan)
        valid = torch.arange(w.k, device="cuda")[None, :] < g.miss_count[:, None]
        deferred_frac = float(((g.install == 2) & valid).sum().item()) / (w.B * w.k)

    per_kernel = {}
    alg = algorithmic(w, lens, hit_frac, install_frac, deferred_frac, staged)
    launch_ms = {n: [] for n in KERNELS}
    for t in timings or []:
        for n, v in t.ms().items():
            launch_ms[n].extend(v)
    # every other launch's time from the n_prof steps run right after the
    # timed region with all events (the input stream keeps running forward);
    # the gather's stays the timed region's own
    for t in prof:
        for n, v in t.ms().items():
            if n != "gather":
                launch_ms[n].extend(v)
    for n in KERNELS:
        if not launch_ms[n]:
            continue
        ms = sum(launch_ms[n]) / len(launch_ms[n])
        per_kernel[n] = roofline_of(n, alg[n], ms, peaks, link)
        steps_n = args.steps if n == "gather" else n_prof
        per_kernel[n]["launches_per_step"] = len(launch_ms[n]) / steps_n
        per_kernel[n]["timed_in"] = ("the timed region" if n == "gather"
                                     else f"{n_prof} steps after the timed region")
    if g.arrived is not None and "sfa" in per_kernel:
        # a streamed attention launch's events also span its wait for the
        # gather's rows: its own time comes from launches back to back on the
        # last timed step's rows (layer 0, every row in place)
        span_ms = per_kernel["sfa"]["ms_per_launch"]
        sfa_ms = sfa_alone_ms(torch, g, q_d[(cursor[0] - 1) % QS])
        per_kernel["sfa"] = roofline_of("sfa", alg["sfa"], sfa_ms, peaks, link)
        per_kernel["sfa"].update({"launches_per_step": w.layers, "in_step_span_ms": span_ms,
                                  "timing": "alone: 10 launches back to back on the last timed "
                                            "step's layer-0 rows (chunks + merge)"})
    # each timed step's span (its first launch's start to its last attention's
    # end, CUDA events): how evenly the steps ran (a rare step on this platform
    # stalls for milliseconds while its host reads slow down)
    step_dist = None
    if timings:
        spans = []
        for t in timings:
            ev = t.events
            first = ev[0] if t.with_topk else ev[2]
            spans.append(first.elapsed_time(ev[2 * (3 + w.layers - 1) + 1]))
        spans = np.asarray(spans)
        med = float(np.median(spans))
        step_dist = {"median_ms": round(med, 4), "p90_ms": round(float(np.percentile(spans, 90)), 4),
                     "max_ms": round(float(spans.max()), 4),
                     "steps_over_2x_median": int(np.sum(spans > 2 * med)),
                     "spans_ms": [round(float(x), 3) for x in spans]}
    # where the launches of the last profiled step sat, in microseconds after
    # its first launch began
    last_spans = None
    if prof:
        t_last = prof[-1]
        first = t_last.events[0] if t_last.with_topk else t_last.events[2]
        last_spans = {n: [(round(a, 1), round(b, 1)) for a, b in v]
                      for n, v in t_last.spans(first).items()}
    rf_line = None
    if per_kernel:
        # the gather bounds the step: its host-link reads are the step's
        # largest transfer (with streamed attention, an attention launch's
        # events also span its wait for the gather's rows)
        dom = "gather" if "gather" in per_kernel else max(
            per_kernel, key=lambda n: per_kernel[n]["ms_per_launch"]
            * per_kernel[n]["launches_per_step"])
        rf = dict(per_kernel[dom])
        rf_line = {"kernel": dom, "bound": rf["bound"], "achieved": rf["achieved"],
                   "peak": rf["peak"], "unit": rf["unit"], "frac": rf["frac"],
                   "traffic": None,
                   "peak_source": peaks["source"] if rf["bound"] != "host_link"
                   else "H2D DMA copy of registered host memory, measured in this run"}
        dram, link_bytes = traffic_record(dom, w.name, g.layout)
        rf_line["traffic"] = dram
        if link_bytes is not None:
            rf_line["link_traffic"] = link_bytes

    # end to end through the same schedule with host buffers: per step the
    # scores and queries are copied in from pinned host memory and the
    # attention output copied back; the input stream keeps running forward
    e2e = None
    if n_e2e:
        s_bytes = w.B * w.ctx_stride * 4
        q_bytes = w.layers * w.B * w.H * 576 * 2
        o_bytes = g.out.numel() * 2

        def e2e_step(timing=None):
            i = cursor[0]
            cursor[0] += 1
            # the step's inputs in and its attention output out, copied by the
            # SMs inside the step (dsa_group_step_host): the scores ahead of the
            # top-k, the queries beside the gather, each layer's output after
            # its attention and refill
            g.step_host(scores_pin.dev + i * s_bytes, q_pin.dev + (i % QS) * q_bytes,
                        out_pin.dev, timing=timing)

        e2e_settle = (settle(torch, g, e2e_step, args.e2e_settle_steps)
                      if args.e2e_settle_steps > 0 else 0)
        for _ in range(args.warmup):
            e2e_step()
        # every launch's events on a few end-to-end steps right behind the
        # timed ones (the copies themselves are not timed)
        e2e_prof = [g.timing() for _ in range(n_e2e_prof)]
        torch.cuda.synchronize()
        barrier(world)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(g.main)
        for _ in range(n_e2e):
            e2e_step()
        g.join(g.main)
        f1.record(g.main)
        for t in e2e_prof:
            e2e_step(t)
        torch.cuda.synchronize()
        if g.synchronize():
            raise RuntimeError("device error in the end-to-end steps")
        e2e_ms = max_over_ranks(f0.elapsed_time(f1) / n_e2e, world, "cuda")
        e2e = {"value": rows_step / (e2e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": int(s_bytes + q_bytes), "d2h_bytes_per_step": int(o_bytes),
               "steps": n_e2e, "ms_per_step": e2e_ms, "settle_steps": e2e_settle,
               "copies": "inside the step (dsa_group_step_host: SM copies from / to page-locked "
                         "host memory from ts_host_alloc, overlapped with the step's work)"}
        if e2e_prof:
            # the launches of the last profiled end-to-end step, in microseconds
            # after its top-k began (the scores' copy comes before it)
            t_last = e2e_prof[-1]
            e2e["last_step_spans_us"] = {
                n: [(round(a, 1), round(b, 1)) for a, b in v]
                for n, v in t_last.spans(t_last.events[0]).items()}

    clocks = sampler.summary(t_wall0, t_wall1)
    scores_steps = scores_pin.array[:first_timed + args.steps].copy() if rank == 0 else None
    host.close()
    scores_pin.close()
    q_pin.close()
    out_pin.close()
    link_buf.close()

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and args.policy != "reuse":
        cpu = cpu_baseline_leg(args, w, overrides)
        reqs = [0] if w.ctx > 131072 else sorted({0, w.B // 2, w.B - 1})
        cpu["plan_check"] = oracle_hit_check(w, scores_steps, lens, first_timed, args.steps,
                                             miss_host, reqs, args.policy)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": config_of(args, w, world),
        "roofline": rf_line,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * (topk_launches(w) + LAUNCHES_PLAN + LAUNCHES_GATHER
                                      + w.layers * (sfa_launches(w) + LAUNCHES_POST
                                                    + (1 if args.policy == "fifo" else 0))),
        "clocks": clocks,
        "hit_rate": hit_frac,
        "deferred_install_frac": deferred_frac,
        "host_enqueue_ms_per_step": (t_enq1 - t_enq0) * 1e3 / args.steps,
        "settle_steps": settled,
        "distinct_input_steps": cursor[0],
        "link_peak_gbs": link,
        "step_span_distribution": step_dist,
        "last_step_spans_us": last_spans,
        "kernels": {n: {k2: (round(v, 4) if isinstance(v, float) else v)
                        for k2, v in per_kernel[n].items()} for n in per_kernel},
    }
    print(json.dumps(line), flush=True)


def sfa_alone_ms(torch, g, q, n=10):
    """Mean CUDA-event time of the staged attention (chunks + merge) on layer
    0's rows as the last step left them, launched n times back to back on
    the main stream after 3 untimed launches."""
    from decode_dsa_kv_gb300 import _abi as abi

    def launch():
        abi.check(abi.sfa_mla_decode_pool(q[0], g.pool[0], g.P, g.src_map, g.miss_ids,
                                          g.miss_pos, g.miss_count, g.miss_rows, g.B, g.H, g.k,
                                          g.scale, g.out[0], g.lse[0], g.sfa_ws, g.sfa_ws_bytes,
                                          g.err, g.main), "sfa_mla_decode_pool")
    g.join(g.main)
    for _ in range(3):
        launch()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(g.main)
    for _ in range(n):
        launch()
    e1.record(g.main)
    e1.synchronize()
    return e0.elapsed_time(e1) / n


def run_only(args, w, g, scores, q, peaks, link, lens, host, rank):
    """One kernel, --steps launches on the main stream, on the pool state and
    plan the warm-up left (each launch is idempotent on that state)."""
    import torch

    from decode_dsa_kv_gb300 import _abi as abi
    B, k = w.B, w.k
    m = g.main
    staged = g.layout == "staged"
    launch = {
        "topk": lambda: abi.ts_topk(scores, g.ctx_stride, g.ctx_len, B, g.max_ctx, k, g.ids,
                                    g.topk_ws, g.topk_ws_bytes, g.err, m),
        "plan": lambda: abi.dsa_plan(g.ids, g.ctx_len, B, k, g.tags, g.fifo_ptr, g.S, g.W,
                                     g.src_map, g.miss_ids, g.miss_pos, g.victim, g.install,
                                     g.miss_count, g.miss_rows, g.ptr_next, g.err, m),
        "gather": (lambda: abi.dsa_stage_misses(g.miss_ids, g.miss_pos, g.miss_count, None, None,
                                                B, k, g.pool[0], g.P, host.layer_ptr(0),
                                                g.ctx_stride, g.ctx_len, g.err, m)) if staged
        else (lambda: abi.dsa_gather_kv(g.src_map, g.miss_ids, g.miss_pos, g.miss_count,
                                        g.miss_rows, B, k, g.pool[0], g.P, host.layer_ptr(0),
                                        g.ctx_stride, g.ctx_len, g.sel[0], g.err, m)),
        "sfa": (lambda: abi.sfa_mla_decode_pool(q[0], g.pool[0], g.P, g.src_map, g.miss_ids,
                                                g.miss_pos, g.miss_count, g.miss_rows, B, g.H, k,
                                                g.scale, g.out[0], g.lse[0], g.sfa_ws,
                                                g.sfa_ws_bytes, g.err, m)) if staged
        else (lambda: abi.sfa_mla_decode(q[0], g.sel[0], B, g.H, k, g.scale, g.out[0],
                                         g.lse[0], g.sfa_ws, g.sfa_ws_bytes, g.err, m)),
        # (no metadata update: every launch leaves the same pool state)
        "refill": (lambda: abi.dsa_refill_pool_staged(g.miss_ids, g.miss_pos, g.victim,
                                                      g.install, g.miss_count, B, k, g.pool[0],
                                                      g.P, 0, g.tags, g.fifo_ptr, g.ptr_next,
                                                      g.S, g.W, g.err, m)) if staged
        else (lambda: abi.dsa_refill_pool(g.miss_ids, g.miss_pos, g.victim, g.install,
                                          g.miss_count, B, k, g.sel[0], g.pool[0], g.P, 0,
                                          g.tags, g.fifo_ptr, g.ptr_next, g.S, g.W, g.err, m)),
    }[args.only]
    abi.check(launch(), args.only)
    torch.cuda.synchronize()
    misses = g.miss_count.double().sum().item()
    hit = 1.0 - misses / (B * k)
    # a quarter second of launches right before the timed ones: host reads
    # run slowly for a while after the GPU idles
    t_end = time.time() + 0.25
    while time.time() < t_end:
        for _ in range(8):
            abi.check(launch(), args.only)
        torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(m)
    for _ in range(args.steps):
        abi.check(launch(), args.only)
    e1.record(m)
    torch.cuda.synchronize()
    if g.synchronize():
        raise RuntimeError("device error")
    ms = e0.elapsed_time(e1) / args.steps
    # the per-layer entry points move one layer per launch
    alg = algorithmic(wl.scaled(w, layers=1), lens, hit, 1.0 - hit, staged=staged)[args.only]
    rf = roofline_of(args.only, alg, ms, peaks, link)
    host.close()
    if rank == 0:
        print(json.dumps({"only": args.only, "workload": w.name, "B": B, "launches": args.steps,
                          "hit_rate": hit, "link_peak_gbs": link, **rf}), flush=True)


def main(argv=None):
    args = parse(argv)
    if args.oracle_worker:
        print(json.dumps(oracle_worker(json.loads(args.oracle_worker))), flush=True)
        return
    rank, world, local = dist_env()
    w = wl.get(args.workload)
    overrides = {}
    if args.B:
        overrides["B"] = args.B
    if args.mtp:
        overrides["H"] = w.H * (1 + args.mtp)
    if args.sets:
        overrides["S"] = args.sets
    if overrides:
        w = wl.scaled(w, **overrides)
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    run_native(args, w, rank, world, local, overrides)


if __name__ == "__main__":
    main()
