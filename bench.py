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
# + plan 1 + gather 1 (every layer) + layers x (sfa 2 + refill 1; the reuse
# policy has no refill)
LAUNCHES_PLAN, LAUNCHES_GATHER, LAUNCHES_SFA = 1, 1, 2


def topk_launches(w) -> int:
    return 1 if w.ctx <= 131072 else 2


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--workload", default="decode_batch", choices=sorted(wl.BY_NAME))
    ap.add_argument("--period", type=int, default=64,
                    help="distinct input steps generated; steps cycle through them forward "
                         "and back, so the score process has no jump")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--settle-s", type=float, default=6.0,
                    help="longest settle phase before the warm-up (0: none, for profiler runs)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--only", choices=KERNELS, default=None,
                    help="after the warm-up steps, launch only this kernel --steps times "
                         "(on the state the warm-up left) and report its time per launch")
    ap.add_argument("--B", type=int, default=None, help="override the workload's request count")
    ap.add_argument("--sets", type=int, default=None,
                    help="override the pool's sets (16 ways each): 512 = 8K entries, 1024 = 16K")
    ap.add_argument("--policy", choices=("fifo", "reuse"), default="fifo",
                    help="device pool: the set-associative FIFO pool (default) or the base "
                         "design's adjacent-step reuse of the previous selection")
    ap.add_argument("--mtp", type=int, default=0, choices=(0, 1, 2, 3),
                    help="MTP draft steps whose queries are folded into the heads "
                         "(the step attends (1 + N) x H query rows over one selection)")
    ap.add_argument("--no-kernel-events", action="store_true",
                    help="time the steps without per-kernel events (no per-kernel roofline)")
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


def palindrome_index(s: int, period: int) -> int:
    """Step s -> input slot, walking 0..T-1 then T-2..1 and again (no jump)."""
    if period <= 1:
        return 0
    cyc = 2 * period - 2
    r = s % cyc
    return r if r < period else cyc - r


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
                 "--format=csv,noheader,nounits", "-lms", "100"],
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


def settle(torch, g, step, chunk=20, limit_s=6.0, tol=0.03, min_steps=0):
    """Run steps until the step time is steady: on this platform, zero-copy
    reads of host memory run slow for a second or two after host memory is
    registered, copied by DMA or freed. Untimed (extra warm-up); returns the
    steps run. Stops when two consecutive chunks agree within `tol` and are
    within `tol` of the fastest chunk seen, or after `limit_s` seconds."""
    t_end = time.time() + limit_s
    times, s = [], 0
    while time.time() < t_end:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(g.main)
        for _ in range(chunk):
            step(s)
            s += 1
        g.join(g.main)
        b.record(g.main)
        b.synchronize()
        times.append(a.elapsed_time(b))
        if len(times) >= 2 and s >= min_steps:
            lo = min(times)
            if abs(times[-1] - times[-2]) <= tol * lo and times[-1] <= (1 + tol) * lo:
                break
    return s


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


def traffic_record(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current device code of that kernel's source file (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(f"{kernel}/{workload}")
    if not rec:
        return None
    src = os.path.join(ROOT, "decode_dsa_kv_gb300", "csrc", rec["source"])
    if not os.path.exists(src):
        return None
    ok = device_digest(rec["source"]) == rec.get("device_digest")
    return rec["bytes_per_launch"] if ok else None


# ---------------------------------------------------------------------------
# algorithmic bytes / flops per launch
# ---------------------------------------------------------------------------

def algorithmic(w: wl.Workload, lens, hit_frac: float, install_frac: float,
                deferred_frac: float = None):
    """Per-launch algorithmic work of every kernel, with the measured hit and
    install fractions (per selected row). The gather writes the installs
    whose victim slots no hit of the step reads; the refill copies the rest
    (`deferred_frac`; all installs when None, as in the per-layer calls)."""
    direct = 0.0 if deferred_frac is None else install_frac - deferred_frac
    deferred = install_frac if deferred_frac is None else deferred_frac
    rows = w.B * w.k
    row = 1152
    out = {}
    out["topk"] = {"hbm_bytes": float(np.sum(lens)) * 4 + rows * 4, "link_bytes": 0.0}
    out["plan"] = {"hbm_bytes": rows * (4 + 4) + w.B * (w.P * 4 + 2 * w.S * 4)
                   + rows * (1 - hit_frac) * (4 * 3 + 1), "link_bytes": 0.0}
    # one launch gathers every layer
    out["gather"] = {"hbm_bytes": w.layers * rows * (hit_frac * row + row + direct * row + 4),
                     "link_bytes": w.layers * rows * (1 - hit_frac) * row}
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
            "requests_per_gpu": w.B,
            "distinct_input_steps": max(1, min(args.period, args.warmup + args.steps)),
            "l2": "inputs larger than L2 (host KV, pools and per-step inputs)",
            "parallelism": f"requests sharded over {world} GPU(s), no collective"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(w: wl.Workload, budget_s: float, layers_per_request: int | None = None,
                  first: int = 0):
    """Run the oracle's decode step on requests of the workload (full
    contexts), one request at a time, for about `budget_s` seconds of CPU work.
    Returns (rows served, seconds, requests, layers)."""
    import oracle
    L = w.layers if layers_per_request is None else layers_per_request
    lens = wl.ctx_lens(w, first)
    stream = wl.ScoreStream(w, first)
    scores = stream.next()
    q = wl.queries(w, 0, first_request=first)
    rows = secs = 0.0
    n = 0
    for b in range(w.B):
        host = np.zeros((L, 1, w.ctx_stride, 576), np.uint16)
        for l in range(L):
            n_ctx = int(lens[b])
            wl.normal_bf16(n_ctx, 576, w.seed, 1, l, first + b, 0, host[l, 0, :n_ctx])
        st = oracle.init_state(L, w.S, w.W)
        t0 = time.perf_counter()
        oracle.decode_step(st, scores[b], int(lens[b]), w.k, w.S, w.W, host[:, 0], q[:L, b],
                           1 / math.sqrt(576))
        secs += time.perf_counter() - t0
        rows += L * w.k
        n += 1
        if secs >= budget_s:
            break
    return rows, secs, n, L


def run_reference(args, w, rank, world):
    """`--impl reference`: the CPU oracle, on the host cores, timed step by
    step on a bounded sample of the workload (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    lens = wl.ctx_lens(w)
    stream = wl.ScoreStream(w)
    scores = stream.next()
    q = wl.queries(w, 0)
    b = 0
    host = np.zeros((1, w.ctx_stride, 576), np.uint16)
    n_ctx = int(lens[b])
    wl.normal_bf16(n_ctx, 576, w.seed, 1, 0, b, 0, host[0, :n_ctx])
    st = oracle.init_state(1, w.S, w.W)
    scale = 1 / math.sqrt(576)

    def one():
        oracle.decode_step(st, scores[b], n_ctx, w.k, w.S, w.W, host, q[:1, b], scale)

    # each step: one request, one layer of the group (top-k, plan, gather,
    # SFA over all heads, refill); the first timed probe sizes the run
    for _ in range(min(args.warmup, 3)):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    value = args.steps * w.k / dt
    sample = (f"each step: 1 request x 1 layer of {w.name} (ctx {n_ctx}, k {w.k}, "
              f"{w.H} heads): top-k, plan, gather, fp64 SFA, refill")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": min(args.warmup, 3),
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(args, w, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

def run_native(args, w, rank, world, local):
    import torch
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    import decode_dsa_kv_gb300 as dk

    first = first_request(rank, w)
    lens = wl.ctx_lens(w, first)
    host = dk.HostKV(w.layers, w.B, w.ctx_stride)
    wl.fill_host_kv(w, host.array, first_request=first)
    T = max(1, min(args.period, args.warmup + args.steps))
    stream = wl.ScoreStream(w, first)
    # every registered host buffer of the run is made here, before any timing
    # (registering host memory slows zero-copy reads for a while afterwards)
    scores_pin = dk.PinnedHost((T, w.B, w.ctx_stride), np.float32)
    q_pin = dk.PinnedHost((T, w.layers, w.B, w.H, 576), np.int16)
    out_pin = dk.PinnedHost((w.layers, w.B, w.H, 512), np.int16)
    link_buf = dk.PinnedHost((1 << 30,), np.uint8, kind="register")  # a DMA source
    for t in range(T):
        scores_pin.array[t] = stream.next()
        wl.queries(w, t, out=q_pin.array[t].view(np.uint16), first_request=first)
    # device-resident copies of every input slot, moved by the SMs (no DMA
    # from these buffers)
    from decode_dsa_kv_gb300 import _abi as abi
    scores_d = torch.empty(scores_pin.array.shape, dtype=torch.float32, device="cuda")
    q_d = torch.empty(q_pin.array.shape, dtype=torch.int16, device="cuda")
    abi.check(abi.ts_copy(scores_d, scores_pin.dev, scores_pin.array.nbytes, None), "ts_copy")
    abi.check(abi.ts_copy(q_d, q_pin.dev, q_pin.array.nbytes, None), "ts_copy")
    torch.cuda.synchronize()
    g = dk.DecodeGroup(w.B, w.layers, w.k, w.S, w.W, w.H, lens, w.ctx_stride, host,
                       policy=args.policy)
    peaks = measured_peaks()
    link = link_peak_gbs(torch, link_buf)

    base = [0]  # steps run before warm-up step 0 (the settle phase)

    def step(s, timing=None):
        i = palindrome_index(base[0] + s, T)
        g.step(scores_d[i], q_d[i], timing=timing)

    # settle, then warm-up; the score process runs on without a jump
    base[0] = settle(torch, g, step, limit_s=args.settle_s) if args.settle_s > 0 else 0
    for s in range(args.warmup):
        step(s)
    g.join()
    torch.cuda.synchronize()
    if g.synchronize():
        raise RuntimeError("device error during warm-up")

    if args.only:
        i = palindrome_index(base[0] + args.warmup, T)
        return run_only(args, w, g, scores_d[i], q_d[i], peaks, link, lens, host, rank)

    # timed region: K steps, per-kernel events on the launching streams
    miss_log = torch.zeros((args.steps, w.B), dtype=torch.int32, device="cuda")
    inst_log = torch.zeros((args.steps,), dtype=torch.int64, device="cuda")
    # per-launch timing events of every timed step, created before the region
    timings = (None if args.no_kernel_events
               else [g.timing() for _ in range(args.steps)])
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(g.main)
    t_enq0 = time.perf_counter()
    for s in range(args.steps):
        step(args.warmup + s, timings[s] if timings else None)
        with torch.cuda.stream(g.main):
            miss_log[s].copy_(g.miss_count, non_blocking=True)
    t_enq1 = time.perf_counter()
    g.join(g.main)
    e1.record(g.main)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    time.sleep(0.2)
    sampler.stop()
    ms_total = e0.elapsed_time(e1)
    bits = g.synchronize()
    if bits:
        raise RuntimeError(f"device error bits {bits:#x} in the timed region")
    ms_step = max_over_ranks(ms_total / args.steps, world, "cuda")
    rows_step = w.rows_per_step * world
    value = rows_step / (ms_step * 1e-3)

    # hit and install fractions over the timed region (plan outputs)
    misses = miss_log.double().sum().item()
    hit_frac = 1.0 - misses / (args.steps * w.B * w.k)
    install_frac = (1.0 - hit_frac)   # installs ~ misses (overflow sets install fewer)
    deferred_frac = None
    if args.policy == "fifo":
        # installs into slots read as hits in the same step (the last step's plan)
        valid = torch.arange(w.k, device="cuda")[None, :] < g.miss_count[:, None]
        deferred_frac = float(((g.install == 2) & valid).sum().item()) / (w.B * w.k)

    per_kernel = {}
    alg = algorithmic(w, lens, hit_frac, install_frac, deferred_frac)
    launch_ms = {n: [] for n in KERNELS}
    for t in timings or []:
        for n, v in t.ms().items():
            launch_ms[n].extend(v)
    for n in KERNELS:
        if not launch_ms[n]:
            continue
        ms = sum(launch_ms[n]) / len(launch_ms[n])
        per_kernel[n] = roofline_of(n, alg[n], ms, peaks, link)
        per_kernel[n]["launches_per_step"] = len(launch_ms[n]) / args.steps
    rf_line = None
    if per_kernel:
        dom = max(per_kernel, key=lambda n: per_kernel[n]["ms_per_launch"]
                  * per_kernel[n]["launches_per_step"])
        rf = dict(per_kernel[dom])
        rf_line = {"kernel": dom, "bound": rf["bound"], "achieved": rf["achieved"],
                   "peak": rf["peak"], "unit": rf["unit"], "frac": rf["frac"],
                   "traffic": traffic_record(dom, w.name),
                   "peak_source": peaks["source"] if rf["bound"] != "host_link"
                   else "H2D DMA copy of registered host memory, measured in this run"}

    # end to end through the same schedule with host buffers: per step the
    # scores and queries are copied in from pinned host memory and the
    # attention output copied back
    e2e = None
    if not args.no_e2e:
        from decode_dsa_kv_gb300 import _abi as abi
        ins_s = torch.empty((w.B, w.ctx_stride), dtype=torch.float32, device="cuda")
        ins_q = torch.empty((w.layers, w.B, w.H, 576), dtype=torch.int16, device="cuda")
        s_bytes, q_bytes = ins_s.numel() * 4, ins_q.numel() * 2
        o_bytes = g.out.numel() * 2
        n_e2e = min(args.e2e_steps, args.steps)
        e0 = [base[0] + args.warmup + args.steps]

        def e2e_step(s):
            i = palindrome_index(e0[0] + s, T)
            # the step's inputs in and its attention output out, through the SMs
            abi.check(abi.ts_copy(ins_s, scores_pin.dev + i * s_bytes, s_bytes, g.main), "ts_copy")
            abi.check(abi.ts_copy(ins_q, q_pin.dev + i * q_bytes, q_bytes, g.main), "ts_copy")
            g.step(ins_s, ins_q)
            abi.check(abi.ts_copy(out_pin.dev, g.out, o_bytes, g.main), "ts_copy")

        # warm-up of the end-to-end loop: settle (the first zero-copy touch of
        # each host page is slow) and at least one pass over every input slot
        e2e_settle = (settle(torch, g, e2e_step, min_steps=2 * T, limit_s=args.settle_s)
                      if args.settle_s > 0 else 0)
        e0[0] += e2e_settle
        for s in range(args.warmup):
            e2e_step(s)
        e0[0] += args.warmup
        torch.cuda.synchronize()
        barrier(world)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(g.main)
        for s in range(n_e2e):
            e2e_step(s)
        g.join(g.main)
        f1.record(g.main)
        torch.cuda.synchronize()
        if g.synchronize():
            raise RuntimeError("device error in the end-to-end steps")
        e2e_ms = max_over_ranks(f0.elapsed_time(f1) / n_e2e, world, "cuda")
        e2e = {"value": rows_step / (e2e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": int(s_bytes + q_bytes), "d2h_bytes_per_step": int(o_bytes),
               "steps": n_e2e, "ms_per_step": e2e_ms, "settle_steps": e2e_settle,
               "copies": "ts_copy (SM copies) from / to page-locked host memory (ts_host_alloc)"}

    clocks = sampler.summary(t_wall0, t_wall1)
    host.close()
    scores_pin.close()
    q_pin.close()
    out_pin.close()
    link_buf.close()

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and args.policy == "fifo":
        rows, secs, nreq, L = oracle_sample(w, args.cpu_seconds)
        cpu = {"value": rows / secs, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{nreq} request(s) x {L} layers of {w.name}, one decode step each "
                         f"(cold pool), full contexts; numpy with its default threads",
               "seconds": secs}
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
                                      + w.layers * (LAUNCHES_SFA
                                                    + (1 if args.policy == "fifo" else 0))),
        "clocks": clocks,
        "hit_rate": hit_frac,
        "deferred_install_frac": deferred_frac,
        "host_enqueue_ms_per_step": (t_enq1 - t_enq0) * 1e3 / args.steps,
        "settle_steps": base[0],
        "link_peak_gbs": link,
        "kernels": {n: {k2: (round(v, 4) if isinstance(v, float) else v)
                        for k2, v in per_kernel[n].items()} for n in per_kernel},
    }
    print(json.dumps(line), flush=True)


def run_only(args, w, g, scores, q, peaks, link, lens, host, rank):
    """One kernel, --steps launches on the main stream, on the pool state and
    plan the warm-up left (each launch is idempotent on that state)."""
    import torch

    from decode_dsa_kv_gb300 import _abi as abi
    B, k = w.B, w.k
    m = g.main
    launch = {
        "topk": lambda: abi.ts_topk(scores, g.ctx_stride, g.ctx_len, B, g.max_ctx, k, g.ids,
                                    g.topk_ws, g.topk_ws_bytes, g.err, m),
        "plan": lambda: abi.dsa_plan(g.ids, g.ctx_len, B, k, g.tags, g.fifo_ptr, g.S, g.W,
                                     g.src_map, g.miss_ids, g.miss_pos, g.victim, g.install,
                                     g.miss_count, g.miss_rows, g.ptr_next, g.err, m),
        "gather": lambda: abi.dsa_gather_kv(g.src_map, g.miss_ids, g.miss_pos, g.miss_count,
                                            g.miss_rows, B, k, g.pool[0], g.P, host.layer_ptr(0),
                                            g.ctx_stride, g.ctx_len, g.sel[0], g.err, m),
        "sfa": lambda: abi.sfa_mla_decode(q[0], g.sel[0], B, g.H, k, g.scale, g.out[0],
                                          g.lse[0], g.sfa_ws, g.sfa_ws_bytes, g.err, m),
        "refill": lambda: abi.dsa_refill_pool(g.miss_ids, g.miss_pos, g.victim, g.install,
                                              g.miss_count, B, k, g.sel[0], g.pool[0], g.P, 0,
                                              g.tags, g.fifo_ptr, g.ptr_next, g.S, g.W, g.err,
                                              m),
    }[args.only]
    abi.check(launch(), args.only)
    torch.cuda.synchronize()
    misses = g.miss_count.double().sum().item()
    hit = 1.0 - misses / (B * k)
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
    alg = algorithmic(wl.scaled(w, layers=1), lens, hit, 1.0 - hit)[args.only]
    rf = roofline_of(args.only, alg, ms, peaks, link)
    host.close()
    if rank == 0:
        print(json.dumps({"only": args.only, "workload": w.name, "B": B, "launches": args.steps,
                          "hit_rate": hit, "link_peak_gbs": link, **rf}), flush=True)


def main(argv=None):
    args = parse(argv)
    rank, world, local = dist_env()
    w = wl.get(args.workload)
    if args.B:
        w = wl.scaled(w, B=args.B)
    if args.mtp:
        w = wl.scaled(w, H=w.H * (1 + args.mtp))
    if args.sets:
        w = wl.scaled(w, S=args.sets)
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    run_native(args, w, rank, world, local)


if __name__ == "__main__":
    main()
