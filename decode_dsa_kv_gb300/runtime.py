"""Device state of one IndexShare group and its per-step schedule.

The schedule is the one of the GLM-5.2 shared-Indexer KV Cache Offload page,
§4.4 (SFA first, refill later) and §5.1 (one plan per group, per-layer serve,
refill on a side stream synchronised by events, metadata update at the group's
last layer). It is enqueued by the library's dsa_group_step in one native call
per step:

  main stream   : ts_topk -> [wait refilled of the previous step] -> dsa_plan
                  -> signal planned
                  -> for each layer l: [wait gathered[l]] -> sfa_mla_decode(l)
  gather stream : [wait planned] -> one gather launch for layers 0..3; the
                  kernel signals gathered[l] as soon as layer l's rows are in
  side stream   : for each layer l: [wait gathered[l]] -> dsa_refill_pool(l)
                  (the last layer also updates tags and FIFO pointers)
                  -> signal refilled

Waits are stream memory operations on device words (the library's `sync`
words), polled by the GPU's front end in HBM; no kernel waits on another.

The plan is shared by the group, so every layer's gather can start as soon as
it exists: the host-link transfers of layer l+1 overlap the attention of
layer l, and each layer's attention still starts the moment its own rows are
in (SFA first); each refill runs beside its layer's attention on a few SMs. Memory and streams come from PyTorch; this module only fills
the descriptor; the arithmetic runs in libdsakv's kernels.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import torch

from . import _abi as abi

D = 576
DV = 512


def plan_metrics(miss_rows, miss_count, miss_ids, install, k: int, S: int) -> dict:
    """Per-request counts of one step's plan, from its outputs as host arrays
    ([B], [B], [B][k], [B][k] or None): positions that hit (k minus the
    positions that miss, repeats included), distinct misses, misses installed
    (install code 1 or 2) and overflow sets (sets that missed more tokens than
    they have ways: their earliest misses are not installed). Each a list of
    B ints; installs and overflow sets are None without an install array
    (the reuse policy installs nothing)."""
    miss_rows = np.asarray(miss_rows)
    miss_count = np.asarray(miss_count)
    B = miss_count.shape[0]
    out = {"hits": [int(k - miss_rows[b]) for b in range(B)],
           "misses": [int(miss_count[b]) for b in range(B)],
           "installs": None, "overflow_sets": None}
    if install is not None:
        install = np.asarray(install)
        miss_ids = np.asarray(miss_ids)
        out["installs"], out["overflow_sets"] = [], []
        for b in range(B):
            M = int(miss_count[b])
            codes = install[b, :M]
            out["installs"].append(int(np.count_nonzero(codes)))
            dropped = miss_ids[b, :M][codes == 0]
            out["overflow_sets"].append(int(np.unique(dropped % S).size))
    return out


class PinnedHost:
    """A page-locked host buffer the device reads and writes in place, seen as
    a numpy array (zero-filled). kind="alloc" (default): ts_host_alloc memory,
    which the SMs read and write fastest (ts_copy, gathers); kind="register":
    numpy memory registered with ts_host_register, for buffers that DMA copies
    read (on GB300, zero-copy reads stalled for a while after a large DMA from
    ts_host_alloc memory; not after one from registered memory)."""

    def __init__(self, shape, dtype, kind: str = "alloc"):
        nbytes = int(np.prod(shape)) * np.dtype(dtype).itemsize
        self.kind = kind
        self._host = 0
        self.dev = 0
        if nbytes == 0:
            self.array = np.zeros(shape, dtype=dtype)
        elif kind == "alloc":
            self._host, self.dev = abi.ts_host_alloc(nbytes)
            buf = (ctypes.c_uint8 * nbytes).from_address(self._host)
            self.array = np.frombuffer(buf, dtype=dtype).reshape(shape)
            self.array[...] = 0
        elif kind == "register":
            self.array = np.zeros(shape, dtype=dtype)
            self._host = self.array.ctypes.data
            self.dev = abi.ts_host_register(self._host, nbytes)
        else:
            raise ValueError(kind)

    def tensor(self) -> torch.Tensor:
        return torch.from_numpy(self.array)

    def close(self):
        if self._host:
            if self.kind == "alloc":
                self.array = None
                abi.ts_host_free(self._host)
            else:
                abi.ts_host_unregister(self._host)
        self._host = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HostKV:
    """Full latent KV of a group in pinned host memory, read in place by the
    gather: uint16 (bf16 bits) [layers][B][ctx_stride][576]. By default the
    memory comes from ts_host_alloc (the gathers read it fastest); a caller's
    own C-contiguous array is registered instead."""

    def __init__(self, layers: int, B: int, ctx_stride: int, array: np.ndarray | None = None):
        shape = (layers, B, ctx_stride, D)
        self.layers, self.B, self.ctx_stride = layers, B, ctx_stride
        self.layer_bytes = B * ctx_stride * D * 2
        nbytes = layers * self.layer_bytes
        if array is None:
            self._host, self.dev = abi.ts_host_alloc(nbytes)
            self._owned = True
            buf = (ctypes.c_uint16 * (nbytes // 2)).from_address(self._host)
            self.array = np.frombuffer(buf, dtype=np.uint16).reshape(shape)
        else:
            assert array.shape == shape and array.dtype == np.uint16
            assert array.flags["C_CONTIGUOUS"]
            self.array = array
            self._host = array.ctypes.data
            self.dev = abi.ts_host_register(self._host, array.nbytes)
            self._owned = False

    def layer_ptr(self, l: int) -> int:
        return self.dev + l * self.layer_bytes

    def close(self):
        if self._host:
            self.array = None
            if self._owned:
                abi.ts_host_free(self._host)
            else:
                abi.ts_host_unregister(self._host)
            self._host = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class StepTiming:
    """CUDA timing events for the launches of one step, created (and recorded
    once, which makes them valid) ahead of use, in the order dsa_group_step
    fills them: top-k, plan, gather (every layer), sfa[l], refill[l].
    light=True hands the step only the top-k's start, the gather's start and
    end and the last attention's end (the step's span and the gather's time);
    the other entries stay unrecorded."""

    def __init__(self, layers: int, stream=None, refills: bool = True, light: bool = False):
        self.layers = layers
        self.refills = refills  # the reuse policy runs no refill
        self.light = light
        n = 2 * (3 + 2 * layers)
        st = torch.cuda.current_stream() if stream is None else stream
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in self.events:
            e.record(st)
        keep = {0, 4, 5, 2 * (3 + layers - 1) + 1} if light else set(range(n))
        self.array = (ctypes.c_void_p * n)(*[e.cuda_event if i in keep else None
                                             for i, e in enumerate(self.events)])
        self.with_topk = True

    def ms(self) -> dict:
        """name -> per-launch milliseconds (after the step completed); with
        light timing the gather only."""
        L = self.layers
        ev = self.events

        def pair(i):
            return ev[2 * i].elapsed_time(ev[2 * i + 1])

        if self.light:
            return {"gather": [pair(2)]}

        out = {"topk": [pair(0)] if self.with_topk else [], "plan": [pair(1)]}
        out["gather"] = [pair(2)]
        out["sfa"] = [pair(3 + l) for l in range(L)]
        out["refill"] = [pair(3 + L + l) for l in range(L)] if self.refills else []
        return out

    def spans(self, t0) -> dict:
        """name -> [(start, end)] in microseconds after event t0."""
        L = self.layers
        ev = self.events

        def span(i):
            return (t0.elapsed_time(ev[2 * i]) * 1e3, t0.elapsed_time(ev[2 * i + 1]) * 1e3)

        out = {"topk": [span(0)] if self.with_topk else [], "plan": [span(1)]}
        out["gather"] = [span(2)]
        out["sfa"] = [span(3 + l) for l in range(L)]
        out["refill"] = [span(3 + L + l) for l in range(L)] if self.refills else []
        return out


class DecodeGroup:
    """Pool state and buffers for B requests of one IndexShare group.

    policy "fifo": the set-associative FIFO pool of S sets x W ways;
    policy "lru": a fully associative pool of S x W entries, least recently
    used first (tags and the slots' recency order per request);
    policy "reuse": the base design's adjacent-step reuse, where the device
    keeps only the previous step's selection (S and W are then unused).
    After a step, `ids` and `sel` hold that step's ids and selection.

    layout "selection": every layer's rows are gathered into `sel`, which the
    attention reads; layout "staged" (FIFO or LRU): the attention reads its rows
    straight from the pool, which then holds P + k rows per request (rows P..
    stage the step's misses at their first positions) and `sel` is None.
    With `streamed` (staged only; B <= 1024) each layer's attention starts
    while the gather runs, every CTA waiting for its own request's rows, each
    layer on a stream of its own (launched once the previous layer's CTAs all
    run); otherwise each layer's attention waits for the whole layer."""

    def __init__(self, B: int, layers: int, k: int, S: int, W: int, H: int,
                 ctx_len, ctx_stride: int, host: HostKV, scale: float | None = None,
                 device: str = "cuda", max_ctx: int | None = None, policy: str = "fifo",
                 layout: str = "selection", streamed: bool = True):
        if policy not in ("fifo", "reuse", "lru"):
            raise ValueError(policy)
        if layout not in ("selection", "staged") or (layout == "staged" and policy == "reuse"):
            raise ValueError(layout)
        self.policy = policy
        self.layout = layout
        self.B, self.L, self.k, self.S, self.W, self.H = B, layers, k, S, W, H
        self.P = S * W
        self.ctx_stride = ctx_stride
        self.scale = 1.0 / math.sqrt(D) if scale is None else scale
        self.host = host
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.ctx_len = torch.as_tensor(np.asarray(ctx_len, np.int32), **i32)
        self.max_ctx = int(np.max(ctx_len)) if max_ctx is None else max_ctx
        # pool state: data per (layer, request), metadata per request (the
        # reuse policy keeps the previous step's ids and selection instead)
        reuse = policy == "reuse"
        P = 1 if reuse else self.P
        rows = P + k if layout == "staged" else P
        self.pool = torch.zeros((layers, B, rows, D), dtype=torch.int16, device=dev)
        self.tags = torch.full((B, P), -1, **i32)
        self.fifo_ptr = torch.zeros((B, S if policy == "fifo" else 1), **i32)
        # LRU pool: each request's slots from least to most recently used
        # (the identity order of a cold pool)
        self.lru_order = (torch.arange(P, **i32).repeat(B, 1) if policy == "lru"
                          else torch.zeros((1,), **i32))
        # plan outputs
        self.ids = torch.empty((B, k), **i32)
        self.src_map = torch.empty((B, k), **i32)
        self.miss_ids = torch.empty((B, k), **i32)
        self.miss_pos = torch.empty((B, k), **i32)
        self.victim = torch.empty((B, k), **i32)
        self.install = torch.empty((B, k), dtype=torch.uint8, device=dev)
        self.miss_count = torch.zeros((B,), **i32)
        self.miss_rows = torch.zeros((B,), **i32)
        self.ptr_next = torch.empty((B, S if policy == "fifo" else 1), **i32)
        # per-layer selection buffers and attention outputs
        self.sel = (None if layout == "staged"
                    else torch.empty((layers, B, k, D), dtype=torch.int16, device=dev))
        if reuse:
            self.prev_ids = torch.full((B, k), -1, **i32)
            self.prev_sel = torch.zeros((layers, B, k, D), dtype=torch.int16, device=dev)
            self._bufs = {t.data_ptr(): t for t in (self.ids, self.prev_ids, self.sel,
                                                    self.prev_sel)}
        self.out = torch.empty((layers, B, H, DV), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((layers, B, H), dtype=torch.float32, device=dev)
        # workspaces and the device error word
        self.topk_ws_bytes = abi.ts_topk_workspace_size(B, self.max_ctx, k)
        streamed = layout == "staged" and streamed
        # streamed: one attention workspace per layer and a stream per layer
        # (the library runs the layers' attention side by side where one
        # layer's CTAs fill at most half of the SMs, else on the main stream)
        self.sfa_ws_bytes = abi.sfa_workspace_size(B, H, k) * (layers if streamed else 1)
        self.topk_ws = torch.empty(self.topk_ws_bytes, dtype=torch.uint8, device=dev)
        self.sfa_ws = torch.empty(self.sfa_ws_bytes, dtype=torch.uint8, device=dev)
        self.err = torch.zeros((1,), **i32)
        # streams and events
        # the critical path (top-k, plan, attention) has the higher priority:
        # when CTAs of several kernels wait for SMs, its CTAs go first
        self.main = torch.cuda.Stream(device=dev, priority=-1)
        self.gstream = torch.cuda.Stream(device=dev, priority=0)
        self.side = torch.cuda.Stream(device=dev, priority=0)
        self.lstreams = ([torch.cuda.Stream(device=dev, priority=-1) for _ in range(layers)]
                         if streamed else [])
        self._lstream_handles = (ctypes.c_void_p * max(1, layers))(
            *[st.cuda_stream for st in self.lstreams])
        # cross-stream signals: device words written and waited on by the
        # streams themselves (zero before the first step)
        self.sync = torch.zeros((5 + 3 * layers,), **i32)
        # staged layout: per (layer, request) arrival counts of the gather, so
        # that each attention CTA starts once its own request's rows are in;
        # the gather's start words; each layer's started attention CTAs
        self.arrived = (torch.zeros((layers * B + 3 + layers,), **i32)
                        if streamed else None)
        # device staging of dsa_group_step_host (made on first use)
        self._io_scores = None
        self._io_q = None
        self.desc = self._descriptor()

    def staged_rows(self, l: int, b: int):
        """Staged layout: the rows the step staged for request b of layer l
        (int16 [k][576]; row j holds the host row of a miss first selected at
        position j, the other rows are stale)."""
        return self.pool[l, b, self.P:]

    def timing(self, light: bool = False) -> StepTiming:
        """Timing events for one step of this group (see StepTiming)."""
        return StepTiming(self.L, self.main, refills=self.policy == "fifo", light=light)

    def _descriptor(self):
        d = abi.DsaGroup()
        d.B, d.layers, d.k, d.S, d.W, d.H = self.B, self.L, self.k, self.S, self.W, self.H
        d.max_ctx, d.ctx_stride, d.scale = self.max_ctx, self.ctx_stride, self.scale
        d.ctx_len = self.ctx_len.data_ptr()
        d.pool, d.pool_tags, d.fifo_ptr = (self.pool.data_ptr(), self.tags.data_ptr(),
                                           self.fifo_ptr.data_ptr())
        d.host_kv = self.host.dev
        for name in ("ids", "src_map", "miss_ids", "miss_pos", "victim", "install",
                     "miss_count", "miss_rows", "ptr_next", "sel", "out", "lse"):
            t = getattr(self, name)
            setattr(d, name, 0 if t is None else t.data_ptr())
        d.layout = abi.DSA_LAYOUT_STAGED if self.layout == "staged" else abi.DSA_LAYOUT_SELECTION
        d.topk_ws, d.topk_ws_bytes = self.topk_ws.data_ptr(), self.topk_ws_bytes
        d.sfa_ws, d.sfa_ws_bytes = self.sfa_ws.data_ptr(), self.sfa_ws_bytes
        d.err = self.err.data_ptr()
        d.arrived = 0 if self.arrived is None else self.arrived.data_ptr()
        d.layer_streams = (ctypes.addressof(self._lstream_handles) if self.lstreams else 0)
        if self.policy == "lru":
            d.policy = abi.DSA_POLICY_LRU
            d.lru_order = self.lru_order.data_ptr()
        if self.policy == "reuse":
            d.policy = abi.DSA_POLICY_REUSE
            d.prev_ids = self.prev_ids.data_ptr()
            d.prev_sel = self.prev_sel.data_ptr()
        d.main_stream = self.main.cuda_stream
        d.gather_stream = self.gstream.cuda_stream
        d.side_stream = self.side.cuda_stream
        d.sync = self.sync.data_ptr()
        d.step = 0
        return d

    # -- the step --------------------------------------------------------
    def step(self, scores: torch.Tensor, q: torch.Tensor, ids: torch.Tensor | None = None,
             timing: StepTiming | None = None) -> None:
        """Enqueue one decode step (one native call). scores: float32
        [B][ctx_stride] (device); q: bf16 bits [layers][B][H][576] (device).
        With `ids` given (int32 [B][k]), the top-k is skipped and those ids are
        planned. `timing`, when given, receives (start, end) events around
        every launch."""
        if timing is not None:
            timing.with_topk = ids is None
        abi.check(abi.dsa_group_step(self.desc, scores, q, ids,
                                     None if timing is None else timing.array),
                  "dsa_group_step")
        if self.policy == "reuse":
            # the step swapped its buffers: this step's ids and selection are
            # now the descriptor's previous ones
            self.ids = self._bufs[self.desc.prev_ids]
            self.sel = self._bufs[self.desc.prev_sel]

    def step_host(self, scores_h: int, q_h: int, out_h: int,
                  timing: StepTiming | None = None) -> None:
        """Enqueue one decode step whose inputs and output live in page-locked
        host memory (device-accessible addresses of float32 [B][ctx_stride]
        scores, bf16 [layers][B][H][576] queries and bf16 [layers][B][H][512]
        output): the library copies them inside the step (dsa_group_step_host).
        The output also lands in `out`."""
        if self._io_scores is None:
            dev = self.out.device
            self._io_scores = torch.empty((self.B, self.ctx_stride), dtype=torch.float32,
                                          device=dev)
            self._io_q = torch.empty((2, self.L, self.B, self.H, D), dtype=torch.int16,
                                     device=dev)
        if timing is not None:
            timing.with_topk = True
        abi.check(abi.dsa_group_step_host(self.desc, scores_h, q_h, out_h, self._io_scores,
                                          self._io_q,
                                          None if timing is None else timing.array),
                  "dsa_group_step_host")
        if self.policy == "reuse":
            self.ids = self._bufs[self.desc.prev_ids]
            self.sel = self._bufs[self.desc.prev_sel]

    def join(self, stream=None) -> None:
        """Make `stream` (default: the current stream) wait for all step work."""
        st = torch.cuda.current_stream() if stream is None else stream
        st.wait_stream(self.main)
        st.wait_stream(self.gstream)
        st.wait_stream(self.side)
        for ls in self.lstreams:
            st.wait_stream(ls)

    def metrics(self) -> dict:
        """plan_metrics of the last step's plan (after synchronize())."""
        install = None if self.policy == "reuse" else self.install.cpu().numpy()
        return plan_metrics(self.miss_rows.cpu().numpy(), self.miss_count.cpu().numpy(),
                            self.miss_ids.cpu().numpy(), install, self.k, self.S)

    # -- checkpoint / resume ---------------------------------------------
    def state(self) -> dict:
        """The pool's state after the steps so far, as host arrays (numpy): its
        metadata (tags, FIFO pointers, LRU order) and every layer's slot rows;
        with the reuse policy the previous step's ids and selection instead of
        the pool. Waits for the group's streams first (raises if the device
        reported an error). load_state puts it into a group of the same
        shapes, after which that group continues as this one would; a test
        resumes the oracle from the same arrays (tags, pointers and rows of
        one request)."""
        if self.synchronize():
            raise RuntimeError("device error bits set before the checkpoint")
        st = {"tags": self.tags.cpu().numpy(), "fifo_ptr": self.fifo_ptr.cpu().numpy(),
              "lru_order": self.lru_order.cpu().numpy()}
        if self.policy == "reuse":
            st["prev_ids"] = self._bufs[self.desc.prev_ids].cpu().numpy()
            st["prev_sel"] = self._bufs[self.desc.prev_sel].cpu().numpy()
        else:
            st["pool"] = self.pool[:, :, :self.P].cpu().numpy()
        return st

    def load_state(self, st: dict) -> None:
        """Put a state from state() into this group (its streams idle); the
        group's own step count and ordering words carry on as they are."""
        self.synchronize()

        def put(t: torch.Tensor, a: np.ndarray):
            if tuple(t.shape) != a.shape:
                raise ValueError(f"state of shape {a.shape} for a buffer of {tuple(t.shape)}")
            t.copy_(torch.from_numpy(np.ascontiguousarray(a)))

        put(self.tags, st["tags"])
        put(self.fifo_ptr, st["fifo_ptr"])
        put(self.lru_order, st["lru_order"])
        if self.policy == "reuse":
            put(self._bufs[self.desc.prev_ids], st["prev_ids"])
            put(self._bufs[self.desc.prev_sel], st["prev_sel"])
        else:
            put(self.pool[:, :, :self.P], st["pool"])
        torch.cuda.synchronize(self.pool.device)

    def synchronize(self) -> int:
        """Wait for everything and return (and clear) the device error bits."""
        self.main.synchronize()
        self.gstream.synchronize()
        self.side.synchronize()
        for ls in self.lstreams:
            ls.synchronize()
        return abi.ts_read_error(self.err, self.main)
