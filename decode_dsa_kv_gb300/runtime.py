"""Device state and the per-step schedule of one IndexShare group.

The schedule is the one of the GLM-5.2 shared-Indexer KV Cache Offload page,
§4.4 (SFA first, refill later) and §5.1 (one plan per group, per-layer serve,
refill on a side stream synchronised by events, metadata update at the group's
last layer):

  main stream   : ts_topk -> [wait refill_done of the previous step] -> dsa_plan
                  -> record planned
                  -> for each layer l: [wait gathered[l]] -> sfa_mla_decode(l)
  gather stream : [wait planned] -> dsa_gather_kv(0..3), recording gathered[l]
                  after each layer
  side stream   : for each layer l: [wait gathered[l]] -> dsa_refill_pool(l)
                  (the last layer also updates tags and FIFO pointers)
                  -> record refill_done

The plan is shared by the group, so every layer's gather can start as soon as
it exists: the host-link transfers of layer l+1 overlap the attention of
layer l, and each layer's attention still starts the moment its own rows are
in (SFA first). Ordering argument: refill(l) overwrites pool slots that
gather(l) reads, so it waits for gather(l); the next step's plan reads the
tags the last refill writes and rewrites the plan every gather and refill
reads, so it waits for refill_done and comes after the last SFA, which waited
for the last gather; the next step's gather(l) rewrites sel[l], which SFA(l)
and refill(l) read, and it waits for that plan. Memory comes from PyTorch;
the arithmetic runs in libdsakv's kernels only.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import _abi as abi

D = 576
DV = 512


class PinnedHost:
    """A page-locked host buffer owned by numpy and registered with the CUDA
    driver (cudaHostRegister through ts_host_register). Used instead of
    cudaHostAlloc'd memory for every host buffer the device touches: on this
    GB300 platform the first zero-copy read after a large DMA from
    cudaHostAlloc'd memory stalled for about a hundred milliseconds, which
    registered memory does not do."""

    def __init__(self, shape, dtype):
        self.array = np.zeros(shape, dtype=dtype)
        self._host = self.array.ctypes.data
        self.dev = abi.ts_host_register(self._host, self.array.nbytes) if self.array.nbytes else 0

    def tensor(self) -> torch.Tensor:
        return torch.from_numpy(self.array)

    def close(self):
        if self._host and self.array.nbytes:
            abi.ts_host_unregister(self._host)
        self._host = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HostKV:
    """Full latent KV of a group in pinned host memory, read in place by the
    gather: uint16 (bf16 bits) [layers][B][ctx_stride][576]."""

    def __init__(self, layers: int, B: int, ctx_stride: int, array: np.ndarray | None = None):
        shape = (layers, B, ctx_stride, D)
        self.array = np.zeros(shape, dtype=np.uint16) if array is None else array
        assert self.array.shape == shape and self.array.dtype == np.uint16
        assert self.array.flags["C_CONTIGUOUS"]
        self.layers, self.B, self.ctx_stride = layers, B, ctx_stride
        self._host = self.array.ctypes.data
        self.dev = abi.ts_host_register(self._host, self.array.nbytes)
        self.layer_bytes = B * ctx_stride * D * 2

    def layer_ptr(self, l: int) -> int:
        return self.dev + l * self.layer_bytes

    def close(self):
        if self._host:
            abi.ts_host_unregister(self._host)
            self._host = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DecodeGroup:
    """Pool state and buffers for B requests of one IndexShare group."""

    def __init__(self, B: int, layers: int, k: int, S: int, W: int, H: int,
                 ctx_len, ctx_stride: int, host: HostKV, scale: float | None = None,
                 device: str = "cuda", max_ctx: int | None = None):
        self.B, self.L, self.k, self.S, self.W, self.H = B, layers, k, S, W, H
        self.P = S * W
        self.ctx_stride = ctx_stride
        self.scale = 1.0 / math.sqrt(D) if scale is None else scale
        self.host = host
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.ctx_len = torch.as_tensor(np.asarray(ctx_len, np.int32), **i32)
        self.max_ctx = int(np.max(ctx_len)) if max_ctx is None else max_ctx
        # pool state: data per (layer, request), metadata per request
        self.pool = torch.zeros((layers, B, self.P, D), dtype=torch.int16, device=dev)
        self.tags = torch.full((B, self.P), -1, **i32)
        self.fifo_ptr = torch.zeros((B, S), **i32)
        # plan outputs
        self.ids = torch.empty((B, k), **i32)
        self.src_map = torch.empty((B, k), **i32)
        self.miss_ids = torch.empty((B, k), **i32)
        self.miss_pos = torch.empty((B, k), **i32)
        self.victim = torch.empty((B, k), **i32)
        self.install = torch.empty((B, k), dtype=torch.uint8, device=dev)
        self.miss_count = torch.zeros((B,), **i32)
        self.miss_rows = torch.zeros((B,), **i32)
        self.ptr_next = torch.empty((B, S), **i32)
        # per-layer selection buffers and attention outputs
        self.sel = torch.empty((layers, B, k, D), dtype=torch.int16, device=dev)
        self.out = torch.empty((layers, B, H, DV), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((layers, B, H), dtype=torch.float32, device=dev)
        # workspaces and the device error word
        self.topk_ws_bytes = abi.ts_topk_workspace_size(B, self.max_ctx, k)
        self.sfa_ws_bytes = abi.sfa_workspace_size(B, H, k)
        self.topk_ws = torch.empty(self.topk_ws_bytes, dtype=torch.uint8, device=dev)
        self.sfa_ws = torch.empty(self.sfa_ws_bytes, dtype=torch.uint8, device=dev)
        self.err = torch.zeros((1,), **i32)
        # streams and events
        # the critical path (top-k, plan, attention) has the higher priority:
        # when CTAs of several kernels wait for SMs, its CTAs go first
        self.main = torch.cuda.Stream(device=dev, priority=-1)
        self.gstream = torch.cuda.Stream(device=dev, priority=0)
        self.side = torch.cuda.Stream(device=dev, priority=0)
        self.planned = torch.cuda.Event()
        self.gathered = [torch.cuda.Event() for _ in range(layers)]
        self.refill_done = torch.cuda.Event()
        self.refill_done.record(self.side)

    # -- the step --------------------------------------------------------
    def step(self, scores: torch.Tensor, q: torch.Tensor, ids: torch.Tensor | None = None,
             kernel_events=None) -> None:
        """Enqueue one decode step. scores: float32 [B][ctx_stride] (device);
        q: bf16 [layers][B][H][576] (device). With `ids` given (int32 [B][k]),
        the top-k is skipped and those ids are planned. `kernel_events`, when
        given, is a dict name -> list of (start, end) CUDA event pairs that are
        recorded around every launch of that kernel on its own stream."""
        B, k, L = self.B, self.k, self.L
        m, s = self.main, self.side

        def timed(name, stream, fn):
            if kernel_events is not None and name in kernel_events:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                st = fn()
                b.record(stream)
                kernel_events[name].append((a, b))
                return st
            return fn()

        if ids is None:
            abi.check(timed("topk", m, lambda: abi.ts_topk(
                scores, self.ctx_stride, self.ctx_len, B, self.max_ctx, k, self.ids,
                self.topk_ws, self.topk_ws_bytes, self.err, m)), "ts_topk")
            ids = self.ids
        m.wait_event(self.refill_done)
        abi.check(timed("plan", m, lambda: abi.dsa_plan(
            ids, self.ctx_len, B, k, self.tags, self.fifo_ptr, self.S, self.W, self.src_map,
            self.miss_ids, self.miss_pos, self.victim, self.install, self.miss_count,
            self.miss_rows, self.ptr_next, self.err, m)), "dsa_plan")
        self.planned.record(m)
        gs = self.gstream
        gs.wait_event(self.planned)
        for l in range(L):
            abi.check(timed("gather", gs, lambda: abi.dsa_gather_kv(
                self.src_map, self.miss_ids, self.miss_pos, self.miss_count, self.miss_rows, B, k,
                self.pool[l],
                self.P, self.host.layer_ptr(l),
                self.ctx_stride, self.ctx_len, self.sel[l], self.err, gs)), "dsa_gather_kv")
            self.gathered[l].record(gs)
        for l in range(L):
            m.wait_event(self.gathered[l])
            abi.check(timed("sfa", m, lambda: abi.sfa_mla_decode(
                q[l], self.sel[l], B, self.H, k, self.scale, self.out[l], self.lse[l],
                self.sfa_ws, self.sfa_ws_bytes, self.err, m)), "sfa_mla_decode")
            s.wait_event(self.gathered[l])
            last = l == L - 1
            abi.check(timed("refill", s, lambda: abi.dsa_refill_pool(
                self.miss_ids, self.miss_pos, self.victim, self.install, self.miss_count, B, k,
                self.sel[l], self.pool[l], self.P, int(last), self.tags, self.fifo_ptr,
                self.ptr_next, self.S, self.W, self.err, s)), "dsa_refill_pool")
        self.refill_done.record(s)

    def join(self, stream=None) -> None:
        """Make `stream` (default: the current stream) wait for all step work."""
        st = torch.cuda.current_stream() if stream is None else stream
        st.wait_stream(self.main)
        st.wait_stream(self.gstream)
        st.wait_stream(self.side)

    def synchronize(self) -> int:
        """Wait for everything and return (and clear) the device error bits."""
        self.main.synchronize()
        self.gstream.synchronize()
        self.side.synchronize()
        return abi.ts_read_error(self.err, self.main)
