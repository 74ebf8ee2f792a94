"""The C ABI's host-side checks: argument and shape errors come back as status
codes before anything is enqueued, and the workspace-size functions agree with
the layouts they describe. Run without a device: every call below must be
refused by a check (a check that failed to fire would go on to enqueue work
on the fake addresses used here, so these tests are skipped where a GPU is
visible)."""
import ctypes
import math

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="host checks are exercised on machines without a GPU")

from _util import ensure_library  # noqa: E402

ensure_library()
from decode_dsa_kv_gb300 import _abi  # noqa: E402

L = _abi._lib
OK, INVALID, UNSUPPORTED, WORKSPACE = (_abi.TS_OK, _abi.TS_ERR_INVALID_ARG,
                                       _abi.TS_ERR_UNSUPPORTED, _abi.TS_ERR_WORKSPACE)
A = 0x10000          # a fake, 256-byte aligned address (never dereferenced)
A2 = 0x20000
MIS = A + 8          # 8 bytes off a 16-byte boundary


def test_status_strings_are_distinct():
    codes = [OK, INVALID, UNSUPPORTED, WORKSPACE, _abi.TS_ERR_CUDA, _abi.TS_ERR_DEVICE_CHECK]
    texts = [_abi.ts_status_string(c) for c in codes]
    assert len(set(texts)) == len(texts)
    assert _abi.ts_status_string(12345) == "unknown status"


def test_workspace_sizes():
    assert L.ts_topk_workspace_size(0, 4096, 256) == 0
    assert L.ts_topk_workspace_size(1, 0, 256) == 0
    # histograms, counters, candidate list and bitmap of every request
    B, n = 32, 65536
    assert L.ts_topk_workspace_size(B, n, 2048) >= B * 4096 * 4 + B * n * 8 + B * n // 8
    assert L.ts_topk_workspace_size(2 * B, n, 2048) > L.ts_topk_workspace_size(B, n, 2048)
    assert L.sfa_workspace_size(0, 128, 2048) == 0
    # fp32 partials [B][head tiles][chunks][512][128] and (max, sum) pairs
    B, H, k = 32, 128, 2048
    slots = B * 1 * math.ceil(k / 512) * 128
    want = -(-slots * 512 * 4 // 256) * 256 + -(-slots * 8 // 256) * 256
    assert L.sfa_workspace_size(B, H, k) == want
    assert L.sfa_workspace_size(B, 129, k) == 2 * want      # a second head tile


def topk(scores=A, stride=4096, ctx_len=A, B=1, max_ctx=4096, k=256, ids=A, ws=A2, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = L.ts_topk_workspace_size(B, max_ctx, k)
    return L.ts_topk(scores, stride, ctx_len, B, max_ctx, k, ids, ws, ws_bytes, None, None)


@pytest.mark.parametrize("kw, want", [
    (dict(scores=None), INVALID),
    (dict(ids=None), INVALID),
    (dict(B=0), INVALID),
    (dict(k=0), INVALID),
    (dict(k=5000), INVALID),                  # k above the context
    (dict(stride=1000), INVALID),             # row stride below the context
    (dict(stride=4098), INVALID),             # stride not a multiple of 4 floats
    (dict(scores=MIS), INVALID),
    (dict(k=9000, max_ctx=10000, stride=10000), UNSUPPORTED),   # k past the largest supported
    (dict(B=70000), UNSUPPORTED),
    (dict(ws=None), INVALID),
    (dict(ws=A2 + 16), WORKSPACE),            # workspace not 256-byte aligned
    (dict(ws_bytes=1024), WORKSPACE),         # workspace too small
])
def test_topk_refusals(kw, want):
    assert topk(**kw) == want


def test_topk_noalloc_limits():
    f = L.ts_topk_noalloc
    assert f(None, 4096, A, 1, 4096, 256, A, None, None) == INVALID
    assert f(A, 4096, A, 129, 4096, 256, A, None, None) == UNSUPPORTED        # B past 128
    assert f(A, 65536, A, 128, 65536, 2048, A, None, None) == UNSUPPORTED     # 8M positions


def plan(ids=A, ctx=A, B=1, k=256, tags=A, ptr=A, S=256, W=4, outs=A):
    return L.dsa_plan(ids, ctx, B, k, tags, ptr, S, W, outs, outs, outs, outs, outs, outs, outs,
                      outs, None, None)


@pytest.mark.parametrize("kw, want", [
    (dict(ids=None), INVALID),
    (dict(outs=None), INVALID),
    (dict(B=0), INVALID),
    (dict(W=0), INVALID),
    (dict(S=0), INVALID),
    (dict(W=33), UNSUPPORTED),                 # more ways than a warp's lanes
    (dict(k=100000), UNSUPPORTED),
    (dict(S=1 << 20, W=32), UNSUPPORTED),      # pool past 2^24 entries
])
def test_plan_refusals(kw, want):
    assert plan(**kw) == want


def test_plan_reuse_refusals():
    f = L.dsa_plan_reuse
    assert f(None, A, A, 1, 256, A, A, A, A, A, None, None) == INVALID
    assert f(A, A, A, 0, 256, A, A, A, A, A, None, None) == INVALID
    assert f(A, A, A, 1, 20000, A, A, A, A, A, None, None) == UNSUPPORTED


def gather(pool=A, host=A, sel=A, B=1, k=256, P=1024, stride=4096, maps=A):
    return L.dsa_gather_kv(maps, maps, maps, maps, maps, B, k, pool, P, host, stride, maps, sel,
                           None, None)


@pytest.mark.parametrize("kw, want", [
    (dict(maps=None), INVALID),
    (dict(pool=None), INVALID),
    (dict(B=0), INVALID),
    (dict(P=0), INVALID),
    (dict(stride=0), INVALID),
    (dict(pool=MIS), INVALID),
    (dict(host=MIS), INVALID),
    (dict(sel=MIS), INVALID),
])
def test_gather_refusals(kw, want):
    assert gather(**kw) == want


def test_refill_refusals():
    f = L.dsa_refill_pool
    args = [A, A, A, A, A, 1, 256, A, A, 1024, 1, A, A, A, 256, 4, None, None]
    bad_sel = list(args)
    bad_sel[7] = MIS
    assert f(*bad_sel) == INVALID
    no_tags = list(args)
    no_tags[11] = None                          # metadata update without the tags
    assert f(*no_tags) == INVALID
    zero_b = list(args)
    zero_b[5] = 0
    assert f(*zero_b) == INVALID


def sfa(q=A, sel=A, B=1, H=16, k=256, scale=1 / 24, out=A, ws=A2, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = L.sfa_workspace_size(max(B, 1), max(H, 1), max(k, 1))
    return L.sfa_mla_decode(q, sel, B, H, k, scale, out, None, ws, ws_bytes, None, None)


@pytest.mark.parametrize("kw, want", [
    (dict(q=None), INVALID),
    (dict(out=None), INVALID),
    (dict(ws=None), INVALID),
    (dict(B=0), INVALID),
    (dict(k=0), INVALID),
    (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID),
    (dict(q=MIS), INVALID),
    (dict(sel=MIS), INVALID),
    (dict(B=70000), UNSUPPORTED),
    (dict(ws=A2 + 16), WORKSPACE),
    (dict(ws_bytes=256), WORKSPACE),
])
def test_sfa_refusals(kw, want):
    assert sfa(**kw) == want


def test_small_entry_points():
    assert L.ts_copy(None, A, 64, None) == INVALID
    assert L.ts_copy(A, MIS, 64, None) == INVALID
    assert L.ts_copy(A, A2, 20, None) == INVALID       # not a multiple of 16 bytes
    assert L.ts_read_error(None, None, None) == INVALID
    dev = ctypes.c_void_p()
    assert L.ts_host_register(None, 64, ctypes.byref(dev)) == INVALID
    assert L.ts_host_alloc(0, ctypes.byref(dev), ctypes.byref(dev)) == INVALID
    assert L.ts_host_free(None) == INVALID
    assert L.dsa_group_step(None, A, A, None, None) == INVALID


def test_group_step_refusals():
    g = _abi.DsaGroup()
    g.B, g.layers, g.k, g.S, g.W, g.H = 1, 1, 256, 256, 4, 16
    g.sync = A
    assert L.dsa_group_step(ctypes.byref(g), None, A, None, None) == INVALID   # no scores, no ids
    g.layers = 0
    assert L.dsa_group_step(ctypes.byref(g), A, A, None, None) == INVALID
    g.layers, g.policy = 1, 7
    assert L.dsa_group_step(ctypes.byref(g), A, A, None, None) == INVALID     # unknown policy
    g.policy, g.sync = 0, A + 2
    assert L.dsa_group_step(ctypes.byref(g), A, A, None, None) == INVALID     # sync word misaligned


def test_group_step_layer_stream_refusals():
    # layer streams (streamed staged layout): none of them NULL, and one
    # attention workspace per layer; refused before anything is enqueued
    g = _abi.DsaGroup()
    g.B, g.layers, g.k, g.S, g.W, g.H = 2, 2, 16, 8, 4, 128
    g.layout, g.policy = _abi.DSA_LAYOUT_STAGED, _abi.DSA_POLICY_FIFO
    g.sync, g.arrived = A, A2
    streams = (ctypes.c_void_p * 2)(0x1234, None)
    g.layer_streams = ctypes.addressof(streams)
    assert L.dsa_group_step(ctypes.byref(g), A, A, None, None) == INVALID     # a NULL layer stream
    streams[1] = 0x5678
    g.sfa_ws_bytes = L.sfa_workspace_size(2, 128, 16)                          # one layer's only
    assert L.dsa_group_step(ctypes.byref(g), A, A, None, None) == _abi.TS_ERR_WORKSPACE
    g.sfa_ws_bytes = 2 * L.sfa_workspace_size(2, 128, 16)
    assert L.dsa_group_step(ctypes.byref(g), A, A, None, None) == INVALID     # null buffers next
    assert g.step == 0
