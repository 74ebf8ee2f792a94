"""ctypes binding of libdsakv.so: the same entry points as include/dsakv.h,
with argument marshalling only (tensors -> device pointers, streams -> handles).
Every step of the path runs in the library's CUDA kernels; nothing here
computes. Importing this module fails loudly when the library is missing."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsakv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m decode_dsa_kv_gb300.build` "
        "(the decode path has no fallback)")
_lib = ctypes.CDLL(LIB_PATH)

TS_OK = 0
TS_ERR_INVALID_ARG = -1
TS_ERR_UNSUPPORTED = -2
TS_ERR_WORKSPACE = -3
TS_ERR_CUDA = -4
TS_ERR_DEVICE_CHECK = -5

TS_DEVERR_ID_RANGE = 0x01
TS_DEVERR_NAN = 0x02
TS_DEVERR_SLOT_RANGE = 0x04
TS_DEVERR_PTR_RANGE = 0x08
TS_DEVERR_CTX = 0x10
TS_DEVERR_TIMEOUT = 0x20
TS_DEVERR_COUNT = 0x40
TS_DEVERR_ORDER = 0x80

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float

# name -> (restype, argtypes), in header order
_SIGS = {
    "ts_status_string": (ctypes.c_char_p, [_I]),
    "ts_host_register": (_I, [_P, _SZ, ctypes.POINTER(ctypes.c_void_p)]),
    "ts_host_unregister": (_I, [_P]),
    "ts_host_alloc": (_I, [_SZ, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p)]),
    "ts_host_free": (_I, [_P]),
    "ts_copy": (_I, [_P, _P, _SZ, _P]),
    "ts_read_error": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "ts_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "ts_topk_workspace_size": (_SZ, [_I, _I, _I]),
    "ts_topk": (_I, [_P, _I64, _P, _I, _I, _I, _P, _P, _SZ, _P, _P]),
    "ts_topk_noalloc": (_I, [_P, _I64, _P, _I, _I, _I, _P, _P, _P]),
    "dsa_plan": (_I, [_P, _P, _I, _I, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dsa_plan_reuse": (_I, [_P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "dsa_plan_lru": (_I, [_P, _P, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dsa_gather_kv": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _I, _P, _I64, _P, _P, _P, _P]),
    "dsa_stage_misses": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _I, _P, _I64, _P, _P, _P]),
    "dsa_refill_pool": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _P, _P, _P, _I, _I,
                             _P, _P]),
    "dsa_refill_pool_staged": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _I, _I, _P, _P, _P, _I, _I,
                                    _P, _P]),
    "sfa_workspace_size": (_SZ, [_I, _I, _I]),
    "sfa_mla_decode": (_I, [_P, _P, _I, _I, _I, _F, _P, _P, _P, _SZ, _P, _P]),
    "sfa_mla_decode_pool": (_I, [_P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _F, _P, _P, _P, _SZ,
                                 _P, _P]),
    "dsa_group_step": (_I, [_P, _P, _P, _P, _P]),
    "dsa_group_step_host": (_I, [_P, _P, _P, _P, _P, _P, _P]),
}

EXPORTS = tuple(_SIGS)

TS_MAX_LAYERS = 16
DSA_POLICY_FIFO = 0
DSA_POLICY_REUSE = 1
DSA_POLICY_LRU = 2
DSA_LAYOUT_SELECTION = 0
DSA_LAYOUT_STAGED = 1


class DsaGroup(ctypes.Structure):
    """The dsa_group descriptor of dsakv.h, field for field."""
    _fields_ = [
        ("B", _I), ("layers", _I), ("k", _I), ("S", _I), ("W", _I), ("H", _I),
        ("max_ctx", _I),
        ("ctx_stride", _I64),
        ("scale", _F),
        ("ctx_len", _P),
        ("pool", _P), ("pool_tags", _P), ("fifo_ptr", _P),
        ("host_kv", _P),
        ("ids", _P), ("src_map", _P), ("miss_ids", _P), ("miss_pos", _P), ("victim", _P),
        ("install", _P), ("miss_count", _P), ("miss_rows", _P), ("ptr_next", _P),
        ("sel", _P), ("out", _P), ("lse", _P),
        ("topk_ws", _P), ("topk_ws_bytes", _SZ), ("sfa_ws", _P), ("sfa_ws_bytes", _SZ),
        ("err", _P),
        ("main_stream", _P), ("gather_stream", _P), ("side_stream", _P),
        ("sync", _P),
        ("step", ctypes.c_uint32),
        ("policy", _I),
        ("prev_ids", _P),
        ("prev_sel", _P),
        ("layout", _I),
        ("lru_order", _P),
        ("arrived", _P),
        ("layer_streams", _P),
    ]

for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class DsaKvError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def ts_status_string(status: int) -> str:
    return _lib.ts_status_string(int(status)).decode()


status_string = ts_status_string


def ptr(x) -> int | None:
    """Device pointer of a tensor (or an int / None passed through)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def stream_handle(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def check(status: int, what: str = "") -> None:
    if status != TS_OK:
        raise DsaKvError(status, what)


# ---------------------------------------------------------------------------
# Entry points: same names and argument order as include/dsakv.h.
# Pointer arguments take tensors, ints or None; the status code is returned.
# ---------------------------------------------------------------------------

def ts_host_register(host_addr: int, nbytes: int) -> int:
    """Page-lock and map host memory; returns the device-accessible address."""
    dev = ctypes.c_void_p()
    check(_lib.ts_host_register(host_addr, nbytes, ctypes.byref(dev)), "ts_host_register")
    return int(dev.value)


def ts_host_unregister(host_addr: int) -> int:
    return _lib.ts_host_unregister(host_addr)


def ts_host_alloc(nbytes: int) -> tuple[int, int]:
    """Page-locked, device-mapped host memory; returns (host, device) addresses."""
    host = ctypes.c_void_p()
    dev = ctypes.c_void_p()
    check(_lib.ts_host_alloc(nbytes, ctypes.byref(host), ctypes.byref(dev)), "ts_host_alloc")
    return int(host.value), int(dev.value)


def ts_host_free(host_addr: int) -> int:
    return _lib.ts_host_free(host_addr)


def ts_copy(dst, src, nbytes: int, stream=None) -> int:
    return _lib.ts_copy(ptr(dst), ptr(src), nbytes, stream_handle(stream))


def ts_read_error(err, stream=None) -> int:
    """Waits for the stream, returns the error bits and clears the word."""
    bits = ctypes.c_int32(0)
    st = _lib.ts_read_error(ptr(err), ctypes.byref(bits), stream_handle(stream))
    if st not in (TS_OK, TS_ERR_DEVICE_CHECK):
        raise DsaKvError(st, "ts_read_error")
    return int(bits.value)



def ts_set_wait_limit_ns(ns: int) -> None:
    """Limit of every bounded wait inside the attention kernels launched from
    now on (nanoseconds of the GPU's global timer); 0 restores their own."""
    _lib.ts_set_wait_limit_ns(int(ns))

def ts_topk_workspace_size(B: int, max_ctx: int, k: int) -> int:
    return int(_lib.ts_topk_workspace_size(B, max_ctx, k))


def ts_topk(scores, ctx_stride, ctx_len, B, max_ctx, k, ids, ws, ws_bytes, err=None,
            stream=None) -> int:
    return _lib.ts_topk(ptr(scores), ctx_stride, ptr(ctx_len), B, max_ctx, k, ptr(ids),
                        ptr(ws), ws_bytes, ptr(err), stream_handle(stream))


def ts_topk_noalloc(scores, ctx_stride, ctx_len, B, max_ctx, k, ids, err=None,
                    stream=None) -> int:
    """ts_topk with the library's fixed scratch array instead of a caller
    workspace, for callers that cannot allocate device memory."""
    return _lib.ts_topk_noalloc(ptr(scores), ctx_stride, ptr(ctx_len), B, max_ctx, k, ptr(ids),
                                ptr(err), stream_handle(stream))


def dsa_plan(ids, ctx_len, B, k, pool_tags, fifo_ptr, S, W, src_map, miss_ids, miss_pos,
             victim, install, miss_count, miss_rows, ptr_next, err=None, stream=None) -> int:
    return _lib.dsa_plan(ptr(ids), ptr(ctx_len), B, k, ptr(pool_tags), ptr(fifo_ptr), S, W,
                         ptr(src_map), ptr(miss_ids), ptr(miss_pos), ptr(victim), ptr(install),
                         ptr(miss_count), ptr(miss_rows), ptr(ptr_next), ptr(err),
                         stream_handle(stream))


def dsa_plan_reuse(ids, prev_ids, ctx_len, B, k, src_map, miss_ids, miss_pos, miss_count,
                   miss_rows, err=None, stream=None) -> int:
    return _lib.dsa_plan_reuse(ptr(ids), ptr(prev_ids), ptr(ctx_len), B, k, ptr(src_map),
                               ptr(miss_ids), ptr(miss_pos), ptr(miss_count), ptr(miss_rows),
                               ptr(err), stream_handle(stream))


def dsa_plan_lru(ids, ctx_len, B, k, pool_tags, lru_order, P, src_map, miss_ids, miss_pos,
                 victim, install, miss_count, miss_rows, err=None, stream=None) -> int:
    return _lib.dsa_plan_lru(ptr(ids), ptr(ctx_len), B, k, ptr(pool_tags), ptr(lru_order), P,
                             ptr(src_map), ptr(miss_ids), ptr(miss_pos), ptr(victim), ptr(install),
                             ptr(miss_count), ptr(miss_rows), ptr(err), stream_handle(stream))

def dsa_gather_kv(src_map, miss_ids, miss_pos, miss_count, miss_rows, B, k, pool_l, P, host_l,
                  ctx_stride, ctx_len, sel_l, err=None, stream=None) -> int:
    return _lib.dsa_gather_kv(ptr(src_map), ptr(miss_ids), ptr(miss_pos), ptr(miss_count),
                              ptr(miss_rows), B, k, ptr(pool_l), P, ptr(host_l), ctx_stride,
                              ptr(ctx_len), ptr(sel_l), ptr(err), stream_handle(stream))


def dsa_refill_pool(miss_ids, miss_pos, victim, install, miss_count, B, k, sel_l, pool_l, P,
                    update_metadata, pool_tags, fifo_ptr, ptr_next, S, W, err=None,
                    stream=None) -> int:
    return _lib.dsa_refill_pool(ptr(miss_ids), ptr(miss_pos), ptr(victim), ptr(install),
                                ptr(miss_count), B, k, ptr(sel_l), ptr(pool_l), P,
                                int(update_metadata), ptr(pool_tags), ptr(fifo_ptr),
                                ptr(ptr_next), S, W, ptr(err), stream_handle(stream))


def dsa_stage_misses(miss_ids, miss_pos, miss_count, victim, install, B, k, pool_l, P, host_l,
                     ctx_stride, ctx_len, err=None, stream=None) -> int:
    return _lib.dsa_stage_misses(ptr(miss_ids), ptr(miss_pos), ptr(miss_count), ptr(victim),
                                 ptr(install), B, k, ptr(pool_l), P, ptr(host_l), ctx_stride,
                                 ptr(ctx_len), ptr(err), stream_handle(stream))


def dsa_refill_pool_staged(miss_ids, miss_pos, victim, install, miss_count, B, k, pool_l, P,
                           update_metadata, pool_tags, fifo_ptr, ptr_next, S, W, err=None,
                           stream=None) -> int:
    return _lib.dsa_refill_pool_staged(ptr(miss_ids), ptr(miss_pos), ptr(victim), ptr(install),
                                       ptr(miss_count), B, k, ptr(pool_l), P,
                                       int(update_metadata), ptr(pool_tags), ptr(fifo_ptr),
                                       ptr(ptr_next), S, W, ptr(err), stream_handle(stream))


def sfa_workspace_size(B: int, H: int, k: int) -> int:
    return int(_lib.sfa_workspace_size(B, H, k))


def sfa_mla_decode(q, sel_l, B, H, k, scale, out, lse, ws, ws_bytes, err=None,
                   stream=None) -> int:
    return _lib.sfa_mla_decode(ptr(q), ptr(sel_l), B, H, k, float(scale), ptr(out), ptr(lse),
                               ptr(ws), ws_bytes, ptr(err), stream_handle(stream))


def sfa_mla_decode_pool(q, pool_l, P, src_map, miss_ids, miss_pos, miss_count, miss_rows, B, H,
                        k, scale, out, lse, ws, ws_bytes, err=None, stream=None) -> int:
    return _lib.sfa_mla_decode_pool(ptr(q), ptr(pool_l), P, ptr(src_map), ptr(miss_ids),
                                    ptr(miss_pos), ptr(miss_count), ptr(miss_rows), B, H, k,
                                    float(scale), ptr(out), ptr(lse), ptr(ws), ws_bytes, ptr(err),
                                    stream_handle(stream))


def dsa_group_step(group: DsaGroup, scores, q, ids=None, timing=None) -> int:
    """One decode step of the group; `timing` is None or a ctypes array of
    2 * (3 + 2 * layers) event handles."""
    return _lib.dsa_group_step(ctypes.byref(group), ptr(scores), ptr(q), ptr(ids),
                               None if timing is None else ctypes.cast(timing, _P))


def dsa_group_step_host(group: DsaGroup, scores_h, q_h, out_h, scores_d, q_d,
                        timing=None) -> int:
    """One decode step with the inputs and the output in page-locked host
    memory (device-accessible addresses), copied inside the step."""
    return _lib.dsa_group_step_host(ctypes.byref(group), ptr(scores_h), ptr(q_h), ptr(out_h),
                                    ptr(scores_d), ptr(q_d),
                                    None if timing is None else ctypes.cast(timing, _P))
