"""GB300-native decode-step KV path of DeepSeek-Sparse-Attention-style serving
with host-offloaded KV and a set-associative FIFO device pool.

The compute lives in libdsakv.so (CUDA C++ for sm_103a, C ABI in
include/dsakv.h). This package holds its build script (`build`), its ctypes
binding (`_abi`, same entry-point names as the header) and the per-step
schedule over PyTorch-owned memory and streams (`runtime`). The binding loads
lazily, so `python -m decode_dsa_kv_gb300.build` works before the library
exists; any use of an entry point without the library raises ImportError.
"""
import importlib

_ABI_NAMES = {
    "ts_status_string", "ts_host_register", "ts_host_unregister", "ts_host_alloc", "ts_host_free",
    "ts_read_error", "ts_copy", "ts_set_wait_limit_ns",
    "ts_topk_workspace_size", "ts_topk", "ts_topk_noalloc", "dsa_plan", "dsa_plan_reuse", "dsa_plan_lru",
    "dsa_gather_kv", "dsa_stage_misses", "dsa_refill_pool", "dsa_refill_pool_staged",
    "sfa_mla_decode_pool",
    "sfa_workspace_size", "sfa_mla_decode", "dsa_group_step", "dsa_group_step_host", "DsaGroup", "DsaKvError", "check", "status_string", "EXPORTS",
    "LIB_PATH",
}
_RUNTIME_NAMES = {"HostKV", "DecodeGroup", "PinnedHost", "StepTiming", "plan_metrics"}


def __getattr__(name):
    if name in _ABI_NAMES:
        return getattr(importlib.import_module("._abi", __name__), name)
    if name in _RUNTIME_NAMES:
        return getattr(importlib.import_module(".runtime", __name__), name)
    raise AttributeError(name)
