"""CPU oracle of the decode-step KV path. TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of what the path computes, in
numpy with float64 for the attention. It exists to check the CUDA path, which
it shares no code with: only `tests/`, `__graft_entry__.smoke()` and the CPU
baseline leg of `bench.py` may import it. The product path never calls it and
never falls back to it.

Sources (the pages the method is described on):
  [GLM] GLM-5.2 shared-Indexer KV Cache Offload (CANN cann-recipes-infer):
        §2.1 sparse-attention data loading, §2.2 adjacent-step reuse,
        §3 larger device pool, §4.1 IndexShare groups, §4.2 shared planning,
        §4.3 set-associative FIFO, §4.4 SFA first / refill later,
        §5 and §5.1 the DsaPlan / DsaServe / DsaInstall operators.
  [TS]  TokenSpeed engine audit, MLA kernel section: the latent row
        (512 latent + 64 rope) is stored once and serves as both K and V.

Every function is pinned by `tests/test_oracle_*.py` against something other
than itself (brute force, a sequential FIFO simulator, closed forms,
invariants); no function here is "parity unpinned".
"""
from .topk import topk_ids
from .plan import Plan, dsa_plan
from .reuse import ReusePlan, plan_reuse
from .lru import LruPool, LruSlots
from .serve import dsa_serve
from .install import dsa_install, metadata_update
from .sfa import bf16_bits_to_f64, round_to_bf16_bits, sfa_decode
from .step import RequestState, decode_step, init_state
