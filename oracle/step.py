"""One decode step of one request through an IndexShare group, in the pages'
order, sequentially.

[GLM] §4.1: one layer runs the indexer and the next layers of the group reuse
its top-k. [GLM] §4.2: the plan is made once for the group. [GLM] §4.4 and
§5.1: each layer serves its selected rows, runs SFA on them, then refills its
own pool from the misses; the metadata update comes at the group's last layer.
"""
from dataclasses import dataclass

import numpy as np

from .install import dsa_install, metadata_update
from .plan import dsa_plan
from .serve import dsa_serve
from .sfa import sfa_decode
from .topk import topk_ids


@dataclass
class RequestState:
    pool: np.ndarray      # uint16 [layers][P][576], the device pool's rows
    tags: np.ndarray      # int32 [P], token id held by each slot, -1 = empty
    fifo_ptr: np.ndarray  # int32 [S]


def init_state(layers: int, S: int, W: int, D: int = 576) -> RequestState:
    """A cold pool: every slot empty, every pointer at way 0."""
    return RequestState(pool=np.zeros((layers, S * W, D), dtype=np.uint16),
                        tags=np.full(S * W, -1, dtype=np.int32),
                        fifo_ptr=np.zeros(S, dtype=np.int32))


def decode_step(state: RequestState, scores, ctx_len: int, k: int, S: int, W: int,
                host_rows, q_bits, scale: float, with_sfa: bool = True):
    """host_rows[l]: uint16 [>= ctx_len][576]; q_bits[l]: uint16 [H][576].
    Mutates `state`; returns a dict of everything the step produced."""
    layers = state.pool.shape[0]
    ids = topk_ids(scores, ctx_len, k)
    plan = dsa_plan(ids, ctx_len, state.tags, state.fifo_ptr, S, W)
    sel, out, lse = [], [], []
    for l in range(layers):
        rows = dsa_serve(plan.src_map, state.pool[l], host_rows[l], ctx_len)
        sel.append(rows)
        if with_sfa:
            o, z = sfa_decode(q_bits[l], rows, scale)
            out.append(o)
            lse.append(z)
        dsa_install(state.pool[l], plan, host_rows[l])
    metadata_update(state.tags, state.fifo_ptr, plan)
    return {"ids": ids, "plan": plan, "sel": sel, "out": out, "lse": lse}
