"""The base design's adjacent-step reuse ([GLM] §2.1 GatherSelectionKvCache and
§2.2): the device keeps only the previous step's selection (k rows, in the
order of the previous step's ids); a token of the current top-k that the
previous step also selected is served from that buffer, every other token is
read from host memory. After the step, the current selection becomes the
buffer the next step reuses.

plan_reuse states it for one request in the same src_map / miss-list form as
DsaPlan (oracle/plan.py): a hit holds the token's position in the previous
step's ids (the row of the previous selection buffer), a miss of token t is
-1 - t, and the misses are listed once each, ascending, with their first
position. Reading taken where the page is silent: prev_ids entries below 0
are empty positions (before the first step), which no token matches.
"""
from dataclasses import dataclass

import numpy as np


@dataclass
class ReusePlan:
    src_map: np.ndarray   # int32 [k]
    miss_ids: np.ndarray  # int32 [M], ascending, unique
    miss_pos: np.ndarray  # int32 [M], first position of each miss in ids

    @property
    def miss_count(self) -> int:
        return int(self.miss_ids.size)

    @property
    def miss_rows(self) -> int:
        return int(np.sum(self.src_map < 0))


def plan_reuse(ids, prev_ids, ctx_len: int) -> ReusePlan:
    ids = [int(t) for t in ids]
    where = {}
    for j, t in enumerate(int(t) for t in prev_ids):
        if t >= 0:
            where.setdefault(t, j)          # the previous selection's row of token t
    src_map = np.empty(len(ids), dtype=np.int32)
    first_pos = {}
    for j, t in enumerate(ids):
        if not 0 <= t < ctx_len:
            raise ValueError(f"token id {t} outside [0, {ctx_len})")
        if t in where:
            src_map[j] = where[t]
        else:
            src_map[j] = -1 - t
            first_pos.setdefault(t, j)
    miss_ids = sorted(first_pos)
    return ReusePlan(src_map, np.array(miss_ids, dtype=np.int32),
                     np.array([first_pos[t] for t in miss_ids], dtype=np.int32))
