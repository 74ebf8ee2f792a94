"""DsaPlan: one shared plan per IndexShare group.

[GLM] §4.2 and §5: once per group, the planner takes the shared top-k ids and
the pool's metadata and records, for every position, whether its row comes
from the device pool or from host memory; it also emits a compact,
deduplicated list of the misses and the slot each miss will replace.
[GLM] §4.3: the pool is set-associative. A token id maps to exactly one set
and may sit in any way of it. Each set keeps one FIFO pointer that advances
once per newly installed entry; hits do not move it; the slot under the
pointer is the one replaced (round-robin, which equals FIFO in install
order). One counter per set: `lru_counter` has shape (batch, pool_size/16).

Readings taken where the page is silent (each listed in the design notes):
  * the set of token t is t mod S;
  * misses are installed in ascending token id;
  * more than W misses in one set in one step: the result is that of
    installing them one by one, so only the last W stay, and the pointer
    advances by the number of misses (mod W);
  * a hit slot is not protected from eviction in the same step (plain FIFO);
    the layer reads it before its own refill runs ([GLM] §4.4);
  * a repeated id is classified once and listed once as a miss, at its first
    position (the page's deduplication of misses, §3 and §4.2);
  * src_map encodes a hit as its slot (>= 0) and a miss of token t as -1 - t.
"""
from dataclasses import dataclass

import numpy as np


@dataclass
class Plan:
    src_map: np.ndarray     # int32 [k]
    miss_ids: np.ndarray    # int32 [M], ascending, unique
    miss_pos: np.ndarray    # int32 [M], first position of each miss in ids
    victim: np.ndarray      # int32 [M], slot each miss replaces
    install: np.ndarray     # bool  [M], miss still resident after the step
    ptr_next: np.ndarray    # int32 [S]

    @property
    def miss_count(self) -> int:
        return int(self.miss_ids.size)

    @property
    def install_code(self) -> np.ndarray:
        """uint8 [M], when each miss may be written into its victim slot:
        0 not installed; 1 the slot is read by no position of this step, so
        the row may go in as soon as it arrives; 2 the slot is read as a hit
        in this step, so the row goes in only after the layer's hits are read
        ([GLM] §4.4: each layer reads its rows before its own refill)."""
        hit_slots = {int(s) for s in self.src_map if s >= 0}
        return np.asarray([0 if not keep else 2 if int(v) in hit_slots else 1
                           for v, keep in zip(self.victim, self.install)], dtype=np.uint8)

    @property
    def miss_rows(self) -> int:
        """Positions that miss, a repeated missed id counted at each position."""
        return int(np.sum((self.src_map < 0) & (self.src_map != np.iinfo(np.int32).min)))


def dsa_plan(ids, ctx_len: int, tags, fifo_ptr, S: int, W: int) -> Plan:
    ids = [int(t) for t in ids]
    tags = [int(t) for t in tags]
    ptr = [int(p) for p in fifo_ptr]
    if len(tags) != S * W or len(ptr) != S:
        raise ValueError("pool metadata shape")
    if any(not 0 <= p < W for p in ptr):
        raise ValueError("FIFO pointer out of range")

    # 1. classify every position against the tags of its set
    src_map = np.empty(len(ids), dtype=np.int32)
    first_pos = {}
    for j, t in enumerate(ids):
        if not 0 <= t < ctx_len:
            raise ValueError(f"token id {t} outside [0, {ctx_len})")
        s = t % S
        way = None
        for w in range(W):              # lowest matching way
            if tags[s * W + w] == t:
                way = w
                break
        if way is not None:
            src_map[j] = s * W + way
        else:
            src_map[j] = -1 - t
            first_pos.setdefault(t, j)

    # 2. compact, deduplicated miss list in ascending id
    miss_ids = sorted(first_pos)
    miss_pos = [first_pos[t] for t in miss_ids]

    # 3. replacement slots: rank of each miss among its set's misses
    count = [0] * S
    rank = []
    for t in miss_ids:
        s = t % S
        rank.append(count[s])
        count[s] += 1
    victim, install = [], []
    for t, r in zip(miss_ids, rank):
        s = t % S
        victim.append(s * W + (ptr[s] + r) % W)
        install.append(r >= count[s] - W)
    ptr_next = [(ptr[s] + count[s]) % W for s in range(S)]

    return Plan(src_map=src_map,
                miss_ids=np.asarray(miss_ids, dtype=np.int32),
                miss_pos=np.asarray(miss_pos, dtype=np.int32),
                victim=np.asarray(victim, dtype=np.int32),
                install=np.asarray(install, dtype=bool),
                ptr_next=np.asarray(ptr_next, dtype=np.int32))
