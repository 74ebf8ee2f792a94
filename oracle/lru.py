"""A fully associative LRU device pool ([GLM] §3: before the set-associative
FIFO, the pages built an 8192-entry device pool managed by LRU and measured
its hit rate on the same Top-K traces as the previous-step reuse). LruPool
counts hits only (the hit-rate comparison of pool policies); LruSlots is the
same policy with slots, the reference of the device's LRU plan. The pages
adopted the set-associative FIFO (§4.3) because managing the LRU pool cost
too much on their hardware; the device path offers both.

Readings taken where the page is silent: one step's selection is looked up
as a whole (the hits are the selected tokens resident before the step); the
hits are touched first, in position order, then the misses are installed in
ascending id, each replacing the least recently used entry (an empty entry
first); a step with more misses than entries keeps the last installed ones.
"""
from collections import OrderedDict

import numpy as np


class LruPool:
    def __init__(self, entries: int):
        self.entries = entries
        self.order = OrderedDict()  # token -> None, least recently used first

    def step(self, ids) -> int:
        """Serve one step's selected ids; returns the number of hits."""
        ids = [int(t) for t in ids]
        resident = set(self.order)
        hits = [t for t in ids if t in resident]
        for t in hits:                      # touch the hits
            self.order.move_to_end(t)
        misses = sorted(set(t for t in ids if t not in resident))
        for t in misses:                    # install, evicting the LRU entry
            if len(self.order) >= self.entries:
                self.order.popitem(last=False)
            self.order[t] = None
        return len(hits)


class LruSlots:
    """The same LRU pool with slots, so that a device pool's state can be
    compared with it entry by entry: tags[P] holds the token of each slot (-1
    empty), last_use[P] the time of the slot's last use, clock the time of
    the latest use. Time counts uses one by one: each touched hit, then each
    installed miss, takes the next tick.

    Readings taken where the page is silent (besides those of LruPool): an
    empty slot is taken before any resident entry is evicted, lowest index
    first; when a step misses more tokens than there are slots its hits do
    not hold, a miss may evict a miss installed earlier in the same step (that
    earlier miss is then not installed, as in the FIFO pool's overflow)."""

    def __init__(self, entries: int):
        self.tags = [-1] * entries
        self.last_use = [0] * entries
        self.clock = 0

    def plan(self, ids, ctx_len: int):
        """Plan one step's selected ids and apply it to the metadata; returns
        a Plan (src_map, ascending deduplicated miss list with first positions,
        victim slots, install flags; ptr_next empty)."""
        from .plan import Plan
        ids = [int(t) for t in ids]
        slot_of = {t: s for s, t in enumerate(self.tags) if t >= 0}
        src_map = np.empty(len(ids), dtype=np.int32)
        first_pos = {}
        for j, t in enumerate(ids):
            if not 0 <= t < ctx_len:
                raise ValueError(f"token id {t} outside [0, {ctx_len})")
            if t in slot_of:
                src_map[j] = slot_of[t]
            else:
                src_map[j] = -1 - t
                first_pos.setdefault(t, j)
        # touch the hits, in position order
        for j, t in enumerate(ids):
            if src_map[j] >= 0:
                self.clock += 1
                self.last_use[int(src_map[j])] = self.clock
        # install the misses in ascending id, each into the least recently
        # used slot (an empty one first, lowest index first). Each install
        # becomes the most recent use, so the victims are the slots in
        # least-recently-used order, one per miss, starting over from the
        # first when a step misses more tokens than there are slots
        P = len(self.tags)
        order = sorted(range(P), key=lambda s: (self.tags[s] >= 0, self.last_use[s], s))
        miss_ids = sorted(first_pos)
        victim, owner = [], {}
        for i, t in enumerate(miss_ids):
            v = order[i % P]
            victim.append(v)
            owner[v] = i
            self.tags[v] = t
            self.clock += 1
            self.last_use[v] = self.clock
        install = [owner.get(v) == i for i, v in enumerate(victim)]
        return Plan(src_map=src_map,
                    miss_ids=np.asarray(miss_ids, dtype=np.int32),
                    miss_pos=np.asarray([first_pos[t] for t in miss_ids], dtype=np.int32),
                    victim=np.asarray(victim, dtype=np.int32),
                    install=np.asarray(install, dtype=bool),
                    ptr_next=np.zeros(0, dtype=np.int32))
