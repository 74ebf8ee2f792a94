"""A fully associative LRU device pool ([GLM] §3: before the set-associative
FIFO, the pages built an 8192-entry device pool managed by LRU and measured
its hit rate on the same Top-K traces as the previous-step reuse). Used here
for the hit-rate comparison of pool policies only; the device path implements
the set-associative FIFO the pages adopted (§4.3).

Readings taken where the page is silent: one step's selection is looked up
as a whole (the hits are the selected tokens resident before the step); the
hits are touched first, in position order, then the misses are installed in
ascending id, each replacing the least recently used entry (an empty entry
first); a step with more misses than entries keeps the last installed ones.
"""
from collections import OrderedDict


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
