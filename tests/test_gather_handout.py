"""The gather's dynamic miss hand-out (csrc/copy.cu, gather_misses_dynamic),
restated on the CPU: warps take tickets from one counter in any interleaving;
every (layer, request, miss) is moved exactly once, every index stays inside
the plan's arrays, every warp counts itself out of every layer exactly once and
in layer order, and a layer is only counted out by a warp after all of that
warp's rows of it were pushed."""
import numpy as np


def prefix_of(counts, k):
    c = np.clip(np.asarray(counts), 0, k)
    return np.concatenate([[0], np.cumsum(c)]).astype(np.int64)


def request_of(prefix, B, g):
    lo, hi = 0, B
    while hi - lo > 1:
        mid = (lo + hi) >> 1
        if prefix[mid] <= g:
            lo = mid
        else:
            hi = mid
    return lo


ROWS = 16   # misses per ticket (kTicketRows)


def simulate(counts, k, layers, nwarps, rng):
    B = len(counts)
    prefix = prefix_of(counts, k)
    total = int(prefix[B])
    nb = (total + ROWS - 1) // ROWS
    end = nb * layers
    ticket = 0
    moved = []
    events = {w: [] for w in range(nwarps)}      # per warp: ("row", l) / ("out", l)
    cur = {w: 0 for w in range(nwarps)}
    # each warp: its current ticket and the prefetched next one
    state = {}
    for w in range(nwarps):
        state[w] = ticket
        ticket += 1
    live = set(range(nwarps))
    while live:
        w = int(rng.choice(sorted(live)))
        t = state[w]
        if t >= end:
            for l in range(cur[w], layers):      # the rest, then the finish
                events[w].append(("out", l))
            live.discard(w)
            continue
        nxt = ticket                             # prefetch
        ticket += 1
        l = t // nb
        while cur[w] < l:
            events[w].append(("out", cur[w]))
            cur[w] += 1
        for lane in range(32):
            g = (t % nb) * ROWS + lane
            if lane < ROWS and g < total:
                b = request_of(prefix, B, g)
                i = g - int(prefix[b])
                assert 0 <= b < B and 0 <= i < min(max(counts[b], 0), k)
                moved.append((l, b, i))
                events[w].append(("row", l))
        state[w] = nxt
    return moved, events


def test_every_miss_moved_once_and_layers_counted_out_in_order():
    rng = np.random.default_rng(9)
    for trial in range(15):
        B = int(rng.integers(1, 40))
        k = int(rng.choice([64, 256, 512]))
        counts = rng.integers(0, k + 1, size=B)
        if trial % 7 == 0:
            counts[:] = 0
        counts[0] = counts[0] if trial % 5 else k + 7   # a corrupt count is clipped to k
        layers = int(rng.integers(1, 5))
        nwarps = int(rng.integers(1, 40))
        moved, events = simulate(list(counts), k, layers, nwarps, rng)
        want = sorted((l, b, i) for l in range(layers) for b in range(B)
                      for i in range(min(max(int(counts[b]), 0), k)))
        assert sorted(moved) == want
        for w, ev in events.items():
            outs = [l for kind, l in ev if kind == "out"]
            assert outs == list(range(layers))          # each layer once, in order
            for idx, (kind, l) in enumerate(ev):
                if kind == "row":                       # pushed before its layer's count-out
                    assert ("out", l) not in ev[:idx]
