"""The gather's per-request arrival counts (csrc/copy.cu: RowPipe's row tags,
publish and store schedule, and count_arrivals, the counting warp), restated
on the CPU. A pipe warp pushes rows tagged with their (layer, request) index
into a ring of kTagRing entries; its stores retire in order, and every fourth
store (or a layer's end, or the finish) makes the rows whose stores are done
count -- either the warp itself adds them up (self_count), or it publishes
how many rows are stored and the CTA's counting warp, sweeping at its own
pace, adds runs of rows of one request. Checked over random row streams and
interleavings: every request's count ends at its number of rows, no count
ever runs ahead of the rows actually stored, and a ring entry is never
overwritten before the counting warp has read it (the pipe's wait on the
consumed word is what guarantees that with the counting warp; with
self_count the ring is read before the pipe gets that far ahead)."""
import numpy as np

kPipeSlots = 12
kPipeLag = 2
kPipeAhead = kPipeSlots - kPipeLag   # loads in flight per warp
kPipeRetire = 4
kTagRing = 48
kNoTag = 0xFFFF


class Pipe:
    """One pipe warp's bookkeeping, in the order the device code runs it."""

    def __init__(self, self_count, counts):
        self.self_count = self_count
        self.counts = counts        # the device's arrival words (shared)
        self.tags = [None] * kTagRing
        self.log = []               # every pushed row's tag (the check's record, not the device's)
        self.issued = self.stored = self.done = 0   # done: stores known complete
        self.published = 0
        self.consumed = 0           # the counting warp's progress (self_count: unused)
        self.finished = False

    def _runs_add(self, lo, hi):
        tag, run = self.tags[lo % kTagRing], 0
        for i in range(lo, hi):
            t = self.tags[i % kTagRing]
            if t != tag:
                if tag != kNoTag:
                    self.counts[tag] += run
                tag, run = t, 0
            run += 1
        if tag != kNoTag and hi > lo:
            self.counts[tag] += run

    def publish(self, n):
        # the caller waited for the store groups below n
        assert n <= self.done
        if n <= self.published:
            return
        if self.self_count:
            self._runs_add(self.published, n)
        self.published = n

    def store_one(self):
        self.stored += 1
        # store groups complete in order; at least those kPipeRetire back
        # are complete once the pipe waits for them
        if self.stored % 4 == 0 and self.stored > kPipeRetire:
            self.done = max(self.done, self.stored - kPipeRetire)
            self.publish(self.stored - kPipeRetire)

    def push(self, tag, counter):
        while self.stored + kPipeAhead <= self.issued:
            self.store_one()
        if not self.self_count:
            # the tag entry this row takes must have been read: wait for the
            # counting warp (here: let it sweep until it has)
            while self.issued - self.consumed >= kTagRing:
                assert counter.sweep(), "the counting warp made no progress"
        assert self.self_count or self.issued - self.consumed < kTagRing
        # with self_count the entry's old row was counted already
        assert self.issued - self.published < kTagRing
        self.tags[self.issued % kTagRing] = tag
        self.log.append(tag)
        self.issued += 1

    def finish(self):
        while self.stored < self.issued:
            self.store_one()
        self.done = self.stored      # every store group complete
        self.publish(self.stored)
        self.finished = True


class Counter:
    """The counting warp: lane w follows pipe w's published rows."""

    def __init__(self, pipes, counts):
        self.pipes = pipes
        self.counts = counts
        self.seen = [0] * len(pipes)

    def sweep(self):
        progress = False
        for w, p in enumerate(self.pipes):
            if p.self_count:
                continue
            hi = p.published
            if hi > self.seen[w]:
                p._runs_add(self.seen[w], hi)
                self.seen[w] = hi
                p.consumed = hi
                progress = True
        return progress


def run(rng, self_count):
    B = int(rng.integers(1, 12))
    layers = int(rng.integers(1, 5))
    misses = rng.integers(0, 40, size=B)
    nwarps = int(rng.integers(1, 6))
    counts = {}
    for l in range(layers):
        for b in range(B):
            counts[l * B + b] = 0
    # rows in ticket order (layer-major, request order), dealt to warps in
    # tickets of a few rows at random
    rows = [l * B + b for l in range(layers) for b in range(B) for _ in range(int(misses[b]))]
    pipes = [Pipe(self_count, counts) for _ in range(nwarps)]
    counter = Counter(pipes, counts)
    i = 0
    while i < len(rows):
        w = int(rng.integers(0, nwarps))
        n = int(rng.integers(1, 17))
        for tag in rows[i:i + n]:
            pipes[w].push(tag, counter)
        i += n
        if rng.random() < 0.3:
            counter.sweep()
        # no count runs ahead of the rows whose stores are done
        for t, c in counts.items():
            assert c <= sum(p.log[:p.done].count(t) for p in pipes), t
    for p in pipes:
        p.finish()
    while counter.sweep():
        pass
    for l in range(layers):
        for b in range(B):
            assert counts[l * B + b] == int(misses[b]), (l, b)


def test_counts_reach_each_request_rows_with_pipe_releases():
    rng = np.random.default_rng(5)
    for _ in range(60):
        run(rng, self_count=True)


def test_counts_reach_each_request_rows_with_counting_warp():
    rng = np.random.default_rng(6)
    for _ in range(60):
        run(rng, self_count=False)


def test_ring_bound_with_pipe_releases():
    # with self_count the pipe never needs the consumed word: between a row's
    # push and its count at most kPipeAhead rows are in flight, kPipeRetire
    # stores wait to retire and 3 more pass before the next publish
    assert kPipeAhead + kPipeRetire + 3 < kTagRing
