"""The group step's stream schedule (csrc/step.cu, enqueue_step), restated on
the CPU and run under random interleavings of its streams.

Each step enqueues, in the order the native call does, waits and writes of
the ordering words and kernels on the main, gather and side streams, and,
with layer streams, each layer's attention on a stream of its own. The model
runs several steps at once: any stream whose next operation can run may go
next (a wait runs once its word has reached the value; the gather runs layer
by layer and writes its per-layer words as it goes; a streamed attention's
body runs once the gather has stored its layer's rows, the in-kernel wait).
Checked, for every layout, policy, host-I/O mix and stream arrangement:

- every wait ends: no interleaving leaves a stream blocked for good;
- the words holding step numbers never decrease, and a wait on a per-step
  count is never met by the count of an earlier step;
- every pair of accesses to one buffer that must not overlap (a write and
  any other access, in two kernels on two streams) is ordered: the earlier
  access happens before the later through stream order, words (a wait and
  the write it saw) and the gather's device-side layer events.

The buffers follow the header's hazards: the plan's outputs, the ids, the
pool's tags, the pool's slots (hits read by the attention, code-2 installs by
the refill, code-1 installs by the next steps' gathers), the staged rows or
selection buffers, the arrival counts, the queries' staging halves, the
attention's workspaces and outputs."""
import random
import sys
from collections import defaultdict, namedtuple

import pytest

Cfg = namedtuple("Cfg", "layout policy streamed lanes L")

Wait = namedtuple("Wait", "word value same_step")
Write = namedtuple("Write", "word value")
Kernel = namedtuple("Kernel", "name step layer phases")
# one phase of a kernel: accesses [(buffer, "R" / "W")], device writes of
# words [(word, value)], and an optional in-kernel wait (the gather's layer)
Phase = namedtuple("Phase", "acc dev needs")

NCTAS = 3  # attention CTAs of one layer (any positive count)
GIVE_UP = False  # streamed attention CTAs whose wait for their rows ran out


def attention_ops(c, s, l, io):
    """One layer's attention: the chunk kernel (its CTAs count themselves in,
    then read their rows and write the partials) and the merge kernel."""
    ws = ("ws", l if c.lanes else 0)
    rows = [("plan", "R"), (("q", s & 1, l) if io else ("qdev", l), "R"), (ws, "W")]
    if c.layout == "staged":
        rows += [(("stage", l), "R"), (("slots", l), "R")]
        if c.streamed:
            rows += [(("counts", l), "R")]
    else:
        rows += [(("sel", l, s & 1 if c.policy == "reuse" else 0), "R")]
    start = Phase([], [(("lstarted", l), NCTAS)] if c.streamed else [], None)
    body = Phase(rows, [], ("layer", l) if c.streamed and not GIVE_UP else None)
    chunk = Kernel("chunk", s, l, [start, body])
    merge = Kernel("merge", s, l, [Phase([(ws, "R"), (("out", l), "W")], [], None)])
    return [chunk, merge]


def gather_kernel(c, s):
    """One launch for every layer: the CTAs start (the started word), then
    layer by layer the rows arrive and the layer's words are written."""
    L = c.L
    phases = [Phase([("plan", "R")], [("started", s)] if c.streamed else [], None)]
    for l in range(L):
        acc = [("plan", "R")]
        if c.layout == "staged":
            acc += [(("stage", l), "W"), (("c1", l), "W")]
            if c.streamed:
                acc += [(("counts", l), "W")]
        elif c.policy == "reuse":
            acc += [(("sel", l, (s - 1) & 1), "R"), (("sel", l, s & 1), "W")]
        else:
            acc += [(("slots", l), "R"), (("sel", l, 0), "W")]
        phases.append(Phase(acc, [(("gathered", l), s), ("layer_done", (s, l))], None))
    return Kernel("gather", s, -1, phases)


def enqueue(c, s, io):
    """Step s's operations per stream, in the order enqueue_step issues them."""
    L = c.L
    staged = c.layout == "staged"
    refills = c.policy == "fifo"
    ops = defaultdict(list)
    m, gs, side = "main", "gather", "side"
    sL = s * L

    def a(l):
        return f"layer{l}" if c.lanes else m

    if c.streamed:
        ops[m].append(Kernel("memset", s, -1, [Phase(
            [(("counts", l), "W") for l in range(L)], [("started", 0)]
            + [(("lstarted", l), 0) for l in range(L)], None)]))
    if io:
        ops[m].append(Kernel("scores_copy", s, -1, [Phase([("scores", "W")], [], None)]))
    ids_w = ("ids", s & 1 if c.policy == "reuse" else 0)
    ops[m].append(Kernel("topk", s, -1, [Phase([("scores", "R"), (ids_w, "W")], [], None)]))
    ops[m].append(Wait("refilled", s - 1, False))
    plan_acc = [(ids_w, "R"), ("plan", "W")]
    if c.policy == "reuse":
        plan_acc += [(("ids", (s - 1) & 1), "R")]
    else:
        plan_acc += [("tags", "W" if c.policy == "lru" else "R")]
    ops[m].append(Kernel("plan", s, -1, [Phase(plan_acc, [], None)]))
    ops[m].append(Write("planned", s))
    ops[gs].append(Wait("planned", s, False))
    if not c.lanes and s > 1:
        ops[m].append(Wait("outcopied", sL - 1, False))
    ops[gs].append(gather_kernel(c, s))
    if io:
        ops[side].append(Wait("planned", s, False))
        for l in range(L):
            ops[side].append(Kernel("qcopy", s, l, [Phase([(("q", s & 1, l), "W")], [], None)]))
            ops[side].append(Write("qcopied", sL + l))
    for l in range(L):
        st = a(l)
        if c.streamed:
            if l == 0 or c.lanes:
                ops[st].append(Wait("started", s, True))
        else:
            ops[st].append(Wait(("gathered", l), s, False))
        if c.lanes and l > 0:
            ops[st].append(Wait(("lstarted", l - 1), NCTAS, True))
        if c.lanes and s > 1:
            ops[st].append(Wait("outcopied", sL - L + l, False))
        if io:
            ops[st].append(Wait("qcopied", sL + l, False))
        ops[st] += attention_ops(c, s, l, io)
        ops[st].append(Write(("attended", l), s))
        if not (io or c.lanes):
            ops[st].append(Write("outcopied", sL + l))
        if refills:
            ops[side].append(Wait(("attended", l) if staged else ("gathered", l), s, False))
            if staged:
                ops[side].append(Wait(("gathered", l), s, False))
            acc = [("plan", "R"), (("slots", l), "W")]
            acc += [(("stage", l), "R")] if staged else [(("sel", l, 0), "R")]
            if l == L - 1:
                acc += [("tags", "W")]
            ops[side].append(Kernel("refill", s, l, [Phase(acc, [], None)]))
            if l == L - 1:
                ops[side].append(Write("refilled", s))
        if io:
            ops[side].append(Wait(("attended", l), s, False))
            ops[side].append(Kernel("outcopy", s, l, [Phase([(("out", l), "R")], [], None)]))
            ops[side].append(Write("outcopied", sL + l))
    if c.lanes:
        for l in range(L):
            ops[m].append(Wait(("attended", l), s, False))
        if not io:
            ops[m].append(Write("outcopied", sL + L - 1))
    if not refills:
        ops[m].append(Write("refilled", s))
    return ops


# words that hold step numbers (or step * layers + layer) and only grow
SEQ_WORDS = ("planned", "refilled", "gathered", "attended", "qcopied", "outcopied")


def seq_word(w):
    return (w if isinstance(w, str) else w[0]) in SEQ_WORDS


class Run:
    """The streams' operations executed one at a time in a random order."""

    def __init__(self, c, ios, rng):
        self.c, self.rng = c, rng
        self.queues = defaultdict(list)
        for s, io in enumerate(ios, start=1):
            for st, ops in enqueue(c, s, io).items():
                self.queues[st] += [(s, op) for op in ops]
        self.pos = {st: 0 for st in self.queues}
        self.phase = {st: 0 for st in self.queues}   # next phase of the head kernel
        self.word = defaultdict(int)
        self.writer = {}        # word -> (event, step) of its last write
        self.events = []        # happens-before sets, by event id
        self.last = {}          # stream -> its last event
        self.layer_event = {}   # (step, layer) -> the gather's event
        self.accesses = []      # (buffer, kind, step, order key, event)

    def head(self, st):
        q = self.queues[st]
        return q[self.pos[st]] if self.pos[st] < len(q) else None

    def runnable(self, st):
        h = self.head(st)
        if h is None:
            return False
        s, op = h
        if isinstance(op, Wait):
            return self.word[op.word] >= op.value
        if isinstance(op, Kernel):
            needs = op.phases[self.phase[st]].needs
            return needs is None or (s, needs[1]) in self.layer_event
        return True

    def new_event(self, st, extra=()):
        hb = set()
        if st in self.last:
            e = self.last[st]
            hb |= self.events[e] | {e}
        for e in extra:
            hb |= self.events[e] | {e}
        self.events.append(hb)
        ev = len(self.events) - 1
        self.last[st] = ev
        return ev

    def write_word(self, w, v, ev, s):
        if seq_word(w):
            assert v >= self.word[w], f"word {w} would drop from {self.word[w]} to {v}"
        self.word[w] = v
        self.writer[w] = (ev, s)

    def step_one(self, st):
        s, op = self.head(st)
        if isinstance(op, Wait):
            if op.same_step:
                # a count (or a word that each step zeroes) must be this
                # step's when the wait sees it reach the value
                assert self.writer[op.word][1] == s, \
                    f"step {s} saw step {self.writer[op.word][1]}'s {op.word}"
            extra = [self.writer[op.word][0]] if op.word in self.writer else []
            self.new_event(st, extra)
            self.pos[st] += 1
        elif isinstance(op, Write):
            ev = self.new_event(st)
            self.write_word(op.word, op.value, ev, s)
            self.pos[st] += 1
        else:
            ph = op.phases[self.phase[st]]
            extra = [self.layer_event[(s, ph.needs[1])]] if ph.needs else []
            ev = self.new_event(st, extra)
            for buf, kind in ph.acc:
                self.accesses.append((buf, kind, s, (op.name, op.layer, self.phase[st]), ev))
            for w, v in ph.dev:
                if w == "layer_done":
                    self.layer_event[v] = ev
                else:
                    self.write_word(w, v, ev, s)
            self.phase[st] += 1
            if self.phase[st] == len(op.phases):
                self.phase[st] = 0
                self.pos[st] += 1

    def run(self):
        while True:
            ready = [st for st in self.queues if self.runnable(st)]
            if not ready:
                stuck = {st: self.head(st) for st in self.queues if self.head(st) is not None}
                assert not stuck, f"blocked for good: {stuck}"
                return
            self.step_one(self.rng.choice(sorted(ready)))


# the order the design requires between two accesses of one buffer: step by
# step; in a step the top-k, plan and the gather's start first, then layer by
# layer its queries, the gather's rows, the attention, its merge, the refill
# and the output's copy
ORDER = {"memset": 0, "scores_copy": 0, "topk": 1, "plan": 2, "qcopy": 3, "gather": 4,
         "chunk": 5, "merge": 6, "refill": 7, "outcopy": 8}


def key(acc):
    buf, kind, s, (name, layer, phase), ev = acc
    if name == "gather":
        layer = phase - 1  # phase 0: the CTAs start; phase l + 1: layer l
    if layer < 0:
        return (s, 0, ORDER[name], 0, phase)
    return (s, 1, layer, ORDER[name], phase)


def conflicts(x, y):
    """Two accesses to one buffer that may not overlap (one writes it). A
    step's code-1 installs go to slots that no hit of that step reads, so
    they only meet the slots' other accesses of other steps."""
    if x[0] != y[0] and not ({x[0][0], y[0][0]} == {"slots", "c1"} and x[0][1] == y[0][1]):
        return False
    if "W" not in (x[1], y[1]):
        return False
    if {x[0][0], y[0][0]} == {"slots", "c1"} and x[2] == y[2]:
        return False
    return True


def check_hazards(run):
    acc = sorted(run.accesses, key=key)
    by_buf = defaultdict(list)
    for a in acc:
        b = a[0]
        by_buf[("slots", b[1]) if isinstance(b, tuple) and b[0] in ("slots", "c1") else b].append(a)
    for group in by_buf.values():
        for i, x in enumerate(group):
            for y in group[i + 1:]:
                if x[4] == y[4] or not conflicts(x, y):
                    continue
                assert x[4] in run.events[y[4]], f"unordered: {x[:4]} then {y[:4]}"


CONFIGS = [Cfg("selection", "fifo", False, False, 4), Cfg("selection", "lru", False, False, 4),
           Cfg("selection", "reuse", False, False, 4),
           Cfg("staged", "fifo", False, False, 4), Cfg("staged", "lru", False, False, 4),
           Cfg("staged", "fifo", True, False, 4), Cfg("staged", "lru", True, False, 4),
           Cfg("staged", "fifo", True, True, 4), Cfg("staged", "lru", True, True, 4),
           Cfg("staged", "fifo", True, True, 1), Cfg("staged", "fifo", True, False, 2)]


@pytest.mark.parametrize("c", CONFIGS, ids=lambda c: "-".join(map(str, c)))
def test_every_wait_ends_and_every_hazard_is_ordered(c):
    rng = random.Random(17)
    for trial in range(40):
        steps = 4
        ios = [rng.random() < 0.5 for _ in range(steps)]
        if trial % 4 == 0:
            ios = [False] * steps
        elif trial % 4 == 1:
            ios = [True] * steps
        run = Run(c, ios, rng)
        run.run()
        check_hazards(run)


def plant(monkeypatch, streams, old, new):
    """Replace an operation of the restated schedule on some streams (a
    planted mistake)."""
    orig = enqueue

    def patched(c, s, io):
        ops = orig(c, s, io)
        for st in ops:
            if st in streams:
                ops[st] = [new if op == old(c, s) else op for op in ops[st]]
                ops[st] = [op for op in ops[st] if op is not None]
        return ops
    monkeypatch.setattr(sys.modules[__name__], "enqueue", patched)


def runs(c, n, ios=(False, False, False)):
    for seed in range(n):
        run = Run(c, list(ios), random.Random(seed))
        run.run()
        yield run


def test_a_dropped_wait_is_caught(monkeypatch):
    # the staged refill without its wait for the attention: the refill's
    # code-2 installs may overwrite slots the attention still reads
    c = Cfg("staged", "fifo", True, True, 2)
    plant(monkeypatch, ("side",), lambda c, s: Wait(("attended", 1), s, False), None)
    with pytest.raises(AssertionError, match=r"unordered: \(\('slots', 1\), 'R'"):
        for run in runs(c, 40):
            check_hazards(run)


def stage_hazards(run):
    # the staged rows only: the gather's writes before the refill's reads
    run.accesses = [a for a in run.accesses if a[0][0] == "stage"
                    and (a[3][0], a[1]) in (("gather", "W"), ("refill", "R"))]
    check_hazards(run)


@pytest.mark.parametrize("lanes", [False, True])
def test_refill_reads_staged_rows_after_the_gather_when_the_attention_gave_up(monkeypatch,
                                                                              lanes):
    # an attention whose wait for its rows ran out ends before they are in;
    # the refill, which copies them into victim slots, still waits for them
    # (what the attention itself computed is then undefined, and reported)
    monkeypatch.setattr(sys.modules[__name__], "GIVE_UP", True)
    for run in runs(Cfg("staged", "fifo", True, lanes, 2), 40):
        stage_hazards(run)


def test_refill_without_its_gather_wait_is_caught_when_the_attention_gave_up(monkeypatch):
    monkeypatch.setattr(sys.modules[__name__], "GIVE_UP", True)
    plant(monkeypatch, ("side",), lambda c, s: Wait(("gathered", 1), s, False), None)
    c = Cfg("staged", "fifo", True, True, 2)
    with pytest.raises(AssertionError, match=r"unordered: \(\('stage', 1\), 'W'"):
        for run in runs(c, 60):
            stage_hazards(run)


def test_a_layer_stream_without_its_started_wait_is_caught(monkeypatch):
    # a layer stream that does not wait for this step's gather to run may
    # see the previous step's count of the layer before (same-step check)
    # or read rows the gather has not stored
    c = Cfg("staged", "fifo", True, True, 2)
    plant(monkeypatch, ("layer1",), lambda c, s: Wait("started", s, True), None)
    with pytest.raises(AssertionError, match=r"saw step \d+'s \('lstarted', 0\)"):
        for run in runs(c, 60):
            check_hazards(run)
