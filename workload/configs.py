"""The five seeded synthetic workloads of the decode-step KV path.

Each workload fixes the shapes of one decode step of a 4-layer IndexShare group
(one `full` layer that runs the indexer and three `shared` layers that reuse its
top-k) and the statistics of the indexer scores from step to step. Sizes follow
the GLM-5.2 shared-Indexer KV Cache Offload page (CANN cann-recipes-infer):
top-k 2048 (§2.1), pool 8192 or 16384 entries in sets of 16 ways (§4.3, §6.2),
one FIFO counter per set (§4.3), groups of 4 layers (§4.1). Latent rows hold
576 bf16 values: 512 latent ("nope") + 64 rope, used as both K and V in
absorbed-MLA decode (TokenSpeed engine audit, MLA kernel section).

The score processes stand in for the pages' full-model Top-K traces, which are
not public: adjacent steps' top-k overlap about 60% (§2.2).
"""
from __future__ import annotations

from dataclasses import dataclass, field

D_LATENT = 512          # V / "nope" part of a latent row
D_ROPE = 64
D = D_LATENT + D_ROPE   # 576 values per row
ROW_BYTES = D * 2       # bf16


@dataclass(frozen=True)
class Workload:
    name: str
    index: int              # position in the list below; seed = 1000 + index
    B: int                  # requests
    layers: int             # layers in the IndexShare group
    ctx: int                # context length (fixed), or the upper bound
    ctx_lo: int             # lower bound when contexts are drawn, else == ctx
    k: int                  # top-k
    S: int                  # sets
    W: int                  # ways per set
    H: int                  # query heads
    steps: int              # decode steps of the workload
    scores: str             # 'walk' | 'ar1' | 'ar1_hot' | 'iid_ties'
    overlap: float = 0.60   # target adjacent-step top-k overlap (ar1*)
    hot_frac: float = 0.0   # fraction of positions in the hot set
    hot_offset: float = 0.0  # score offset of hot positions, in sigma
    hot_drift: float = 0.0  # fraction of hot members replaced per step
    walk_sigma: float = 0.3  # 'walk': per-step noise
    tie_frac: float = 0.0   # 'iid_ties': fraction of scores put on a grid
    tie_grid: float = 0.125  # 'iid_ties': grid step
    overflow_request: int = -1  # 'iid_ties': request whose top-k floods a set
    overflow_count: int = 0     # positions forced into that set per step
    overflow_set: int = 7
    overflow_boost: float = 10.0
    notes: str = field(default="", compare=False)

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def P(self) -> int:
        return self.S * self.W

    @property
    def ctx_stride(self) -> int:
        """Row stride of the per-request score and host-KV arrays."""
        return ((self.ctx + 31) // 32) * 32

    @property
    def rows_per_step(self) -> int:
        """Selected KV rows one decode step serves: one per (request, layer, k)."""
        return self.B * self.layers * self.k


TINY = Workload(
    name="tiny", index=0, B=1, layers=1, ctx=4096, ctx_lo=4096, k=256, S=256,
    W=4, H=16, steps=4, scores="walk",
    notes="1 request, 1 layer; scores: step 0 U(0,1), then + N(0, 0.3) per step")

DECODE_BATCH = Workload(
    name="decode_batch", index=1, B=32, layers=4, ctx=65536, ctx_lo=65536,
    k=2048, S=512, W=16, H=128, steps=64, scores="ar1", overlap=0.60,
    notes="AR(1) scores calibrated to ~60% adjacent-step top-k overlap")

LONG_CONTEXT = Workload(
    name="long_context", index=2, B=8, layers=4, ctx=200000, ctx_lo=30000,
    k=2048, S=1024, W=16, H=128, steps=128, scores="ar1_hot", overlap=0.60,
    hot_frac=0.10, hot_offset=2.0, hot_drift=0.01,
    notes="contexts U[30K, 200K]; AR(1) + drifting hot set (10% of positions, +2 sigma)")

LARGE_BATCH = Workload(
    name="large_batch", index=3, B=128, layers=4, ctx=32768, ctx_lo=32768,
    k=2048, S=512, W=16, H=128, steps=32, scores="ar1", overlap=0.60,
    notes="miss-path throughput: 19 GB of host KV read zero-copy")

ADVERSARIAL = Workload(
    name="adversarial", index=4, B=4, layers=4, ctx=1048576, ctx_lo=1048576,
    k=2048, S=512, W=16, H=128, steps=32, scores="iid_ties",
    tie_frac=0.05, tie_grid=0.125, overflow_request=3, overflow_count=48,
    overflow_set=7, overflow_boost=10.0,
    notes="independent scores each step; 5% on a 1/8 grid (exact ties); "
          "request 3 floods set 7 with 48 tokens per step (FIFO overflow)")

WORKLOADS = [TINY, DECODE_BATCH, LONG_CONTEXT, LARGE_BATCH, ADVERSARIAL]
BY_NAME = {w.name: w for w in WORKLOADS}


def get(name: str) -> Workload:
    return BY_NAME[name]


def scaled(w: Workload, **overrides) -> Workload:
    """A copy of `w` with some fields changed (smaller parity cases)."""
    d = {f: getattr(w, f) for f in w.__dataclass_fields__}
    d.update(overrides)
    if "ctx" in overrides and "ctx_lo" not in overrides and w.ctx_lo == w.ctx:
        d["ctx_lo"] = d["ctx"]
    return Workload(**d)
