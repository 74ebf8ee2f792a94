"""Index arithmetic of the attention variant that reads its rows straight from
the pool (csrc/sfa.cu, the kPool producer), restated on the CPU: over every
score and value stage, the 4-row gathers of the 32 producer lanes land inside
their stage's tile, cover every 128-byte row block of it exactly once, and put
selection position p at tile row p (so the tile equals the one a plain tile
load of the selection gives); and the pool row each position reads stays inside
the pool tensor, for hits, misses and bad entries alike."""
import numpy as np

kHeads, kChunk, kHalf, kKB = 128, 512, 256, 9
kQBytes = kHeads * 128
kKBytes = kHalf * 128
kVBox = 64 * 128
kVBytes = 4 * kVBox
INT_MIN = -(1 << 31)


def test_score_and_value_gathers_cover_their_tiles_once():
    for nh in range(2):
        seen = {}
        for lane in range(32):
            for g, first in ((lane, nh * kHalf + 4 * lane), (lane + 32, nh * kHalf + 128 + 4 * lane)):
                dst = g * 512
                assert 0 <= dst and dst + 512 <= kKBytes
                for i in range(4):
                    row_block = (dst + i * 128) // 128
                    assert row_block not in seen
                    seen[row_block] = first + i
        # tile row r (128-byte block r of the K area) holds position nh*256 + r
        assert seen == {r: nh * kHalf + r for r in range(kHalf)}
    for rb in range(8):
        for half in range(2):
            seen = {}
            for lane in range(32):
                g, jb = lane & 15, lane >> 4
                for box in (jb, jb + 2):
                    dst = box * kVBox + g * 512
                    assert 0 <= dst and dst + 512 <= kVBytes
                    col = half * 256 + box * 64
                    assert 0 <= col and col + 64 <= 512
                    for i in range(4):
                        key = (box, (g * 512 + i * 128) // 128)
                        assert key not in seen
                        seen[key] = (rb * 64 + 4 * g + i, col)
            assert seen == {(box, r): (rb * 64 + r, half * 256 + box * 64)
                            for box in range(4) for r in range(64)}


def _pool_row(src_map, miss_ids, miss_pos, M, repeats, b, k, j, P, prow):
    """The kernel's pool_row, restated."""
    src = int(src_map[b, j])
    rel, bad = P + j, 0
    if src >= 0:
        if src < P:
            rel = src
        else:
            bad |= 4
    elif src == INT_MIN:
        bad |= 1
    elif repeats:
        t = -1 - src
        ids = list(miss_ids[b, :M])
        f = miss_pos[b, ids.index(t)] if t in ids else -1
        if 0 <= f < k:
            rel = P + f
        else:
            bad |= 1
    return b * prow + rel, bad


def test_pool_rows_stay_inside_the_pool():
    rng = np.random.default_rng(3)
    B, k, P = 3, 700, 64
    prow = P + k
    src = rng.integers(-5000, P + 10, size=(B, k)).astype(np.int64)
    src[0, :5] = INT_MIN
    miss_ids = np.zeros((B, k), np.int64)
    miss_pos = np.zeros((B, k), np.int64)
    for b in range(B):
        first = {}
        for j in range(k):
            if src[b, j] < 0 and src[b, j] != INT_MIN:
                first.setdefault(-1 - int(src[b, j]), j)
        ts = sorted(first)
        miss_ids[b, :len(ts)] = ts
        miss_pos[b, :len(ts)] = [first[t] for t in ts]
    for b in range(B):
        M = int(np.sum(miss_ids[b] != 0))
        for repeats in (False, True):
            for c in range((k + kChunk - 1) // kChunk):
                for p in range(kChunk):
                    j = min(c * kChunk + p, k - 1)
                    row, _ = _pool_row(src, miss_ids, miss_pos, M, repeats, b, k, j, P, prow)
                    assert b * prow <= row < (b + 1) * prow
