"""Index arithmetic of the attention variant that reads its rows straight from
the pool (csrc/sfa.cu, the kPool loader warps), restated on the CPU: over every
score and value stage, the 16-byte copies of the 256 loader threads land inside
their stage's tile, cover it exactly once, and put 16-byte column c of
selection row p where a 128-byte-swizzled tile load of the selection would
(row p at p * 128, column c at (c ^ (p & 7)) * 16); every source piece lies
inside its 1152-byte row; and the pool row each position reads stays inside
the pool tensor, for hits, misses and bad entries alike."""
import numpy as np

kHeads, kChunk, kHalf, kKB = 128, 512, 256, 9
kQBytes = kHeads * 128
kKBytes = kHalf * 128
kVBox = 64 * 128
kVBytes = 4 * kVBox
kLoaders = 256
INT_MIN = -(1 << 31)


def _swz(row, col):
    return row * 128 + ((col ^ (row & 7)) << 4)


def test_score_stage_copies_cover_q_and_k_tiles_once():
    for nh in range(2):
        for kb in range(kKB):
            q_seen, k_seen = {}, {}
            for lt in range(kLoaders):
                for i in range(kHeads * 8 // kLoaders):
                    pc = lt + kLoaders * i
                    h, col = pc >> 3, pc & 7
                    dst = _swz(h, col)
                    assert 0 <= dst and dst + 16 <= kQBytes and dst not in q_seen
                    src = kb * 128 + col * 16        # inside the head's row
                    assert 0 <= src and src + 16 <= 1152
                    q_seen[dst] = (h, kb * 64 + col * 8)
                for i in range(kHalf * 8 // kLoaders):
                    pc = lt + kLoaders * i
                    r, col = pc >> 3, pc & 7
                    dst = kQBytes + _swz(r, col)
                    assert kQBytes <= dst and dst + 16 <= kQBytes + kKBytes and dst not in k_seen
                    src = kb * 128 + col * 16
                    assert 0 <= src and src + 16 <= 1152
                    k_seen[dst] = (nh * kHalf + r, kb * 64 + col * 8)
            assert len(q_seen) == kQBytes // 16 and len(k_seen) == kKBytes // 16
            # what a swizzled tile load puts there: position / dims per 16 bytes
            assert k_seen == {kQBytes + _swz(r, c): (nh * kHalf + r, kb * 64 + c * 8)
                              for r in range(kHalf) for c in range(8)}


def test_value_stage_copies_cover_the_tile_once():
    for half in range(2):
        for rb in range(8):
            seen = {}
            for lt in range(kLoaders):
                for i in range(64 * 32 // kLoaders):
                    pc = lt + kLoaders * i
                    r, j, col = pc >> 5, (pc >> 3) & 3, pc & 7
                    dst = j * kVBox + _swz(r, col)
                    assert 0 <= dst and dst + 16 <= kVBytes and dst not in seen
                    src = (half * 256 + j * 64) * 2 + col * 16
                    assert 0 <= src and src + 16 <= 1024      # inside the 512 value dims
                    seen[dst] = (rb * 64 + r, half * 256 + j * 64 + col * 8)
            assert seen == {j * kVBox + _swz(r, c): (rb * 64 + r, half * 256 + j * 64 + c * 8)
                            for j in range(4) for r in range(64) for c in range(8)}


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
