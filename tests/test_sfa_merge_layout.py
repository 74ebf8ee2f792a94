"""Layout of the attention's in-cluster merge (csrc/sfa.cu, merge_in_cluster),
restated on the CPU for clusters of 1, 2 and 4 chunk CTAs: every remote write
lands inside the receive region below the published (m, l) block, no two
writes collide, every owner reads back exactly what its peers wrote, and every
(unit, head) of the output is written by one CTA."""


def test_merge_layout():
    kHeads, kUnits, kUnitBytes = 128, 16, 128 * 128
    kTileBytes = 8 * 128 * 128 + 2 * (128 * 128 + 256 * 128)
    kMlOffset = kTileBytes - kHeads * 8
    for C in (1, 2, 4):
        upo = kUnits // C
        writes = {}      # (owner, byte offset) -> (src, unit, head, j)
        for rank in range(C):
            for part in range(2):
                for row in range(kHeads):
                    for u in range(part, kUnits, 2):
                        o = u // upo
                        if o == rank:
                            continue
                        slot = (rank - o - 1 + C) % C
                        assert 0 <= slot <= C - 2
                        base = slot * upo * kUnitBytes + ((u % upo) * kHeads + row) * 128
                        for j in range(8):
                            off = base + ((j ^ (row & 7)) << 4)
                            assert 0 <= off and off + 16 <= kMlOffset, (C, off)
                            key = (o, off)
                            assert key not in writes, ("collision", C, key)
                            writes[key] = (rank, u, row, j)
        # reads: owner o for its units sums slots 0..C-2; every read location was written by a
        # distinct source, and the sources of a unit are exactly the other ranks
        outputs = set()
        for o in range(C):
            for part in range(2):
                for row in range(kHeads):
                    for u in range(part, kUnits, 2):
                        if u // upo != o:
                            continue
                        outputs.add((u, row))
                        srcs = set()
                        for sl in range(C - 1):
                            base = sl * upo * kUnitBytes + ((u % upo) * kHeads + row) * 128
                            for j in range(8):
                                off = base + ((j ^ (row & 7)) << 4)
                                rank, uu, rr, jj = writes[(o, off)]
                                assert (uu, rr, jj) == (u, row, j), (C, o, u, row, j, uu, rr, jj)
                                srcs.add(rank)
                        assert srcs == set(range(C)) - {o}, (C, o, u, srcs)
        assert outputs == {(u, r) for u in range(kUnits) for r in range(kHeads)}
        assert len(writes) == (C - 1) * kUnits * kHeads * 8
        # bank check: 8 consecutive heads, same unit and j, hit 8 different 16-byte bank groups
        for j in range(8):
            groups = {(((j ^ (row & 7)) << 4) // 16) for row in range(8)}
            assert len(groups) == 8
