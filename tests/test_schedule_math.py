"""The tensor-core attention kernels' work split, checked on the host: per head group the tiles
of all sequences form one list, CTA k takes tiles [floor(T*k/n), floor(T*(k+1)/n)), each
(CTA, sequence) piece writes partial slot k + b, and the combine merges the slot interval
[kf + b, kl + b] with kf = ceil((P+1)*n/T) - 1, kl = ceil((P+len)*n/T) - 1. CTAs whose empty
range sits strictly inside a sequence mark their slot empty. These are the formulas the kernels
evaluate; this test proves they cover every tile once and never leave a merged slot unwritten.

The SM-pair kernel puts `seg_cost` extra units ahead of each (valid) sequence in the list, so
that a pair starting a new sequence takes fewer tiles; P is then the position of the
sequence's first tile, and a share may hold no tile at all."""
import numpy as np
import pytest


def ceil_div(a, b):
    return -(-a // b)


def schedule(ntiles, ncg, seg_cost=0):
    width = [n + seg_cost if n > 0 else 0 for n in ntiles]
    T = int(sum(width))
    # list position of each sequence's first tile
    P = (np.concatenate([[0], np.cumsum(width)[:-1]]) + seg_cost).astype(int)
    written = {}       # slot -> ("data", b, lo, hi) | ("empty", b)
    for k in range(ncg):
        r0, r1 = (T * k) // ncg, (T * (k + 1)) // ncg
        if r0 < r1:
            for b, (p, n) in enumerate(zip(P, ntiles)):
                lo, hi = max(r0, p), min(r1, p + n)
                if n > 0 and hi > lo:
                    assert k + b not in written
                    written[k + b] = ("data", b, lo - p, hi - p)
        else:
            for b, (p, n) in enumerate(zip(P, ntiles)):
                if n > 0 and p < r0 < p + n:
                    assert k + b not in written
                    written[k + b] = ("empty", b)
    meta = []
    for b, (p, n) in enumerate(zip(P, ntiles)):
        if n == 0:
            meta.append((0, 0))
            continue
        kf = ceil_div((p + 1) * ncg, T) - 1
        kl = ceil_div((p + n) * ncg, T) - 1
        meta.append((kf + b, kl - kf + 1))
    return T, written, meta


@pytest.mark.parametrize("seg_cost", [0, 3])
@pytest.mark.parametrize("seed", range(40))
def test_every_tile_once_and_every_merged_slot_written(seed, seg_cost):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 70))
    ncg = int(rng.integers(1, 160))
    lens = rng.integers(0, 40, size=B)          # tiles per sequence (0 = invalid length)
    if rng.random() < 0.3:
        lens = rng.integers(0, 3, size=B)        # few tiles: many CTAs have empty ranges
    T, written, meta = schedule(lens, ncg, seg_cost)
    n_slots = ncg + B - 1
    assert all(0 <= s < n_slots for s in written)
    covered = {b: [] for b in range(B)}
    for slot, w in written.items():
        if w[0] == "data":
            covered[w[1]].append((w[2], w[3]))
    for b in range(B):
        first, count = meta[b]
        if lens[b] == 0:
            assert count == 0
            continue
        # the tiles of b are covered exactly once by data slots
        segs = sorted(covered[b])
        assert segs[0][0] == 0 and segs[-1][1] == lens[b]
        assert all(segs[i][1] == segs[i + 1][0] for i in range(len(segs) - 1))
        # every slot in b's interval was written for b, and every data slot of b is inside it
        for s in range(first, first + count):
            assert s in written and written[s][1] == b, (b, s, written.get(s))
        data_slots = [s for s, w in written.items() if w[0] == "data" and w[1] == b]
        assert min(data_slots) >= first and max(data_slots) < first + count


def test_worked_example_ten_tiles_four_ctas():
    # shares [0,2) [2,5) [5,7) [7,10); a sequence on tiles 3..5 is merged from CTAs 1 and 2
    T, written, meta = schedule([3, 3, 4], 4)
    assert meta[1] == (1 + 1, 2)
    assert written[2] == ("data", 1, 0, 2) and written[3] == ("data", 1, 2, 3)


def test_worked_example_with_a_switch_cost():
    # list positions: seq 0 switch [0,3) tiles [3,6); seq 1 switch [6,9) tiles [9,12); seq 2
    # switch [12,15) tiles [15,19). T = 19; four pairs take [0,4) [4,9) [9,14) [14,19)
    T, written, meta = schedule([3, 3, 4], 4, seg_cost=3)
    assert T == 19
    assert written[0] == ("data", 0, 0, 1)        # pair 0: tile 0 of seq 0
    assert written[1] == ("data", 0, 1, 3)        # pair 1: tiles 1-2, then seq 1's switch
    assert written[3] == ("data", 1, 0, 3)        # pair 2: all of seq 1, then seq 2's switch
    assert written[5] == ("data", 2, 0, 4)        # pair 3: all of seq 2
    assert len(written) == 4
    assert meta == [(0, 2), (3, 1), (5, 1)]
