"""Work division of the pair-symmetric path, checked on the host.

The pair kernel numbers its units (i-block I, source tile t) block by block,
block I taking the tiles from its own first tile, TB * I, to the last; the
units before block I number I * ntiles - TB * I (I - 1) / 2.  A tile of the
block itself is evaluated from both sides (each target sums all its sources);
a later tile once, the term going to the target and its negative (with the
masses swapped) to the source.  The units are divided evenly over a wave of
CTAs (unit_begin / unit_owner), and the pass may be cut into chunks of whole
i-blocks.  These tests restate that enumeration and walk it the way a CTA
does, and check the property the sum rests on: every ordered pair (i, j),
i != j, of the n bodies reaches a_i exactly once — not twice, not never.
"""
import itertools

import numpy as np
import pytest


def units_before(I, ntiles, tb):
    return I * ntiles - tb * (I * (I - 1) // 2)


def unit_begin(units, grid, c):
    return units * c // grid


def unit_owner(units, grid, u):
    return ((u + 1) * grid - 1) // units


def walk(n, block, tj, grid, chunks=None):
    """Count how often each ordered pair (i, j) reaches a_i."""
    assert block % tj == 0
    tb = block // tj
    ntiles, nblocks = -(-n // tj), -(-n // block)
    hits = np.zeros((n, n), dtype=np.int64)
    bounds = chunks or [0, nblocks]
    for I0, I1 in zip(bounds[:-1], bounds[1:]):
        u_base = units_before(I0, ntiles, tb)
        units = units_before(I1, ntiles, tb) - u_base
        g = min(units, grid)
        for c in range(g):
            lo = u_base + unit_begin(units, g, c)
            count = unit_begin(units, g, c + 1) - unit_begin(units, g, c)
            # the CTA's first unit: the largest I with units_before(I) <= lo
            I = max(k for k in range(nblocks) if units_before(k, ntiles, tb) <= lo)
            t = tb * I + (lo - units_before(I, ntiles, tb))
            for _ in range(count):
                targets = range(I * block, min(n, (I + 1) * block))
                sources = range(t * tj, min(n, (t + 1) * tj))
                diag = t < tb * (I + 1)
                for i, j in itertools.product(targets, sources):
                    if i == j:
                        continue  # r = 0: adds exactly nothing
                    hits[i, j] += 1
                    if not diag:
                        hits[j, i] += 1  # the reaction
                t += 1
                if t == ntiles:
                    I += 1
                    t = tb * I
    return hits


@pytest.mark.parametrize("n,block,tj,grid", [
    (1, 8, 4, 3), (7, 8, 4, 3), (8, 8, 4, 3), (9, 8, 4, 3), (33, 8, 4, 5), (40, 8, 2, 7),
    (50, 12, 4, 1), (50, 12, 4, 4), (61, 12, 6, 9), (64, 16, 8, 200), (97, 24, 8, 6),
])
def test_every_pair_reaches_each_body_once(n, block, tj, grid):
    hits = walk(n, block, tj, grid)
    want = np.ones((n, n), dtype=np.int64) - np.eye(n, dtype=np.int64)
    assert np.array_equal(hits, want)


@pytest.mark.parametrize("n,block,tj,grid,chunks", [
    (40, 8, 4, 3, [0, 1, 2, 5]), (57, 8, 4, 5, [0, 3, 4, 8]), (97, 24, 8, 6, [0, 1, 2, 3, 5]),
])
def test_chunks_of_blocks_cover_the_same_pairs(n, block, tj, grid, chunks):
    hits = walk(n, block, tj, grid, chunks)
    want = np.ones((n, n), dtype=np.int64) - np.eye(n, dtype=np.int64)
    assert np.array_equal(hits, want)


def test_unit_numbering_closed_form():
    """units_before matches a direct count, and every unit has one owner."""
    for ntiles, tb in [(10, 2), (17, 3), (64, 8)]:
        nblocks = -(-ntiles // tb)
        total = 0
        for I in range(nblocks + 1):
            assert units_before(I, ntiles, tb) == total
            if I < nblocks:
                total += ntiles - tb * I
        for grid in (1, 5, 152):
            g = min(total, grid)
            owners = [unit_owner(total, g, u) for u in range(total)]
            for c in range(g):
                span = range(unit_begin(total, g, c), unit_begin(total, g, c + 1))
                assert all(owners[u] == c for u in span)


@pytest.mark.parametrize("n,block,tj,grid", [
    (20000, 2048, 256, 152), (16384, 2048, 256, 152), (1048576, 4096, 512, 152),
    (1048576, 3584, 512, 152), (65537, 2048, 512, 152), (5000, 512, 128, 7)])
def test_block_segments_of_sharing_ctas(n, block, tj, grid):
    """The finishing passes read, for a block shared by CTAs c0..c1, the first
    segment of every CTA after c0 and, of c0 itself, the first segment when c0
    starts at the block's first unit, else its last: every CTA after c0 starts
    inside the block."""
    nblocks, ntiles, tb = -(-n // block), -(-n // tj), block // tj
    units = units_before(nblocks, ntiles, tb)
    grid = min(grid, units)
    for I in range(nblocks):
        u0 = units_before(I, ntiles, tb)
        u1 = units_before(I + 1, ntiles, tb) - 1
        c0, c1 = unit_owner(units, grid, u0), unit_owner(units, grid, u1)
        assert unit_begin(units, grid, c0) <= u0 < unit_begin(units, grid, c0 + 1)
        for cc in range(c0 + 1, c1 + 1):
            assert u0 < unit_begin(units, grid, cc) <= u1
