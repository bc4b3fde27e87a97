"""The warp reduce-scatter of the pair kernel, restated over 32 lanes on the host.

Each lane holds one partial sum per source of a batch of NB sources (8 or 16).
Each butterfly level across lane mask m = 16, 8, ... halves the values a lane
keeps: the lanes with the mask bit keep the upper half, the others the lower
half, and each adds its partner's copy of the half it keeps. After log2(NB)
levels one value is left per lane; the remaining masks sum it over the rest
of the warp. The kernel then reads source l >> (5 - log2 NB) in lane l, and
the lanes whose low 5 - log2 NB bits are zero write it. These tests pin that
mapping and that every source's total is the sum over all 32 lanes.

The kernel's other variant rotates the sources through the lanes instead: at
step s of a group of 32 sources lane l evaluates source (l + s) mod 32 and
carries that source's running sum, taken from lane l + 1; after 32 steps lane
l holds the total of source (l + 31) mod 32.
"""
import numpy as np
import pytest

LANES = 32


def reduce_scatter(v):
    """v: (32, NB) per-lane partial sums -> (32,) value each lane ends with."""
    v = v.copy()
    nb = v.shape[1]
    levels = nb.bit_length() - 1
    lane = np.arange(LANES)
    for level in range(levels):
        half = (nb >> level) >> 1
        m = 16 >> level
        up = (lane & m) != 0
        keep = np.where(up[:, None], v[:, half:2 * half], v[:, :half])
        send = np.where(up[:, None], v[:, :half], v[:, half:2 * half])
        v[:, :half] = keep + send[lane ^ m]
    out = v[:, 0].copy()
    m = 16 >> levels
    while m >= 1:
        out = out + out[lane ^ m]
        m >>= 1
    return out


@pytest.mark.parametrize("nb", [8, 16])
def test_lane_holds_its_source_total(nb):
    rng = np.random.default_rng(nb)
    v = rng.standard_normal((LANES, nb))
    out = reduce_scatter(v)
    shift = 5 - (nb.bit_length() - 1)
    totals = v.sum(axis=0)
    for lane in range(LANES):
        assert out[lane] == pytest.approx(totals[lane >> shift], rel=1e-12, abs=1e-12)
    writers = [lane for lane in range(LANES) if lane & ((1 << shift) - 1) == 0]
    assert sorted(lane >> shift for lane in writers) == list(range(nb))


@pytest.mark.parametrize("nb", [8, 16])
def test_shuffle_count(nb):
    """3 components x (NB - 1 halving shuffles + the summing levels)."""
    levels = nb.bit_length() - 1
    halving = sum((nb >> level) >> 1 for level in range(levels))
    summing = 5 - levels
    assert halving == nb - 1
    assert 3 * (halving + summing) == {8: 27, 16: 48}[nb]


def test_integer_sums_are_exact():
    """With small integers every addition is exact, so the mapping is checked
    without rounding: each lane's total equals its source's column sum."""
    v = np.arange(LANES * 16, dtype=np.float64).reshape(LANES, 16) % 7
    out = reduce_scatter(v)
    assert np.array_equal(out, v.sum(axis=0)[np.arange(LANES) >> 1])


def rotate_through_lanes(c):
    """c: (32, 32) contribution of lane l to source s of a group.

    Each step every lane takes the running sum from lane l + 1 (mod 32), then
    adds its contribution to source (l + step) mod 32.  Returns the (32,) sum
    each lane holds after the 32 steps, the additions in the order they ran.
    """
    lane = np.arange(LANES)
    carry = np.zeros(LANES)
    order = [[] for _ in range(LANES)]  # lanes each source's sum passed through
    held = (lane - 1) % LANES  # source whose (zero) sum each lane carries before step 0
    for step in range(LANES):
        carry = carry[(lane + 1) % LANES]
        held = held[(lane + 1) % LANES]
        src = (lane + step) % LANES
        assert np.array_equal(held, src)  # the sum arrives where its source is evaluated
        carry = carry + c[lane, src]
        for l in range(LANES):
            order[src[l]].append(l)
    return carry, order


def test_rotation_leaves_each_source_total_in_lane_before():
    rng = np.random.default_rng(7)
    c = rng.standard_normal((LANES, LANES))
    out, order = rotate_through_lanes(c)
    totals = c.sum(axis=0)
    for lane in range(LANES):
        src = (lane + 31) % LANES
        assert out[lane] == pytest.approx(totals[src], rel=1e-12, abs=1e-12)
    # every source visited every lane exactly once, in a fixed order
    for src in range(LANES):
        assert sorted(order[src]) == list(range(LANES))


def test_rotation_integer_sums_are_exact():
    c = (np.arange(LANES * LANES).reshape(LANES, LANES) * 37 % 11).astype(np.float64)
    out, _ = rotate_through_lanes(c)
    assert np.array_equal(out, c.sum(axis=0)[(np.arange(LANES) + 31) % LANES])


@pytest.mark.parametrize("tj,groups", [(512, 1), (512, 2), (256, 2), (640, 1)])
def test_rotation_covers_each_source_of_a_tile(tj, groups):
    """The kernel's indices for a tile of tj sources: group g (32 * groups
    sources), step s, lane l and group h read source g + 32 h + (l + s) mod 32;
    lane l stores the sum of source g + 32 h + (l + 31) mod 32.  Every source
    is read once by every lane and stored by exactly one lane."""
    lane = np.arange(LANES)
    reads = np.zeros((tj, LANES), dtype=np.int64)
    stores = np.zeros(tj, dtype=np.int64)
    for g in range(0, tj, 32 * groups):
        for h in range(groups):
            for step in range(LANES):
                np.add.at(reads, (g + 32 * h + (lane + step) % LANES, lane), 1)
            np.add.at(stores, g + 32 * h + (lane + 31) % LANES, 1)
    assert np.all(reads == 1) and np.all(stores == 1)
