"""The warp reduce-scatter of the pair kernel, restated over 32 lanes on the host.

Each lane holds one partial sum per source of a batch of NB sources (8 or 16).
Each butterfly level across lane mask m = 16, 8, ... halves the values a lane
keeps: the lanes with the mask bit keep the upper half, the others the lower
half, and each adds its partner's copy of the half it keeps. After log2(NB)
levels one value is left per lane; the remaining masks sum it over the rest
of the warp. The kernel then reads source l >> (5 - log2 NB) in lane l, and
the lanes whose low 5 - log2 NB bits are zero write it. These tests pin that
mapping and that every source's total is the sum over all 32 lanes.
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
