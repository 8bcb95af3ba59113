"""The test helpers that excuse GPU/oracle mismatches (no GPU).

bf16_near_tie decides which bf16 differences the GPU parity tests accept, so a
mistake in it would widen every staged check.  It must flag exact rounding
midpoints, including the top of a binade, and must not flag values whose bf16
rounding an fp32 evaluation cannot change.
"""
import numpy as np

import oracle
from helpers import bf16_near_tie


def _bf16(x):
    return np.array([oracle.bf16_from_double(float(v)) for v in np.ravel(x)], np.uint16)


def test_midpoints_are_flagged_and_grid_points_are_not():
    rs = np.random.RandomState(0)
    grid = oracle.bf16_to_f64(_bf16(rs.standard_normal(2000) * np.exp2(rs.randint(-20, 20, 2000))))
    grid = grid[grid != 0]
    a = np.abs(grid)
    q = np.exp2(np.floor(np.log2(a)) - 7)              # the bf16 quantum of each value's binade
    mid = np.sign(grid) * (a + q / 2)                  # halfway to the next bf16 value up
    assert np.all(bf16_near_tie(mid, abs_frac=0.0))
    assert not np.any(bf16_near_tie(grid, abs_frac=0.0))


def test_the_band_is_relative():
    x = np.array([1.0 + 2.0 ** -8])                  # the midpoint between 1 and 1 + 2^-7
    for rel_off, flagged in ((5e-6, True), (-5e-6, True), (3e-5, False), (-3e-5, False)):
        assert bf16_near_tie(x * (1 + rel_off), abs_frac=0.0)[0] == flagged, rel_off


def test_top_of_a_binade():
    top = 2.0 - 2.0 ** -7                            # the largest bf16 value below 2
    mid = (top + 2.0) / 2
    assert bf16_near_tie(np.array([mid]), abs_frac=0.0)[0]
    assert not bf16_near_tie(np.array([top, 2.0]), abs_frac=0.0).any()


def test_outside_the_band_fp32_cannot_change_the_rounding():
    """Away from the band, rounding the value to fp32 first (as a GPU stage
    that computes in fp32 does) gives the same bf16 as rounding it once from
    fp64: fp32's own error (2^-24 relative) is far inside the 1e-5 band."""
    import torch
    rs = np.random.RandomState(1)
    x = rs.standard_normal(20000) * np.exp2(rs.randint(-10, 10, 20000))
    keep = ~bf16_near_tie(x, abs_frac=0.0)
    assert keep.mean() > 0.99
    via32 = torch.from_numpy(x[keep].astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(via32.view(np.uint16), _bf16(x[keep]))


def test_zero_and_the_absolute_term():
    assert not bf16_near_tie(np.array([0.0]))[0]
    # a value far below the tensor's rms is flagged through the absolute term,
    # whose tolerance there exceeds the value's whole bf16 quantum (cancellation)
    x = np.array([3e-6, 100.0, -100.0])
    assert bf16_near_tie(x, rel=0.0, abs_frac=1e-5)[0]
    assert not bf16_near_tie(x, rel=0.0, abs_frac=0.0)[0]


def _case():
    rs = np.random.RandomState(2)
    exact = rs.standard_normal(4000)
    ref = _bf16(exact)
    return exact, ref


def test_bits_match_accepts_equal_and_midpoint_differences():
    from helpers import bits_match
    exact, ref = _case()
    bits_match(ref.copy(), ref, exact, "equal")
    # move elements that sit on a midpoint by one step: excused however many
    mid = exact.copy()
    idx = np.arange(0, 4000, 7)
    a = np.abs(exact[idx])
    q = np.exp2(np.floor(np.log2(a)) - 7)
    mid[idx] = np.sign(exact[idx]) * (np.floor(a / q) * q + q / 2)
    ref_mid = _bf16(mid)
    got = ref_mid.copy()
    got[idx] = ref_mid[idx] ^ 1            # the other neighbour of each midpoint
    bits_match(got, ref_mid, mid, "midpoints")


def test_bits_match_counts_and_sizes_the_other_differences():
    import pytest
    from helpers import bits_match
    exact, ref = _case()
    away = np.flatnonzero(~bf16_near_tie(exact))[:10]
    got = ref.copy()
    got[away[:2]] += 1                      # two one-step differences: always allowed
    bits_match(got, ref, exact, "two")
    got[away[2]] += 1                       # a third needs slack
    with pytest.raises(AssertionError):
        bits_match(got, ref, exact, "three")
    bits_match(got, ref, exact, "three with slack", slack=3)
    got = ref.copy()
    got[away[0]] += 2                       # two steps: never allowed
    with pytest.raises(AssertionError):
        bits_match(got, ref, exact, "two steps", slack=100)
    excl = np.zeros(ref.shape, bool)
    excl[away[0]] = True
    bits_match(got, ref, exact, "excluded", exclude=excl)


def test_untile_inverts_the_documented_tiling():
    """untile_codes against the tiled layout written out element by element:
    byte (r, c) of a [rows][row_bytes] code tensor sits in tile
    (r / 128) * ceil(row_bytes / 128) + c / 128, at row r % 128, byte c % 128;
    tile bytes beyond row_bytes are zero."""
    from helpers import tiled_expert_bytes, untile_codes
    rs = np.random.RandomState(0)
    for rows, rb in ((256, 448), (128, 192), (384, 64), (128, 128)):
        src = rs.randint(0, 256, size=(rows, rb)).astype(np.uint8)
        kb = -(-rb // 128)
        tiles = np.zeros(rows // 128 * kb * 16384, np.uint8)
        for r in range(rows):
            for c in range(rb):
                t = (r // 128) * kb + c // 128
                tiles[t * 16384 + (r % 128) * 128 + c % 128] = src[r, c]
        assert np.array_equal(untile_codes(tiles, rows, rb), src)
        assert tiles.size == tiled_expert_bytes(rows, rb)
        # a plausible mistake -- K-block outermost -- does not pass
        wrong = tiles.reshape(rows // 128, kb, 128, 128).transpose(1, 0, 2, 3).reshape(-1)
        if kb > 1 and rows > 128:
            assert not np.array_equal(untile_codes(wrong, rows, rb), src)


def test_band_widens_the_near_tie_test():
    from helpers import bf16_near_tie
    x = np.array([1.0 + 2.0 ** -8 + 1e-4, 1.0 + 2.0 ** -8 + 1e-6])   # above a midpoint by 1e-4, 1e-6
    assert list(bf16_near_tie(x)) == [False, True]
    assert list(bf16_near_tie(x, band=np.array([2e-4, 0.0]))) == [True, True]
    assert list(bf16_near_tie(x, band=np.array([5e-5, 0.0]))) == [False, True]
