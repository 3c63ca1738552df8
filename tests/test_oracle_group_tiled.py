"""Pins of the oracle's group-tiled scale layout (scale_group_tiled): each
group's rows tiled on their own by the (separately pinned) MMA-tiled layout,
groups concatenated.  Checked against reductions to the plain tiling and a
hand-placed example."""
import numpy as np

from oracle import oracle


def _scales(rows, groups, seed):
    return np.random.default_rng(seed).integers(1, 255, size=(rows, groups), dtype=np.uint8)


def test_one_group_is_the_plain_tiling():
    s = _scales(300, 12, 1)
    assert np.array_equal(oracle.scale_group_tiled(s, [0, 300]), oracle.scale_tiled(s))


def test_groups_on_128_row_bands_give_the_plain_tiling():
    s = _scales(512, 8, 2)
    assert np.array_equal(oracle.scale_group_tiled(s, [0, 128, 384, 512]), oracle.scale_tiled(s))


def test_hand_placed_example():
    """rows 5, 4 groups (one atom per band), groups [0, 3) and [3, 5): row r
    of a band holds its 4 scales at bytes 16 r .. 16 r + 3 (r < 32); group 1
    starts a new 512-byte band; everything else is zero."""
    s = np.arange(1, 21, dtype=np.uint8).reshape(5, 4)
    want = np.zeros(1024, np.uint8)
    for r in range(3):
        want[16 * r:16 * r + 4] = s[r]
    for lr in range(2):
        want[512 + 16 * lr:512 + 16 * lr + 4] = s[3 + lr]
    assert np.array_equal(oracle.scale_group_tiled(s, [0, 3, 5]), want)
    # empty groups add no bands
    assert np.array_equal(oracle.scale_group_tiled(s, [0, 0, 3, 3, 3, 5, 5]), want)


def test_row_of_a_later_band_of_a_later_group():
    """Group 1 of [0, 130) [130, 300) with 12 scale groups: its local row 129 is
    row 1 of its second band; that band is band 3 overall (group 0 has two), and
    scale group 9 sits in that band's third atom at byte 4 * (1 // 32) + 16 * 1 + 1."""
    s = _scales(300, 12, 3)
    out = oracle.scale_group_tiled(s, [0, 130, 300])
    bands = 2 + 2
    assert out.size == bands * 3 * 512
    band, atom, lr, j = 3, 9 // 4, 1, 9 % 4
    assert out[(band * 3 + atom) * 512 + 16 * lr + 4 * (lr // 32) + j] == s[130 + 129, 9]
    # group 0's second band holds its local rows 128 and 129 (band rows 0, 1):
    # every other row of that band is zero padding (byte 16 (r % 32) + 4 (r // 32) + j)
    band1 = out[3 * 512:6 * 512].reshape(3, 32, 4, 4)      # atom, r % 32, r // 32, j
    live = np.zeros((32, 4), bool)
    live[0, 0] = live[1, 0] = True
    assert not band1[:, ~live, :].any()
    assert np.array_equal(band1[0, 0, 0], s[128, 0:4]) and np.array_equal(band1[2, 1, 0], s[129, 8:12])
