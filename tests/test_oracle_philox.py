"""Pins for the oracle's Philox4x32-10 generator and its draw layout.

The generator follows Salmon et al., "Parallel Random Numbers: As Easy as
1, 2, 3" (SC'11), sec. 3.  Its pins are the known-answer vectors published
with that paper's reference implementation (zero counter and key, all-ones,
and the pi-digits vector) -- three independent 128-bit answers that a wrong
multiplier, Weyl constant, word order or round count cannot all reproduce."""
import numpy as np

import oracle

KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


def test_philox_known_answers():
    for ctr, key, want in KAT:
        assert oracle.philox4x32_10(ctr, key) == want


def test_draws_layout_element_tied():
    """Draws come from counter (index/4, tensor, step) keyed by the seed; word
    index%4 gives m (low half) and v (high half) -- "When Small Updates
    Disappear" sec. 7.3: tied to the element, not to a thread block."""
    seed, step, t = 0x1234_5678_9ABC_DEF0, 7, 3
    for index in (0, 1, 2, 3, 4, 5, 1 << 33, (1 << 33) + 3):
        q = index >> 2
        words = oracle.philox4x32_10((q & 0xFFFFFFFF, q >> 32, t, step),
                                     (seed & 0xFFFFFFFF, seed >> 32))
        w = words[index & 3]
        assert oracle.draws(seed, step, t, index) == (w & 0xFFFF, w >> 16)


def test_draws_change_with_every_key_field():
    base = oracle.draws(5, 10, 2, 1000)
    assert oracle.draws(6, 10, 2, 1000) != base
    assert oracle.draws(5, 11, 2, 1000) != base
    assert oracle.draws(5, 10, 3, 1000) != base
    assert oracle.draws(5, 10, 2, 1001) != base
    assert oracle.draws(5, 10, 2, 1000) == base


def test_draws_roughly_uniform():
    r = np.array([oracle.draws(99, 1, 0, i) for i in range(40000)], dtype=np.float64)
    # mean of U{0..65535} is 32767.5, sd 18918.6; 40000 samples -> se ~95
    assert abs(r[:, 0].mean() - 32767.5) < 600
    assert abs(r[:, 1].mean() - 32767.5) < 600
    assert abs(np.corrcoef(r[:, 0], r[:, 1])[0, 1]) < 0.03


def test_cast_draw_layout_uses_every_half_once():
    """The standalone cast takes one 16-bit draw per element: counter
    (index/8, tensor, step), word (index/2) mod 4, low half for even and high
    half for odd indices, so the eight elements of a counter use its eight
    halves exactly once each."""
    seed, step, t = 0xFEDC_BA98_7654_3210, 12, 5
    for base in (0, 8, 1 << 35):
        q = base >> 3
        words = oracle.philox4x32_10((q & 0xFFFFFFFF, q >> 32, t, step),
                                     (seed & 0xFFFFFFFF, seed >> 32))
        halves = [h for w in words for h in (w & 0xFFFF, w >> 16)]
        got = [oracle.cast_draw(seed, step, t, base + j) for j in range(8)]
        assert got == halves
    assert oracle.cast_draw(seed, step, t, 8) != oracle.cast_draw(seed, step, t, 0) or \
        oracle.cast_draw(seed, step, t, 9) != oracle.cast_draw(seed, step, t, 1)


def test_cast_draws_roughly_uniform_and_uncorrelated():
    r = np.array([oracle.cast_draw(3, 1, 0, i) for i in range(40000)], dtype=np.float64)
    assert abs(r.mean() - 32767.5) < 600
    assert abs(np.corrcoef(r[0::2], r[1::2])[0, 1]) < 0.03
