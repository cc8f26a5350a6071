"""Pins for the oracle's Philox4x32-10 generator and its draw layout.

The generator follows Salmon et al., "Parallel Random Numbers: As Easy as
1, 2, 3" (SC'11), sec. 3.  It is pinned against an independent
implementation: the host-side Philox4_32_10 generator of the cuRAND library
in the CUDA toolkit, which runs on the CPU.  That generator's output stream
is laid out in blocks of four words; block b is the generator's output for
counter (b // 65536 low, b // 65536 high, b mod 65536, 0) under the key
(seed low, seed high) -- so comparisons at chosen offsets check the round
function, both multipliers, the key schedule, the output word order and
counter words x, y and z.  (Word w enters the rounds as word y does; the
draw tests below check that it changes the draws.)"""
import ctypes
import os

import numpy as np
import pytest

import oracle

_CURAND_PATHS = ["/usr/local/cuda/lib64/libcurand.so", "libcurand.so", "libcurand.so.10"]
_PHILOX4_32_10 = 161          # curandRngType_t of the Philox4x32-10 generator


def _curand():
    for path in _CURAND_PATHS:
        try:
            return ctypes.CDLL(path)
        except OSError:
            continue
    pytest.skip("cuRAND library not found")


def curand_block(lib, seed: int, block: int):
    """The four words of block `block` of cuRAND's host Philox stream."""
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), _PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(4 * block)) == 0
        out = (ctypes.c_uint32 * 4)()
        assert lib.curandGenerate(gen, out, ctypes.c_size_t(4)) == 0
        return tuple(out)
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed", [0, 7, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
def test_philox_matches_curand(seed):
    lib = _curand()
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for block in (0, 1, 5000, 65535, 65536, 70000, (1 << 20) + 7, (1 << 48) + 65536 * 3 + 11,
                  (1 << 50) + 9, (1 << 60) + (1 << 34) + 12345):
        j, s = divmod(block, 65536)
        ctr = (j & 0xFFFFFFFF, j >> 32, s, 0)
        assert oracle.philox4x32_10(ctr, key) == curand_block(lib, seed, block), (hex(seed), block)


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
