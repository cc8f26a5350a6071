"""Pins for the oracle's state codecs (BF16, E4M3, unsigned E2M2), nearest and
stochastic, against torch casts, brute force and the carry rule of
"When Small Updates Disappear" sec. 6.1 / sec. 3."""
import math
import struct

import numpy as np
import pytest
import torch

import oracle


def f32(x):
    return struct.unpack("<f", struct.pack("<f", x))[0]


def bits(x):
    return struct.unpack("<I", struct.pack("<f", x))[0]


def from_bits(u):
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


# ---------------------------------------------------------------- BF16
def test_bf16_nearest_matches_torch_cast():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 4000),
        np.array([0.0, -0.0, 1e-40, -3e-39, 3.3895e38, 3.40282e38, np.inf, -np.inf,
                  1.00390625, 1.01171875, -1.00390625], dtype=np.float32),
        # exact ties at the dropped half
        np.array([from_bits(0x3F808000), from_bits(0x3F818000), from_bits(0xBF808000)], dtype=np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_encode(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # decode is exact: code << 16
    for c in [0x0000, 0x3F80, 0xBF80, 0x7F7F, 0x0001, 0x8001]:
        assert bits(oracle.bf16_decode(c)) == c << 16


def test_bf16_nearest_nan_inf_kept():
    assert oracle.bf16_encode(float("inf")) == 0x7F80
    assert oracle.bf16_encode(float("-inf")) == 0xFF80
    c = oracle.bf16_encode(float("nan"))
    assert (c & 0x7F80) == 0x7F80 and (c & 0x7F) != 0
    # a NaN whose payload sits only in the dropped bits stays a NaN
    c = oracle.bf16_encode(from_bits(0x7F800001))
    assert (c & 0x7F80) == 0x7F80 and (c & 0x7F) != 0


@pytest.mark.parametrize("x", [1.0 + 2 ** -9, 0.3, -0.3, 123.456, -7.77e-3, 1e-39, 3.3e38])
def test_bf16_stochastic_carry_count_is_dropped_bits(x):
    """sec. 6.1: a carry happens for exactly l of the 2^16 draws."""
    x = f32(x)
    w = bits(x)
    ell = w & 0xFFFF
    kept = w >> 16
    ups = 0
    for r in range(1 << 16):
        c = oracle.bf16_encode(x, True, r)
        assert c in (kept, kept + 1)
        ups += c == kept + 1
    assert ups == ell


def test_bf16_stochastic_unbiased_and_variance_exact():
    """sec. 3.1: E[q] = x and Var = (x - q-)(q+ - x), over all 2^16 draws."""
    for x in [f32(1.3), f32(-2.71828), f32(5e-3)]:
        codes = np.array([oracle.bf16_encode(x, True, r) for r in range(1 << 16)], dtype=np.uint32)
        q = (codes << 16).astype(np.uint32).view(np.float32).astype(np.float64)
        qm = from_bits(bits(x) & 0xFFFF0000)
        qp = from_bits((bits(x) & 0xFFFF0000) + 0x10000)
        assert math.isclose(q.mean(), x, rel_tol=0, abs_tol=0)  # exact in double
        var = ((q - x) ** 2).mean()
        assert var == pytest.approx(abs((x - qm) * (qp - x)), rel=1e-12)


def test_bf16_stochastic_exact_values_never_move():
    for x in [1.0, -2.5, 0.0, 65280.0, 1.5 * 2 ** -120]:
        c0 = oracle.bf16_encode(x)
        for r in range(0, 1 << 16, 97):
            assert oracle.bf16_encode(x, True, r) == c0


def test_bf16_stochastic_small_update_example(pages):
    """sec. 3.3: an update of 0.2 u -- nearest never moves, SR moves ~20 %."""
    ex = pages["sr_small_update_example"]
    base = 1.0
    u = 2.0 ** -7
    x = f32(base + ex["update_in_ulps"] * u)
    assert oracle.bf16_encode(x) == oracle.bf16_encode(base)
    moves = sum(oracle.bf16_encode(x, True, r) != oracle.bf16_encode(base) for r in range(1 << 16))
    assert moves / 65536 == pytest.approx(ex["stochastic_moves_fraction"], abs=1e-4)


# ---------------------------------------------------------------- E4M3
def e4m3_all():
    return [(c, oracle.e4m3_decode(c)) for c in range(256)]


def test_e4m3_decode_table_facts():
    vals = dict(e4m3_all())
    assert vals[0x7E] == 448.0 and math.isnan(vals[0x7F]) and math.isnan(vals[0xFF])
    assert vals[0x08] == 2.0 ** -6            # smallest normal
    assert vals[0x01] == 2.0 ** -9            # smallest subnormal
    assert vals[0x38] == 1.0 and vals[0xB8] == -1.0
    finite = sorted(v for c, v in vals.items() if not math.isnan(v) and v >= 0 and c < 0x80)
    assert len(finite) == 127 and len(set(finite)) == 127


def test_e4m3_roundtrip_and_ties():
    pos = sorted((v, c) for c, v in e4m3_all() if c < 0x7F)
    for v, c in pos:
        assert oracle.e4m3_encode(v) == c
        assert oracle.e4m3_encode(-v) == (c | 0x80)
    for (a, ca), (b, cb) in zip(pos[:-1], pos[1:]):
        mid = (a + b) / 2
        even = ca if (ca & 1) == 0 else cb
        assert oracle.e4m3_encode(mid) == even
        assert oracle.e4m3_encode(np.nextafter(np.float32(mid), np.float32(0))) == ca
        assert oracle.e4m3_encode(np.nextafter(np.float32(mid), np.float32(1e9))) == cb


def test_e4m3_nearest_matches_torch_in_range():
    rng = np.random.default_rng(2)
    vals = (rng.standard_normal(20000) * np.exp(rng.uniform(-12, 6, 20000))).astype(np.float32)
    vals = vals[np.abs(vals) < 464.0]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_saturates_and_nan():
    assert oracle.e4m3_encode(1e6) == 0x7E
    assert oracle.e4m3_encode(-1e6) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    for r in (0, 30000, 65535):
        assert oracle.e4m3_encode(500.0, True, r) == 0x7E


@pytest.mark.parametrize("x", [0.3, 1.7, 100.3, 3e-3, 2.0 ** -6 + 3e-5, 1e-3, 440.0])
def test_e4m3_stochastic_carry_count(x):
    x = f32(x)
    codes = [oracle.e4m3_encode(x, True, r) for r in range(0, 1 << 16)]
    lo = oracle.e4m3_encode(x, True, 0)               # r = 0 never carries unless exact
    ups = sum(c != lo for c in codes)
    a = oracle.e4m3_decode(lo)
    b = oracle.e4m3_decode(lo + 1)
    frac = (x - a) / (b - a)
    assert ups == math.floor(frac * 65536)


# ---------------------------------------------------------------- E2M2
def test_e2m2_grid():
    vals = [oracle.e2m2_decode(c) for c in range(16)]
    assert vals[:4] == [0.0, 0.25, 0.5, 0.75]       # subnormal codes
    assert vals[4] == 1.0 and vals[15] == 7.0
    assert all(b > a for a, b in zip(vals[:-1], vals[1:]))
    # two fraction bits: four values per binade
    for lo in (1.0, 2.0, 4.0):
        assert sum(lo <= v < 2 * lo for v in vals) == 4


def test_e2m2_roundtrip_ties_saturation():
    vals = [oracle.e2m2_decode(c) for c in range(16)]
    for c, v in enumerate(vals):
        assert oracle.e2m2_encode(v) == c
    for c in range(15):
        mid = (vals[c] + vals[c + 1]) / 2
        assert oracle.e2m2_encode(mid) == (c if c % 2 == 0 else c + 1)
    assert oracle.e2m2_encode(7.4) == 15 and oracle.e2m2_encode(1e9) == 15
    assert oracle.e2m2_encode(-1.0) == 0 and oracle.e2m2_encode(float("nan")) == 15


def test_grid_ratios_to_bf16(pages):
    """sec. 2.1: FP8 is 16x and unsigned E2M2 32x coarser than BF16."""
    r = pages["grid_ratios"]
    for v in (1.0, 2.0):
        bf16_step = oracle.bf16_decode(oracle.bf16_encode(v) + 1) - v
        e4 = oracle.e4m3_decode(oracle.e4m3_encode(v) + 1) - v
        e2 = oracle.e2m2_decode(oracle.e2m2_encode(v) + 1) - v
        assert e4 / bf16_step == r["fp8_over_bf16"]
        assert e2 / bf16_step == r["fp4_e2m2_over_bf16"]


@pytest.mark.parametrize("x", [0.3, 1.1, 5.5, 6.9, 0.1])
def test_e2m2_stochastic_carry_count_and_mean(x):
    x = f32(x)
    codes = [oracle.e2m2_encode(x, True, r) for r in range(1 << 16)]
    lo = min(codes)
    a, b = oracle.e2m2_decode(lo), oracle.e2m2_decode(lo + 1)
    ups = sum(c != lo for c in codes)
    assert ups == math.floor((x - a) / (b - a) * 65536)
    mean = sum(oracle.e2m2_decode(c) for c in codes) / 65536
    assert mean == pytest.approx(x, abs=(b - a) / 65536)
