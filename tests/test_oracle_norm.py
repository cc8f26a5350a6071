"""Pins for the oracle's global gradient norm ("perf(training): fused
multi-tensor gradient-norm reduction", 'Numerics' and 'Correctness
properties'): brute force in exact rational arithmetic, closed forms,
the NaN/Inf rules and the clip coefficient."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def bf16_codes(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_values(codes):
    return (codes.astype(np.uint32) << 16).view(np.float32)


def exact_sumsq(arrays):
    s = Fraction(0)
    for a in arrays:
        for x in np.asarray(a, dtype=np.float64).ravel():
            s += Fraction(float(x)) ** 2
    return s


def test_brute_force_tiny_lists():
    rng = np.random.default_rng(3)
    f = [np.array([0.0, 1e-40, -3.5e-39, 65504.0, -1.0e30, 3.0], dtype=np.float32),
         (rng.standard_normal(37) * 10.0 ** rng.integers(-20, 20, 37)).astype(np.float32),
         np.zeros(5, np.float32)]
    b_vals = np.array([0.0, 1e-39, -2.0 ** -133, 65280.0, -3.0e38, 1.5, -7.25], np.float32)
    b = [bf16_codes(b_vals), bf16_codes(rng.standard_normal(29) * 1e3)]
    got = oracle.grad_norm(f + b)
    exact = exact_sumsq(f + [bf16_values(c) for c in b])
    assert abs(Fraction(got["sumsq"]) - exact) <= exact * Fraction(2.0 ** -52)
    assert got["norm2"] == pytest.approx(math.sqrt(float(exact)), rel=1e-15)
    allv = np.concatenate([np.abs(x).astype(np.float64) for x in f + [bf16_values(c) for c in b]])
    assert got["norm_inf"] == allv.max()
    assert got["nan_count"] == 0 and got["inf_count"] == 0 and got["status"] == 0


def test_bf16_sum_is_exact(pages):
    """'exact for BF16': BF16 squares have 16 significant bits, so a double sum
    over a moderate exponent range is exact."""
    assert pages["norm_accuracy"]["bf16_vs_fp64"] == 0.0
    rng = np.random.default_rng(4)
    codes = bf16_codes(rng.standard_normal(5000) * 3.0)
    got = oracle.grad_norm([codes])
    assert Fraction(got["sumsq"]) == exact_sumsq([bf16_values(codes)])


def test_closed_form_constant_tensor():
    """sqrt(sum of n copies of c^2) = sqrt(n) |c|."""
    for n, c in [(4096, 0.5), (10 ** 6, -3.0), (12345, 2.0 ** -60)]:
        got = oracle.grad_norm([np.full(n, c, np.float32)])
        assert got["norm2"] == pytest.approx(math.sqrt(n) * abs(c), rel=1e-15)
        assert got["norm_inf"] == abs(c)


def test_split_invariance_and_order():
    rng = np.random.default_rng(5)
    a = rng.standard_normal(100_001).astype(np.float32)
    whole = oracle.grad_norm([a])
    parts = oracle.grad_norm([a[:333], a[333:70000], a[70000:]])
    assert parts["norm2"] == pytest.approx(whole["norm2"], rel=1e-15)
    assert oracle.grad_norm([a[70000:], a[:70000]])["norm2"] == pytest.approx(whole["norm2"], rel=1e-15)


def test_fp32_accuracy_beats_fp32_tiles(pages):
    """The page's fp32-tile version was ~1e-7 off; the oracle must sit far
    below that bound: check against exact arithmetic on 200k values."""
    rng = np.random.default_rng(6)
    a = (rng.standard_normal(200_000) * np.exp(rng.uniform(-5, 5, 200_000))).astype(np.float32)
    got = oracle.grad_norm([a])
    exact = float(exact_sumsq([a]))
    rel = abs(got["sumsq"] - exact) / exact
    assert rel < pages["norm_accuracy"]["fp32_vs_fp64"] * 10
    assert rel < pages["norm_accuracy"]["fp32_tile_version_error_about"] * 1e-6


def test_nan_inf_semantics():
    a = np.array([1.0, 2.0, np.nan, 3.0, np.inf, -np.inf], np.float32)
    got = oracle.grad_norm([a, np.ones(3, np.float32)], max_norm=1.0)
    assert math.isnan(got["norm2"]) and math.isnan(got["norm_inf"])
    assert got["nan_count"] == 1 and got["inf_count"] == 2 and got["status"] == 1
    b = np.array([1.0, -np.inf, 2.0], np.float32)
    got = oracle.grad_norm([b])
    assert got["norm2"] == math.inf and got["norm_inf"] == math.inf
    assert got["nan_count"] == 0 and got["inf_count"] == 1 and got["status"] == 1
    # BF16 NaN / Inf codes
    c = np.array([0x7FC0, 0x3F80, 0xFF80], np.uint16)
    got = oracle.grad_norm([c])
    assert got["nan_count"] == 1 and got["inf_count"] == 1 and math.isnan(got["norm2"])


def test_clip_coefficient():
    assert oracle.clip_coef(0.5, 1.0) == 1.0
    assert oracle.clip_coef(1.0, 1.0) == np.float32(1.0 / (1.0 + 1e-6))  # the 1e-6 guard
    assert oracle.clip_coef(3.0, 0.0) == 1.0        # no clipping
    assert oracle.clip_coef(3.0, -1.0) == 1.0
    for norm in (2.0, 17.3, 1e6):
        c = oracle.clip_coef(norm, 1.0)
        assert c < 1.0
        assert c * (norm + 1e-6) == pytest.approx(1.0, rel=1e-7)
    got = oracle.grad_norm([np.full(100, 1.0, np.float32)], max_norm=2.0)
    assert got["norm2"] == 10.0
    assert got["clip_coef"] == np.float32(2.0 / (10.0 + 1e-6))
