"""Pins for the oracle's LAMB-style update-norm clipping (reading of
"Investigate SM103 bias-correction broadcast in 32-bit optimizers",
'Problem' / 'B300 result': the max_unorm path measures a tensor's whole
update before applying it)."""
import math

import numpy as np
import pytest

import oracle


def f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


def test_no_clip_equals_adamw():
    """max_unorm <= 0, or a bound never reached: exactly the AdamW step."""
    rng = np.random.default_rng(40)
    n = 777
    hp = oracle.hparams(lr=1e-2, weight_decay=0.1)
    for max_unorm in (0.0, 1e9):
        p1, p2 = f32(rng.standard_normal(n)), None
        p2 = p1.copy()
        m1, v1, m2, v2 = (np.zeros(n, np.float32) for _ in range(4))
        for t in range(1, 6):
            g = f32(rng.standard_normal(n))
            r = oracle.lamb_tensor(p1, g, m1, v1, hp, t, max_unorm)
            assert r == 1.0
            oracle.adam_tensor(oracle.ADAMW, p2, g, m2, v2, hp, t)
        assert np.array_equal(m1, m2) and np.array_equal(v1, v2)
        assert np.max(np.abs(p1.astype(np.float64) - p2)) <= 1e-7 * np.max(np.abs(p2))


def test_constant_gradient_closed_form():
    """With g constant the direction is exactly g/(|g|+eps) at every step, so
    |u| = sqrt(sum (g/(|g|+eps))^2), the ratio is max_unorm |p_t| / |u| while
    that is below 1, and p follows by unrolling."""
    rng = np.random.default_rng(41)
    n, T = 300, 6
    hp = oracle.hparams(lr=1e-2, weight_decay=0.1, eps=1e-8)
    lr, wd, eps = (float(np.float32(x)) for x in (1e-2, 0.1, 1e-8))
    g = f32(rng.choice([-1.0, 1.0], n) * rng.uniform(0.5, 2.0, n))
    p = f32(rng.standard_normal(n) * 0.01)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    want = p.astype(np.float64)
    u = g.astype(np.float64) / (np.abs(g.astype(np.float64)) + eps)
    max_unorm = 0.05
    for t in range(1, T + 1):
        ratio = min(1.0, max_unorm * np.linalg.norm(want) / np.linalg.norm(u))
        got = oracle.lamb_tensor(p, g, m, v, hp, t, max_unorm)
        assert got == pytest.approx(ratio, rel=1e-6)
        assert ratio < 1.0
        want = want * (1 - lr * wd) - lr * ratio * u
    assert np.max(np.abs(p - want)) < 1e-6 * np.max(np.abs(want)) + 1e-9


def test_ratio_scales_the_update_only():
    """The decay term is not scaled: with a tiny bound the step is almost
    pure decay-first weight decay."""
    rng = np.random.default_rng(42)
    n = 128
    hp = oracle.hparams(lr=0.1, weight_decay=0.1)
    p0 = f32(rng.standard_normal(n))
    p = p0.copy()
    r = oracle.lamb_tensor(p, f32(rng.standard_normal(n)), np.zeros(n, np.float32),
                           np.zeros(n, np.float32), hp, 1, 1e-9)
    assert r < 1e-6
    assert np.allclose(p, p0 * np.float32(1 - 0.1 * 0.1), rtol=1e-6, atol=1e-7)
