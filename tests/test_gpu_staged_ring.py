"""The staged step's ring over many tiles per CTA.

With a few tiles per CTA the ring's stages are filled once or twice, and the
consumer warps cannot drift apart.  Here each of the 304 persistent CTAs
takes about thirty tiles, so every stage is refilled many times, in every
mode the staged kernel serves (BF16 v, and stochastic E4M3 / E2M2 v, where a
consumer warp owns a slice of some tiles only): no bounded wait may run out
(the harness reads the plan's status after the last step), and the sampled
codes and values must match the oracle after 1 and 10 steps."""
import numpy as np
import pytest

import workloads as W
from harness import fp32_tol, run_lockstep

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("v_dtype,rounding", [("bf16", "nearest"), ("bf16", "stochastic"),
                                              ("e4m3", "stochastic"), ("e2m2", "stochastic")])
def test_staged_ring_many_tiles_per_cta(v_dtype, rounding):
    sizes = [19_000_017, 1_048_583, 4097, 1]
    w = W.Workload("ring", sizes, "bf16", m_dtype="bf16", v_dtype=v_dtype, steps=10, max_norm=1.0,
                   p_std=0.02, grad_std=1.0, hp=dict(lr=1e-3, weight_decay=0.1))
    rng = np.random.default_rng(12)
    samples = [(0, int(rng.integers(0, (sizes[0] - 8192) // 2)) * 2, 8192),
               (0, sizes[0] - 4097, 4097), (1, 0, 8192), 2, 3]
    run_lockstep(w, w.steps, fp32_tol, samples=samples, rounding=rounding, checkpoints=(1,))
