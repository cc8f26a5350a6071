"""Pins for the analytic stalling model ("When Small Updates Disappear",
sec. 2.3 and 3.2) and a loose check that the oracle's low-precision step
stalls at about the predicted rate (sec. 4: the model is within 2.8 points
of measurements)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import stall_model as sm


def test_printed_predictions(pages):
    pr = pages["stall_predictions_beta2_0p999"]
    b2 = pr["beta2"]
    p = sm.FRACTION_BITS
    assert round(sm.stall_nearest(b2, p["bf16"]), 3) == pr["bf16_nearest"]
    assert round(sm.stall_stochastic(b2, p["bf16"]), 3) == pr["bf16_stochastic"]
    assert round(sm.stall_stochastic(b2, p["e4m3"]), 3) == pr["fp8_stochastic"]
    assert round(sm.stall_stochastic(b2, p["e2m2"]), 3) == pr["fp4_stochastic"]
    assert sm.stall_nearest(b2, p["e4m3"]) > 0.9999
    assert sm.stall_nearest(b2, p["e2m2"]) > 0.9999


def test_model_monotone_in_beta2_and_bits():
    """sec. 2.3: pushing b2 toward one or removing fraction bits grows the
    stalling interval."""
    assert sm.stall_nearest(0.99, 7) < sm.stall_nearest(0.999, 7) < sm.stall_nearest(0.9999, 7)
    assert sm.stall_stochastic(0.999, 7) < sm.stall_stochastic(0.999, 3) < sm.stall_stochastic(0.999, 2)


@pytest.mark.parametrize("stochastic,model", [(False, sm.stall_nearest(0.999, 7)),
                                              (True, sm.stall_stochastic(0.999, 7))])
def test_oracle_bf16_stall_fraction_near_model(stochastic, model):
    n, steps = 20000, 60
    rng = np.random.default_rng(20)
    hp = oracle.hparams(lr=1e-3, beta2=0.999)
    p = np.zeros(n, np.float32)
    m = np.zeros(n, np.uint16)
    v = torch.ones(n).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    fr = []
    for t in range(1, steps + 1):
        g = torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(torch.bfloat16)
        g = g.view(torch.int16).numpy().view(np.uint16).copy()
        same = oracle.adam_tensor(oracle.ADAMW, p, g, m, v, hp, t + 1000, m_dtype="bf16",
                                  v_dtype="bf16", stochastic=stochastic, seed=3)
        fr.append(same / n)
    # loose: the model drops the mantissa's spread and the state's drift
    assert abs(np.mean(fr[10:]) - model) < 0.04
