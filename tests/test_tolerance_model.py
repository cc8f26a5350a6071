"""The FP32 tolerance the long GPU parity runs use (fp32_tol and
update_bound in harness.py), checked on the CPU against an emulation of the
kernel's arithmetic: fp32 moments in the order of the definition, the update
term and p's update as separately rounded fp32 operations (square root and
division correctly rounded here; the kernel's approximate ones add a few ulp,
which the bound's 2^-20 factor on the moves leaves room for).  The oracle
computes the step in double and rounds p once.

The workload is the low-precision GPT-2 one on a single 768-element tensor,
BF16 m and unscaled E2M2 or E4M3 v with nearest rounding, 1,000 steps: the
regime where v sits at zero and the updates explode, so p strays far from its
start and comes back."""
import numpy as np
import pytest

import oracle
import workloads as W
from harness import fp32_tol, update_bound

f32 = np.float32


def emulate(v_dtype: str, steps: int, checkpoints):
    n = 768
    w = W.workload("lowp_gpt2", sizes=[n])
    w.m_dtype, w.v_dtype = "bf16", v_dtype
    p = W.to_numpy_codes(W.make_params(w, "cpu", 0)[0]).copy()
    pk = p.copy()                                   # the emulated kernel's p
    m = W.to_numpy_codes(W.state_storage("bf16", n, "cpu")).copy()
    v = W.to_numpy_codes(W.state_storage(v_dtype, n, "cpu")).copy()
    ohp = oracle.hparams(lr=1e-3, weight_decay=0.1, beta1=0.9, beta2=0.999)
    lr, wd, b1, b2, eps = f32(1e-3), f32(0.1), f32(0.9), f32(0.999), f32(1e-8)
    decay = f32(1.0 - float(lr) * float(wd))
    omb1, omb2 = f32(1.0 - float(b1)), f32(1.0 - float(b2))
    if v_dtype == "e2m2":
        table = np.array([oracle.e2m2_decode(c) for c in range(16)], dtype=np.float32)
    else:
        table = np.array([oracle.e4m3_decode(c) for c in range(256)], dtype=np.float32)
    moved, mag = np.zeros(n), np.zeros(n)
    out = {}
    for t in range(1, steps + 1):
        g = W.to_numpy_codes(W.make_grads(w, "cpu", t, 0)[0])
        gf = (g.astype(np.uint32) << 16).view(np.float32)
        md = (m.astype(np.uint32) << 16).view(np.float32)
        codes = np.stack([v & 0xF, v >> 4], axis=1).ravel()[:n] if v_dtype == "e2m2" else v
        vd = table[codes]
        mf = f32(b1 * md) + f32(omb1 * gf)
        vf = f32(b2 * vd) + f32(omb2 * f32(gf * gf))
        inv_bc1 = f32(1.0 / (1.0 - float(b1) ** t))
        inv_bc2 = f32(1.0 / (1.0 - float(b2) ** t))
        den = np.sqrt(f32(vf * inv_bc2)).astype(np.float32) + eps
        u = (f32(mf * inv_bc1) / den).astype(np.float32)
        pk = (f32(pk * decay) - f32(lr * u)).astype(np.float32)
        before = p.astype(np.float64)
        oracle.adam_tensor(oracle.ADAMW, p, g, m, v, ohp, t, m_dtype="bf16", v_dtype=v_dtype)
        now = p.astype(np.float64)
        moved += np.abs(now - before)
        mag += np.maximum(np.abs(now), np.abs(before))
        if t in checkpoints:
            out[t] = (pk.astype(np.float64), now.copy(), moved.copy(), mag.copy())
    return out


@pytest.mark.parametrize("v_dtype", ["e2m2", "e4m3"])
def test_long_run_fp32_bound_covers_the_kernel_arithmetic(v_dtype):
    res = emulate(v_dtype, 1000, (1, 100, 500, 1000))
    for t, (pk, po, moved, mag) in res.items():
        bound = fp32_tol(t) * (1.0 + np.abs(po))
        if t > 100:
            bound = bound + update_bound(moved, mag)
        diff = np.abs(pk - po)
        assert np.all(diff <= bound), (t, float(diff.max()), float((diff / bound).max()))
    # the run is the degenerate one the bound is for: p strays far from its start
    assert res[1000][3].max() > 1e3 * 0.02
