"""Test harness: drive one workload through the CUDA library (via the Python
binding of the C ABI) and through the CPU oracle, on the same seeded inputs,
and compare.  Test infrastructure only."""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import precision_states_gb300 as ps
import workloads as W

ALGO = {"adamw": oracle.ADAMW, "ademamix": oracle.ADEMAMIX}


def hp_for(w: W.Workload, rounding="nearest", seed=1234, count=False):
    h = dict(lr=1e-3, beta1=0.9, beta2=0.999, beta3=0.9999, alpha=5.0, eps=1e-8, weight_decay=0.0)
    h.update(w.hp)
    gpu = ps.hparams(rounding=rounding, seed=seed, count_unchanged=count, **h)
    orc = oracle.hparams(**h)
    return gpu, orc


class GpuSide:
    """The workload's tensors on the GPU and a plan over them."""

    def __init__(self, w: W.Workload, seed: int = 0, device="cuda"):
        self.w, self.seed = w, seed
        self.params = W.make_params(w, device, seed)
        self.grads = W.make_grads(w, device, 1, seed)
        self.m = [W.state_storage(w.m_dtype, n, device) for n in w.sizes]
        self.v = [W.state_storage(w.v_dtype, n, device) for n in w.sizes]
        self.m2 = ([W.state_storage(w.m_dtype, n, device) for n in w.sizes]
                   if w.algo == "ademamix" else None)
        self.plan = ps.Plan(self.params, self.grads, self.m, self.v, self.m2,
                            m_dtype=w.m_dtype, v_dtype=w.v_dtype)

    def norm(self, max_norm: float):
        return self.plan.grad_norm(max_norm)

    def step(self, t: int, hp, clip: bool):
        d_norm = None
        if clip:
            self.plan.grad_norm(self.w.max_norm, sync=False)
            d_norm = self.plan.norm_buffer()
        if self.w.algo == "ademamix":
            self.plan.ademamix_step(hp, t, d_norm)
        else:
            self.plan.adamw_step(hp, t, d_norm)


class OracleSide:
    """Host copies of the sampled tensors, stepped by the oracle."""

    def __init__(self, gpu: GpuSide, indices):
        self.w = gpu.w
        self.idx = list(indices)
        self.p = [W.to_numpy_codes(gpu.params[i]) for i in self.idx]
        self.m = [W.to_numpy_codes(gpu.m[i]) for i in self.idx]
        self.v = [W.to_numpy_codes(gpu.v[i]) for i in self.idx]
        self.m2 = ([W.to_numpy_codes(gpu.m2[i]) for i in self.idx] if gpu.m2 is not None else None)

    def step(self, t: int, grads_np, ohp, coef: float, stochastic: bool, seed: int):
        """grads_np: host gradient arrays for the sampled tensors (same order)."""
        unchanged = 0
        for k, i in enumerate(self.idx):
            unchanged += oracle.adam_tensor(
                ALGO[self.w.algo], self.p[k], grads_np[k], self.m[k], self.v[k], ohp, t,
                m2=None if self.m2 is None else self.m2[k], m_dtype=self.w.m_dtype,
                v_dtype=self.w.v_dtype, coef=coef, stochastic=stochastic, seed=seed, tensor_index=i)
        return unchanged


def oracle_norm_parallel(grads_np, max_norm: float, threads: int = 16) -> dict:
    """The oracle's global norm, per-tensor sums computed on several host
    threads (the C calls release the GIL) and combined in list order -- the
    same result as oracle.grad_norm."""
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(oracle.tensor_sumsq, grads_np))
    return oracle.norm_finish(parts, max_norm)


def rel_err(a: float, b: float) -> float:
    if a == b:
        return 0.0
    return abs(a - b) / max(abs(b), 1e-300)


def assert_close_scaled(got: np.ndarray, want: np.ndarray, tol: float, what: str):
    """max |got - want| <= tol * (1 + |want|), elementwise."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, what
    bad = np.abs(got - want) > tol * (1.0 + np.abs(want))
    bad |= np.isnan(got) != np.isnan(want)
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} outside {tol}(1+|x|); "
                             f"first at {i}: got {got[i]!r} want {want[i]!r}")


def state_codes(arr: np.ndarray, dtype: str, n: int) -> np.ndarray:
    """Per-element integer codes of a host state array."""
    if dtype == "f32":
        return np.ascontiguousarray(arr).view(np.uint32)
    if dtype == "bf16":
        return arr.view(np.uint16).astype(np.uint32)
    if dtype == "e4m3":
        return arr.astype(np.uint32)
    codes = np.stack([arr & 0xF, arr >> 4], axis=1).ravel()[:n]
    return codes.astype(np.uint32)


_DECODE = {}


def decode(arr: np.ndarray, dtype: str, n: int) -> np.ndarray:
    """Exact fp64 values of a host state array (for tolerance checks)."""
    if dtype == "f32":
        return arr.astype(np.float64)
    if dtype == "bf16":
        return (arr.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype not in _DECODE:
        fn = oracle.e4m3_decode if dtype == "e4m3" else oracle.e2m2_decode
        _DECODE[dtype] = np.array([fn(c) for c in range(256 if dtype == "e4m3" else 16)])
    return _DECODE[dtype][state_codes(arr, dtype, n)]


def compare_codes(got: np.ndarray, want: np.ndarray, dtype: str, n: int, exact: bool, what: str):
    """Low-precision state parity: identical codes (stochastic rounding), or
    >= 99.99 % identical with every differing code one grid step off
    (nearest)."""
    g = state_codes(got, dtype, n)
    w_ = state_codes(want, dtype, n)
    diff = g != w_
    if exact:
        assert not diff.any(), f"{what}: {int(diff.sum())} of {n} codes differ (first at {int(np.argmax(diff))})"
        return
    frac = 1.0 - diff.mean() if n else 1.0
    assert frac >= 0.9999, f"{what}: only {frac:.6f} identical"
    if diff.any():
        gi = g[diff].astype(np.int64)
        wi = w_[diff].astype(np.int64)
        assert np.all(np.abs(gi - wi) == 1), f"{what}: differing codes more than one step apart"
