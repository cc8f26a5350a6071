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

    def __init__(self, w: W.Workload, seed: int = 0, device="cuda", v_scale=None):
        self.w, self.seed = w, seed
        self.v_scale = v_scale
        self.params = W.make_params(w, device, seed)
        self.grads = W.make_grads(w, device, 1, seed)
        self.m = [W.state_storage(w.m_dtype, n, device) for n in w.sizes]
        self.v = [W.state_storage(w.v_dtype, n, device) for n in w.sizes]
        self.m2 = ([W.state_storage(w.m_dtype, n, device) for n in w.sizes]
                   if w.algo == "ademamix" else None)
        self.plan = ps.Plan(self.params, self.grads, self.m, self.v, self.m2,
                            m_dtype=w.m_dtype, v_dtype=w.v_dtype, v_scale=v_scale)

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
    """Host copies of sampled tensors or slices, stepped by the oracle.

    `samples` holds tensor indices (the whole tensor) or (index, start, n)
    slices; start must be even (E2M2 packs two codes per byte).  Element k of
    a slice is element start + k of its tensor, which selects its
    stochastic-rounding draws."""

    def __init__(self, gpu: GpuSide, samples, track_moves: bool = False):
        self.w = gpu.w
        self.v_scale = gpu.v_scale
        self.samples = [(s, 0, gpu.w.sizes[s]) if isinstance(s, int) else tuple(s) for s in samples]
        self.idx = [i for i, _, _ in self.samples]
        self.p = [W.to_numpy_codes(self.cut(gpu.params, k, "f32")) for k in range(len(self.samples))]
        # with track_moves: per element, the sums over steps of |p_t - p_(t-1)|
        # and of max(|p_(t-1)|, |p_t|) in the oracle (see update_bound)
        self.moved = [np.zeros(a.size) for a in self.p] if track_moves else None
        self.mag = [np.zeros(a.size) for a in self.p] if track_moves else None
        self.m = [W.to_numpy_codes(self.cut(gpu.m, k, self.w.m_dtype)) for k in range(len(self.samples))]
        self.v = [W.to_numpy_codes(self.cut(gpu.v, k, self.w.v_dtype)) for k in range(len(self.samples))]
        self.m2 = ([W.to_numpy_codes(self.cut(gpu.m2, k, self.w.m_dtype)) for k in range(len(self.samples))]
                   if gpu.m2 is not None else None)

    def cut(self, tensors, k, dtype):
        """The part of tensor list `tensors` that sample k covers."""
        i, start, n = self.samples[k]
        t = tensors[i]
        if dtype == "e2m2":
            assert start % 2 == 0
            return t[start // 2:(start + n + 1) // 2]
        return t[start:start + n]

    def grads(self, gpu_grads):
        return [W.to_numpy_codes(self.cut(gpu_grads, k, "grad")) for k in range(len(self.samples))]

    def step(self, t: int, grads_np, ohp, coef: float, stochastic: bool, seed: int, threads: int = 1):
        """grads_np: host gradient arrays for the samples (same order).  With
        threads > 1 the samples are stepped concurrently (each is its own
        host array and the C calls release the GIL); the per-element results
        do not depend on it."""
        def one(k):
            i, start, n = self.samples[k]
            return oracle.adam_tensor(
                ALGO[self.w.algo], self.p[k], grads_np[k], self.m[k], self.v[k], ohp, t,
                m2=None if self.m2 is None else self.m2[k], m_dtype=self.w.m_dtype,
                v_dtype=self.w.v_dtype, coef=coef, stochastic=stochastic, seed=seed, tensor_index=i,
                index_base=start, v_scale=1.0 if self.v_scale is None else self.v_scale[i])
        before = [a.astype(np.float64) for a in self.p] if self.moved is not None else None
        if threads <= 1:
            same = sum(one(k) for k in range(len(self.samples)))
        else:
            with ThreadPoolExecutor(max_workers=threads) as ex:
                same = sum(ex.map(one, range(len(self.samples))))
        if before is not None:
            for k, b in enumerate(before):
                now = self.p[k].astype(np.float64)
                self.moved[k] += np.abs(now - b)
                self.mag[k] += np.maximum(np.abs(now), np.abs(b))
        return same

    def compare(self, gpu: GpuSide, tol: float, exact_codes: bool, steps: int = 0):
        """FP32 values within tol (1+|x|) -- for p past 100 steps, when moves
        are tracked, plus update_bound; low-precision codes identical
        (exact_codes) or >= 99.99 % identical and one step off."""
        w = self.w
        for k, (i, start, n) in enumerate(self.samples):
            what = f"tensor {i} [{start}:{start + n}]"
            extra = update_bound(self.moved[k], self.mag[k]) if self.moved is not None and steps > 100 else None
            assert_close_scaled(W.to_numpy_codes(self.cut(gpu.params, k, "f32")), self.p[k], tol, "p " + what,
                                extra)
            gm = W.to_numpy_codes(self.cut(gpu.m, k, w.m_dtype))
            gv = W.to_numpy_codes(self.cut(gpu.v, k, w.v_dtype))
            if w.m_dtype == "f32":
                assert_close_scaled(gm, self.m[k], tol, "m " + what)
                assert_close_scaled(gv, self.v[k], tol, "v " + what)
            else:
                compare_codes(gm, self.m[k], "bf16", n, exact=exact_codes, what="m " + what)
                compare_codes(gv, self.v[k], w.v_dtype, n, exact=exact_codes, what="v " + what)
            if self.m2 is not None:
                assert_close_scaled(W.to_numpy_codes(self.cut(gpu.m2, k, w.m_dtype)), self.m2[k], tol,
                                    "m2 " + what)


def fp32_tol(t: int) -> float:
    """Tolerance on FP32 values, scaled as tol * (1 + |x|), after t steps.

    1e-6 after one step and 1e-5 up to 100 steps are the stated bounds.  Past
    100 steps the dominant difference is systematic: the kernel multiplies p
    by the decay factor 1 - lr wd rounded once to fp32 (at most 2^-25 off,
    relative, for a factor in [1/2, 1)), the oracle by the factor in double,
    so after t steps p differs by up to t 2^-25 relative from that alone.
    The bound adds that term: 1e-5 + t 2^-25 (4.0e-5 at t = 1000)."""
    if t <= 1:
        return 1e-6
    if t <= 100:
        return 1e-5
    return 1e-5 + t * 2.0 ** -25


def update_bound(moved: np.ndarray, mag: np.ndarray) -> np.ndarray:
    """Second term of the FP32 bound on p past 100 steps, per element.

    Each step the kernel forms the update lr u in fp32 with the approximate
    square root and reciprocal of sm_103a (a few ulp in all), and rounds
    p (1 - lr wd), lr u and their difference separately; the oracle computes
    the step in double and rounds p once.  So every step can put p up to
    about 2^-21 |lr u| + 1.5 ulp(max(|p_(t-1)|, |p_t|)) away from the oracle,
    and the differences stay when p later shrinks.  Where a low-precision v
    sits at zero (unscaled E4M3 / E2M2 v below half its first grid step) the
    update is m / (sqrt(v_t) + eps) with v_t from the current gradient alone,
    and both the update and p can grow far beyond p's start.  The bound is
    2^-20 times the oracle's own sum over steps of |p_t - p_(t-1)| (`moved`)
    plus 2^-22 times its sum of max(|p_(t-1)|, |p_t|) (`mag`)."""
    return moved * 2.0 ** -20 + mag * 2.0 ** -22


def run_lockstep(w, steps, tol, samples=None, rounding="nearest", seed=0, hp_seed=77, count=False,
                 checkpoints=(), norm_threads=16, gpu=None, step_threads=1, track_moves=False):
    """Run `steps` steps of workload `w` on the GPU (whole list, clip from the
    GPU's own norm when w.max_norm > 0) and on the oracle (its own norm over
    every gradient, the step on `samples`), comparing the norms every step and
    the sampled states at each checkpoint and at the end.  `tol` is a number,
    or a function of the step count (such as fp32_tol)."""
    tol_at = tol if callable(tol) else (lambda _t: tol)
    gpu = gpu or GpuSide(w, seed=seed)
    orc = OracleSide(gpu, range(len(w.sizes)) if samples is None else samples, track_moves=track_moves)
    ghp, ohp = hp_for(w, rounding=rounding, seed=hp_seed, count=count)
    sr = rounding == "stochastic"
    clip = w.max_norm > 0
    counts = []
    for t in range(1, steps + 1):
        W.fill_grads(w, gpu.grads, t, seed)
        coef = 1.0
        if clip:
            all_np = [W.to_numpy_codes(g) for g in gpu.grads]
            want = oracle_norm_parallel(all_np, w.max_norm, norm_threads)
            got = gpu.plan.grad_norm(w.max_norm)
            assert rel_err(got.norm2, want["norm2"]) <= 1e-12, (t, got.norm2, want["norm2"])
            assert got.clip_coef == want["clip_coef"], t
            coef = want["clip_coef"]
            del all_np
        g_np = orc.grads(gpu.grads)
        gpu.step(t, ghp, clip)
        same = orc.step(t, g_np, ohp, coef, sr, hp_seed, threads=step_threads)
        if count:
            counts.append((gpu.plan.unchanged_count(), same))
        if t in checkpoints:
            torch.cuda.synchronize()
            orc.compare(gpu, tol_at(t), sr, steps=t)
    torch.cuda.synchronize()
    orc.compare(gpu, tol_at(steps), sr, steps=steps)
    assert gpu.plan.status() == 0, "a kernel reported a bounded wait that ran out"
    return gpu, orc, counts


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


def assert_close_scaled(got: np.ndarray, want: np.ndarray, tol: float, what: str, extra=None):
    """|got - want| <= tol * (1 + |want|) (+ extra, per element), elementwise."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, what
    bound = tol * (1.0 + np.abs(want))
    if extra is not None:
        bound = bound + extra
    bad = np.abs(got - want) > bound
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
