"""GPU parity of opt_grad_norm with the oracle: relative error <= 1e-12,
bit-identical repeats, NaN/Inf counts and status, the exact slow path for
extreme magnitudes, dtype buckets, empty and ragged lists."""
import math

import numpy as np
import pytest
import torch

import oracle
import precision_states_gb300 as ps
import workloads as W
from harness import oracle_norm_parallel, rel_err

pytestmark = pytest.mark.gpu

TOL = 1e-12


def plan_for(grads):
    params = [torch.zeros(g.numel(), device="cuda") for g in grads]
    m = [torch.zeros(g.numel(), device="cuda") for g in grads]
    v = [torch.zeros(g.numel(), device="cuda") for g in grads]
    return ps.Plan(params, grads, m, v)


def host(grads):
    return [W.to_numpy_codes(g) for g in grads]


def check(grads, max_norm=1.0):
    plan = plan_for(grads)
    got = plan.grad_norm(max_norm)
    want = oracle.grad_norm(host(grads), max_norm)
    assert got.nan_count == want["nan_count"] and got.inf_count == want["inf_count"]
    assert got.status == want["status"]
    if want["status"] == 0:
        assert rel_err(got.norm2, want["norm2"]) <= TOL, (got.norm2, want["norm2"])
        assert rel_err(got.sumsq, want["sumsq"]) <= 2 * TOL
        assert got.norm_inf == want["norm_inf"]
        assert got.clip_coef == want["clip_coef"]
    else:
        for k in ("norm2", "norm_inf"):
            a, b = getattr(got, k), want[k]
            assert (math.isnan(a) and math.isnan(b)) or a == b, k
    return plan, got


@pytest.mark.parametrize("gdt", ["bf16", "f32"])
def test_sweep_sizes(gdt):
    w = W.workload("sweep", grad_dtype=gdt)
    grads = W.make_grads(w, "cuda", step=1, seed=3)
    check(grads)


def test_mixed_dtype_buckets():
    w = W.workload("sweep")
    g16 = W.make_grads(w, "cuda", step=1, seed=4)
    g32 = W.make_grads(W.workload("sweep", grad_dtype="f32"), "cuda", step=1, seed=5)
    mixed = [g16[i] if i % 3 else g32[i] for i in range(len(g16))]
    check(mixed)


def test_repeatable_bitwise():
    w = W.workload("clip_740")
    grads = W.make_grads(w, "cuda", step=1, seed=6)
    plan = plan_for(grads)
    a = plan.grad_norm(1.0).as_dict()
    for _ in range(3):
        assert plan.grad_norm(1.0).as_dict() == a


def test_clip740_full_size():
    w = W.workload("clip_740")
    grads = W.make_grads(w, "cuda", step=1, seed=7)
    plan = plan_for(grads)
    got = plan.grad_norm(w.max_norm)
    want = oracle_norm_parallel(host(grads), w.max_norm)
    assert rel_err(got.norm2, want["norm2"]) <= TOL
    assert got.norm_inf == want["norm_inf"] and got.clip_coef == want["clip_coef"]


@pytest.mark.parametrize("kinds", [("nan", "+inf", "-inf"), ("nan",), ("+inf",), ("-inf",)])
def test_nonfinite_run(kinds):
    w = W.workload("clip_740")
    grads = W.make_grads(w, "cuda", step=1, seed=8)
    touched = W.inject_nonfinite(grads, seed=21, kinds=kinds)
    assert len(touched) == 7
    _, got = check(grads)
    assert got.status == ps.OPT_ENONFINITE


@pytest.mark.parametrize("gdt", ["bf16", "f32"])
def test_extreme_magnitudes_slow_path(gdt):
    rng = np.random.default_rng(11)
    dt = torch.bfloat16 if gdt == "bf16" else torch.float32
    vals = [np.full(1000, 3.0e30), rng.standard_normal(5000) * 1e-30, np.full(17, 1e-38),
            rng.standard_normal(70001), np.array([1e-45, 2e38, -3e38, 1e-20])]
    grads = [torch.from_numpy(v.astype(np.float32)).to(dt).cuda() for v in vals]
    check(grads, max_norm=0.0)
    # tiny-only list: every chunk on the exact path
    check([torch.from_numpy((rng.standard_normal(9999) * 1e-25).astype(np.float32)).to(dt).cuda()], 0.0)


def test_empty_and_zero_sized():
    plan = ps.Plan([], [], [], [])
    r = plan.grad_norm(1.0)
    assert r.norm2 == 0.0 and r.norm_inf == 0.0 and r.status == 0 and r.clip_coef == 1.0
    z = torch.zeros(0, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(5, dtype=torch.bfloat16, device="cuda")
    _, r = check([z, g, z])
    assert r.norm2 == math.sqrt(5.0)


def test_all_zero_and_no_clip():
    grads = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for n in (1, 33, 70000)]
    _, r = check(grads, max_norm=0.0)
    assert r.norm2 == 0.0 and r.clip_coef == 1.0


@pytest.mark.parametrize("mixed", [False, True])
def test_every_call_finishes_into_its_output(mixed):
    """The finish runs in the CTA that completes last and resets the
    completion counter; a counter left behind would skip the next finish and
    leave the old result in place.  Each call here writes into a buffer
    filled with a sentinel, on gradients scaled by 2^k since the last call:
    scaling by a power of two is exact, so the sum of squares scales by 4^k
    exactly and the result must follow bit for bit."""
    w = W.workload("sweep")
    grads = W.make_grads(w, "cuda", step=1, seed=41)
    if mixed:
        g32 = W.make_grads(W.workload("sweep", grad_dtype="f32"), "cuda", step=1, seed=42)
        grads = [grads[i] if i % 3 else g32[i] for i in range(len(grads))]
    plan = plan_for(grads)
    d_out = torch.empty(6, dtype=torch.float64, device="cuda")
    base = None
    for k in range(4):
        d_out.fill_(float("nan"))
        plan.grad_norm(1.0, d_out=d_out.data_ptr(), sync=False)
        torch.cuda.synchronize()
        r = ps.opt_norm_result.from_buffer_copy(d_out.cpu().numpy().tobytes())
        assert r.status == 0
        if base is None:
            want = oracle.grad_norm(host(grads), 1.0)
            assert rel_err(r.norm2, want["norm2"]) <= TOL
            base = r
        else:
            assert r.sumsq == base.sumsq * 4.0 ** k and r.norm2 == base.norm2 * 2.0 ** k
            assert r.norm_inf == base.norm_inf * 2.0 ** k
        for g in grads:
            g.mul_(2.0)
    plan.close()


def test_two_plans_on_two_streams_concurrently():
    """Each plan owns its slots and its completion counter, so norms of two
    plans issued on two streams at the same time finish independently; each
    result equals the oracle's for its own list, for several rounds."""
    wa, wb = W.workload("clip_740"), W.workload("sweep")
    ga = W.make_grads(wa, "cuda", step=1, seed=51)
    gb = W.make_grads(wb, "cuda", step=1, seed=52)
    pa, pb = plan_for(ga), plan_for(gb)
    want_a = oracle_norm_parallel(host(ga), 1.0)
    want_b = oracle.grad_norm(host(gb), 1.0)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = [(torch.full((6,), float("nan"), dtype=torch.float64, device="cuda"),
             torch.full((6,), float("nan"), dtype=torch.float64, device="cuda")) for _ in range(4)]
    torch.cuda.synchronize()
    for da, db in outs:
        pa.grad_norm(1.0, d_out=da.data_ptr(), sync=False, stream=sa)
        pb.grad_norm(1.0, d_out=db.data_ptr(), sync=False, stream=sb)
    torch.cuda.synchronize()
    for da, db in outs:
        ra = ps.opt_norm_result.from_buffer_copy(da.cpu().numpy().tobytes())
        rb = ps.opt_norm_result.from_buffer_copy(db.cpu().numpy().tobytes())
        assert rel_err(ra.norm2, want_a["norm2"]) <= TOL and ra.clip_coef == want_a["clip_coef"]
        assert rel_err(rb.norm2, want_b["norm2"]) <= TOL and rb.clip_coef == want_b["clip_coef"]
    pa.close()
    pb.close()


def _noalloc_norm(grads, max_norm, d_out):
    import ctypes
    n = len(grads)
    numel = (ctypes.c_int64 * max(n, 1))(*[g.numel() for g in grads])
    ptrs = (ctypes.c_void_p * max(n, 1))(*[g.data_ptr() for g in grads])
    dts = (ctypes.c_int32 * max(n, 1))(*[ps.OPT_BF16 if g.dtype == torch.bfloat16 else ps.OPT_F32 for g in grads])
    assert ps.lib().opt_grad_norm_noalloc(n, numel, ptrs, dts, max_norm, d_out.data_ptr(), None) == ps.OPT_OK
    torch.cuda.synchronize()
    return ps.opt_norm_result.from_buffer_copy(bytes(d_out.cpu().numpy()))


@pytest.mark.parametrize("name", ["clip_740", "llama3_8b", "mixed", "tier8k", "mid"])
def test_norm_counts_every_element_once(name):
    """Every gradient element enters the norm exactly once, over whole lists:
    with BF16 gradients all 1 and FP32 gradients all 2, the sum of squares is
    an integer (exact in the float-float and fp64 accumulators) and must equal
    N_bf16 + 4 N_f32; a chunk skipped, summed twice or counted in the wrong
    bucket changes it by at least 1.  The plan and the no-allocation paths
    both."""
    if name == "mixed":
        sizes = [32768 * 3 + 5, 1, 70001, 32768, 32767, 4097, 0, 9]
        dts = [torch.bfloat16 if i % 2 == 0 else torch.float32 for i in range(len(sizes))]
    elif name == "tier8k":   # a BF16 bucket of 2^28 elements and more: 8K-element chunks
        sizes = [(1 << 28) - 4093, 8195, 9, 4096]
        dts = [torch.bfloat16] * len(sizes)
        assert ps.opt_norm_chunk_elems(sizes, [ps.OPT_BF16] * 4, 1) == 8192
    elif name == "mid":      # a BF16 bucket of 2^29 elements and more: 16K-element chunks
        sizes = [(1 << 29) - 4099, 12345, 7, 4097]
        dts = [torch.bfloat16] * len(sizes)
        assert ps.opt_norm_chunk_elems(sizes, [ps.OPT_BF16] * 4, 1) == 16384
    else:
        w = W.workload(name)
        sizes = w.sizes
        dts = [torch.bfloat16] * len(sizes)
    grads = [torch.full((n,), 1.0 if dt == torch.bfloat16 else 2.0, dtype=dt, device="cuda")
             for n, dt in zip(sizes, dts)]
    want = float(sum(n if dt == torch.bfloat16 else 4 * n for n, dt in zip(sizes, dts)))
    assert want < 2.0 ** 53
    plan = plan_for(grads)
    got = plan.grad_norm(0.0)
    assert got.sumsq == want and got.norm2 == math.sqrt(want), (got.sumsq, want)
    assert got.norm_inf == (2.0 if torch.float32 in dts else 1.0)
    assert got.nan_count == 0 and got.inf_count == 0 and got.status == 0
    plan.close()
    del plan
    torch.cuda.empty_cache()
    d_out = torch.zeros(48, dtype=torch.uint8, device="cuda")
    na = _noalloc_norm(grads, 0.0, d_out)
    assert na.sumsq == want and na.norm_inf == got.norm_inf


def test_mid_size_chunks_match_the_oracle():
    """A BF16 bucket just over 2^29 elements takes the middle chunk size
    (16,384): the norm of seeded values equals the oracle's within 1e-12,
    repeats bit for bit, and the no-allocation path gives the same bits."""
    sizes = [(1 << 28) + 3, (1 << 28) + 77, 5]
    assert ps.opt_norm_chunk_elems(sizes, [ps.OPT_BF16] * 3, 1) == 16384
    gen = torch.Generator(device="cuda").manual_seed(29)
    grads = [(torch.randn(n, generator=gen, device="cuda") * s).to(torch.bfloat16)
             for n, s in zip(sizes, (1e-3, 2.0, 1e4))]
    plan = plan_for(grads)
    got = plan.grad_norm(1.0)
    again = plan.grad_norm(1.0)
    assert again.as_dict() == got.as_dict()
    want = oracle_norm_parallel(host(grads), 1.0, 16)
    assert rel_err(got.norm2, want["norm2"]) <= TOL, (got.norm2, want["norm2"])
    assert got.norm_inf == want["norm_inf"] and got.clip_coef == want["clip_coef"]
    plan.close()
    del plan
    torch.cuda.empty_cache()
    d_out = torch.zeros(48, dtype=torch.uint8, device="cuda")
    na = _noalloc_norm(grads, 1.0, d_out)
    assert na.sumsq == got.sumsq and na.norm2 == got.norm2 and na.clip_coef == got.clip_coef
