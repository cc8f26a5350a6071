"""GPU parity of the fused steps with the oracle on the size sweep (tile edges
and ragged tails): FP32 states within 1e-6 (1+|x|) after one step and 1e-5
(1+|x|) after 100 steps; low-precision state codes identical (stochastic
rounding) or >= 99.99 % identical, one step off (nearest); unchanged counts
exact; non-finite norm skips the step; the BF16 v invariant on the GPU."""
import numpy as np
import pytest
import torch

import oracle
import precision_states_gb300 as ps
import workloads as W
from harness import GpuSide, OracleSide, hp_for, run_lockstep

pytestmark = pytest.mark.gpu


def run_parity(w, steps, tol, rounding="nearest", clip=True, seed=0, count=False, check_every=None):
    if not clip:
        w.max_norm = 0.0
    checkpoints = range(check_every, steps + 1, check_every) if check_every else ()
    gpu, orc, counts = run_lockstep(w, steps, tol, rounding=rounding, seed=seed, count=count,
                                    checkpoints=checkpoints)
    for got, want in counts:
        assert got == want
    return gpu, orc


@pytest.mark.parametrize("algo", ["adamw", "ademamix"])
@pytest.mark.parametrize("gdt", ["bf16", "f32"])
def test_fp32_states_one_step(algo, gdt):
    w = W.workload("sweep", algo=algo, grad_dtype=gdt, hp=dict(lr=0.1, weight_decay=0.1))
    run_parity(w, 1, 1e-6)


@pytest.mark.parametrize("algo", ["adamw", "ademamix"])
def test_fp32_states_hundred_steps(algo):
    w = W.workload("sweep", algo=algo, hp=dict(lr=1e-2, weight_decay=0.1))
    run_parity(w, 100, 1e-5, check_every=25)


def test_adamw_1m_config():
    """The 1M-element AdamW workload itself: lr = wd = 0.1, 10 steps."""
    w = W.workload("adamw_1m")
    run_parity(w, 1, 1e-6, clip=False)
    run_parity(w, 10, 1e-5, clip=False)


@pytest.mark.parametrize("v_dtype", ["bf16", "e4m3", "e2m2"])
@pytest.mark.parametrize("rounding", ["nearest", "stochastic"])
@pytest.mark.parametrize("gdt", ["bf16", "f32"])
def test_lowp_states_codes(v_dtype, rounding, gdt):
    w = W.workload("sweep", grad_dtype=gdt, m_dtype="bf16", v_dtype=v_dtype,
                   hp=dict(lr=1e-3, weight_decay=0.1, beta2=0.999), sigma_decay_steps=12)
    run_parity(w, 12, 1e-6, rounding=rounding, count=True, check_every=4)


SHORT = [1, 3, 2049, 4097, 70001, 300001, 2052]   # seven tensors: the short-list launch shape (2052: a last group of four)


@pytest.mark.parametrize("v_dtype,rounding", [("f32", "nearest"), ("bf16", "nearest"), ("bf16", "stochastic"),
                                              ("e4m3", "nearest"), ("e4m3", "stochastic"),
                                              ("e2m2", "nearest"), ("e2m2", "stochastic")])
@pytest.mark.parametrize("gdt", ["bf16", "f32"])
def test_short_list_path(v_dtype, rounding, gdt):
    """A bucket of at most eight tensors and 4096 tiles takes the short-list
    launch shape (descriptors in the kernel parameters, one CTA per tile, two
    with FP32 states):
    parity with the oracle, clipped, with unchanged counts."""
    m_dtype = "f32" if v_dtype == "f32" else "bf16"
    w = W.workload("sweep", sizes=SHORT, grad_dtype=gdt, m_dtype=m_dtype, v_dtype=v_dtype,
                   hp=dict(lr=1e-3, weight_decay=0.1, beta2=0.999), sigma_decay_steps=6)
    run_parity(w, 6, 1e-5, rounding=rounding, count=v_dtype != "f32", check_every=3)


def test_short_list_path_ademamix():
    w = W.workload("sweep", sizes=SHORT, algo="ademamix", hp=dict(lr=1e-2, weight_decay=0.1))
    run_parity(w, 1, 1e-6)
    run_parity(w, 5, 1e-5)


@pytest.mark.parametrize("v_dtype,rounding", [("f32", "nearest"), ("bf16", "stochastic"), ("e4m3", "nearest"),
                                              ("e2m2", "stochastic")])
def test_short_and_persistent_shapes_agree_bitwise(v_dtype, rounding):
    """The same seven tensors stepped alone (short-list shape) and with three
    one-element tensors appended (ten tensors: the persistent kernel) end
    with the same bits in p, m and v (no clipping: the extra tensors would
    change the norm)."""
    m_dtype = "f32" if v_dtype == "f32" else "bf16"
    out = []
    for sizes in (SHORT, SHORT + [1, 1, 1]):
        w = W.workload("sweep", sizes=sizes, m_dtype=m_dtype, v_dtype=v_dtype,
                       hp=dict(lr=1e-3, weight_decay=0.1), sigma_decay_steps=4)
        gpu = GpuSide(w, seed=11)
        ghp, _ = hp_for(w, rounding=rounding, seed=5)
        for t in range(1, 5):
            W.fill_grads(w, gpu.grads, t, 11)
            gpu.step(t, ghp, clip=False)
        torch.cuda.synchronize()
        out.append([x.clone() for x in gpu.params[:7] + gpu.m[:7] + gpu.v[:7]])
    for a, b in zip(*out):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_nonfinite_norm_skips_step():
    w = W.workload("clip_740")
    gpu = GpuSide(w, seed=3)
    W.inject_nonfinite(gpu.grads, seed=5)
    before = [t.clone() for t in gpu.params + gpu.m + gpu.v]
    ghp, _ = hp_for(w)
    r = gpu.plan.grad_norm(w.max_norm)
    assert r.status == ps.OPT_ENONFINITE
    gpu.step(1, ghp, clip=True)
    torch.cuda.synchronize()
    for a, b in zip(before, gpu.params + gpu.m + gpu.v):
        assert torch.equal(a, b)


@pytest.mark.parametrize("v_dtype", ["bf16", "e4m3", "e2m2"])
@pytest.mark.parametrize("rounding", ["nearest", "stochastic"])
def test_lowp_nonfinite_grads_without_clip(v_dtype, rounding):
    """Without clipping, NaN and +-Inf gradients go into the states as the
    codecs define (reading: plain AdamW propagates them): BF16 keeps NaN
    and Inf, E4M3 stores NaN as 0x7F and saturates Inf to 448, E2M2 stores
    NaN and Inf as its largest code; p becomes NaN there.  Two steps, so the
    second decodes the non-finite codes the first wrote.  Every tensor of the
    size sweep gets a NaN, a +Inf and a -Inf.  NaN codes are compared as a
    class: IEEE fixes neither the sign nor the payload of a NaN that
    arithmetic produces (the GPU returns its canonical NaN, an x86 host a
    negative one), so every BF16 NaN code, and every E4M3 S.1111.111, is
    mapped to one code on both sides first."""
    w = W.workload("sweep", m_dtype="bf16", v_dtype=v_dtype, hp=dict(lr=1e-3, weight_decay=0.1))
    w.max_norm = 0.0
    gpu = GpuSide(w, seed=7)
    orc = OracleSide(gpu, range(len(w.sizes)))
    ghp, ohp = hp_for(w, rounding=rounding, seed=31)
    for t in (1, 2):
        W.fill_grads(w, gpu.grads, t, 7)
        W.inject_nonfinite(gpu.grads, seed=40 + t, frac=1.0)
        g_np = orc.grads(gpu.grads)
        gpu.step(t, ghp, clip=False)
        orc.step(t, g_np, ohp, 1.0, rounding == "stochastic", 31)
    torch.cuda.synchronize()

    def canon(arr, dtype):
        """NaN codes to one code, in place (numpy array or torch tensor)."""
        if dtype == "bf16":
            a = arr.view(np.uint16) if isinstance(arr, np.ndarray) else arr.view(torch.int16)
            mask = 0x7F80
            nan = ((a & mask) == mask) & ((a & 0x7F) != 0)
            a[nan] = 0x7FC0
        elif dtype == "e4m3":
            nan = (arr & 0x7F) == 0x7F
            arr[nan] = 0x7F

    for k, i in enumerate(range(len(w.sizes))):
        for dt, g_t, o_a in (("bf16", gpu.m[i], orc.m[k]), (v_dtype, gpu.v[i], orc.v[k])):
            canon(g_t, dt)
            canon(o_a, dt)
    orc.compare(gpu, 1e-5, rounding == "stochastic", steps=2)
    assert gpu.plan.status() == 0


def test_bf16_v_never_moves_with_zero_grad():
    """"When Small Updates Disappear" sec. 2.2 on the GPU: b2 = 0.999,
    nearest rounding, g = 0 -> every BF16 v code stays put."""
    w = W.workload("sweep", m_dtype="bf16", v_dtype="bf16", hp=dict(beta2=0.999))
    gpu = GpuSide(w, seed=1)
    rng = np.random.default_rng(2)
    for v in gpu.v:
        vals = torch.from_numpy(np.exp(rng.uniform(-10, 2, v.numel())).astype(np.float32))
        v.copy_(vals.to(torch.bfloat16).view(torch.int16).cuda())
    before = [v.clone() for v in gpu.v]
    ghp, _ = hp_for(w, count=True)
    for t in range(1, 6):
        for g in gpu.grads:
            g.zero_()
        gpu.step(t, ghp, clip=False)
        assert gpu.plan.unchanged_count() == w.numel
    for a, b in zip(before, gpu.v):
        assert torch.equal(a, b)


def test_repeatable_and_seed_sensitive():
    w = W.workload("sweep", m_dtype="bf16", v_dtype="e4m3")
    outs = []
    for seed in (5, 5, 6):
        gpu = GpuSide(w, seed=0)
        ghp, _ = hp_for(w, rounding="stochastic", seed=seed)
        for t in (1, 2):
            W.fill_grads(w, gpu.grads, t, 0)
            gpu.step(t, ghp, clip=False)
        torch.cuda.synchronize()
        outs.append(torch.cat([x.view(torch.uint8) for x in gpu.m + gpu.v]))
    assert torch.equal(outs[0], outs[1])
    assert not torch.equal(outs[0], outs[2])


def test_invalid_arguments():
    w = W.workload("sweep")
    gpu = GpuSide(w)
    ghp, _ = hp_for(w)
    with pytest.raises(ps.OptError) as e:
        gpu.plan.adamw_step(ghp, 0)
    assert e.value.status == ps.OPT_EINVAL
    with pytest.raises(ps.OptError) as e:
        gpu.plan.ademamix_step(ghp, 1)          # no m2 buffers in this plan
    assert e.value.status == ps.OPT_EINVAL
    bad = ps.hparams(rounding="nearest")
    bad.rounding = 7
    with pytest.raises(ps.OptError):
        gpu.plan.adamw_step(bad, 1)
    p = torch.zeros(9, device="cuda")
    with pytest.raises(ps.OptError) as e:      # misaligned pointer
        ps.Plan([p[1:]], [torch.zeros(8, device="cuda")], [torch.zeros(8, device="cuda")],
                [torch.zeros(8, device="cuda")])
    assert e.value.status == ps.OPT_EALIGN
    with pytest.raises(ps.OptError) as e:      # FP8 gradients are not supported
        ps.Plan([p[:8]], [torch.zeros(8, dtype=torch.float8_e4m3fn, device="cuda")],
                [torch.zeros(8, device="cuda")], [torch.zeros(8, device="cuda")])
    assert e.value.status == ps.OPT_EUNSUPPORTED


@pytest.mark.parametrize("v_dtype", ["bf16", "e4m3", "e2m2"])
@pytest.mark.parametrize("rounding", ["nearest", "stochastic"])
def test_scaled_v_codes(v_dtype, rounding):
    """Per-tensor power-of-two v scales: the stored codes hold v / scale and
    match the oracle's exactly (stochastic) or to one step (nearest)."""
    w = W.workload("sweep", m_dtype="bf16", v_dtype=v_dtype, hp=dict(lr=1e-3, weight_decay=0.1),
                   sigma_decay_steps=8)
    scales = [2.0 ** k for k in ([-8, -4, 0, 3, -12] * 5)[:len(w.sizes)]]
    gpu = GpuSide(w, seed=2, v_scale=scales)
    _, _, counts = run_lockstep(w, 8, 1e-6, rounding=rounding, count=True, gpu=gpu, checkpoints=(1, 4))
    assert all(got == want for got, want in counts)


@pytest.mark.parametrize("shape", ["persistent", "short"])
def test_ademamix_reset_step_starts_from_zero_states(shape):
    """The reset flag starts AdEMAMix's three moments from zero: its reset
    step equals, bit for bit, a step at t = 1 after zeroing m, v and m2 by
    hand (the warp-dynamic kernel on the sweep list, the short-list kernel on
    seven tensors)."""
    extra = dict(sizes=SHORT) if shape == "short" else {}
    w = W.workload("sweep", algo="ademamix", hp=dict(lr=1e-2, weight_decay=0.1), **extra)
    w.max_norm = 0.0
    a, b = GpuSide(w, seed=6), GpuSide(w, seed=6)
    ghp, _ = hp_for(w)
    for t in (1, 2, 3):                       # both accumulate the same states
        for side in (a, b):
            W.fill_grads(w, side.grads, t, 6)
            side.step(t, ghp, clip=False)
    for side in (a, b):
        W.fill_grads(w, side.grads, 4, 6)
    for x in b.m + b.v + b.m2:
        x.zero_()
    b.step(1, ghp, clip=False)
    rhp = hp_for(w)[0]
    rhp.flags = ps.OPT_STEP_RESET_STATES
    a.step(1, rhp, clip=False)
    torch.cuda.synchronize()
    assert any(bool(x.any()) for x in a.m2)
    for x, y in zip(a.params + a.m + a.v + a.m2, b.params + b.m + b.v + b.m2):
        assert torch.equal(x, y)


@pytest.mark.parametrize("v_dtype,rounding", [("f32", "nearest"), ("bf16", "nearest"), ("e2m2", "nearest"),
                                              ("bf16", "stochastic"), ("e4m3", "stochastic"),
                                              ("e2m2", "stochastic")])
@pytest.mark.parametrize("shape", ["persistent", "short"])
def test_reset_step_starts_from_zero_states(v_dtype, rounding, shape):
    """"When Small Updates Disappear" sec. 5: a reset step starts from zero
    moments.  It must equal (bitwise) a step at t = 1 after zeroing the
    states by hand, and match the oracle run from zeroed states.  Both list
    shapes: the sweep list (persistent kernels) and seven tensors (the
    short-list kernels, four elements per thread with FP32 states)."""
    md = "f32" if v_dtype == "f32" else "bf16"
    extra = dict(sizes=SHORT) if shape == "short" else {}
    w = W.workload("sweep", m_dtype=md, v_dtype=v_dtype, hp=dict(lr=1e-2, weight_decay=0.1), **extra)
    w.max_norm = 0.0
    a, b = GpuSide(w, seed=4), GpuSide(w, seed=4)
    sr = rounding == "stochastic"
    ghp, ohp = hp_for(w, rounding=rounding)
    for t in (1, 2, 3):                       # both accumulate the same states
        for side in (a, b):
            W.fill_grads(w, side.grads, t, 4)
            side.step(t, ghp, clip=False)
    for side in (a, b):
        W.fill_grads(w, side.grads, 4, 4)
    orc = OracleSide(b, range(len(w.sizes)))  # the states the reset discards
    g_np = orc.grads(b.grads)
    for x in b.m + b.v:
        x.zero_()
    b.step(1, ghp, clip=False)
    rhp = hp_for(w, rounding=rounding)[0]
    rhp.flags = ps.OPT_STEP_RESET_STATES
    a.step(1, rhp, clip=False)
    torch.cuda.synchronize()
    for x, y in zip(a.params + a.m + a.v, b.params + b.m + b.v):
        assert torch.equal(x, y)
    for k in range(len(orc.samples)):
        orc.m[k][...] = 0
        orc.v[k][...] = 0
    orc.step(1, g_np, ohp, 1.0, sr, 1234)
    orc.compare(a, 1e-6, sr)
    assert a.plan.status() == 0 and b.plan.status() == 0


def test_invalid_flags_and_scales():
    w = W.workload("sweep")
    gpu = GpuSide(w)
    bad = ps.hparams()
    bad.flags = 2
    with pytest.raises(ps.OptError) as e:
        gpu.plan.adamw_step(bad, 1)
    assert e.value.status == ps.OPT_EINVAL
    x = [torch.zeros(8, device="cuda")]
    with pytest.raises(ps.OptError):          # not a power of two
        ps.Plan(x, [torch.zeros(8, device="cuda")], [torch.zeros(8, dtype=torch.int16, device="cuda")],
                [torch.zeros(8, dtype=torch.uint8, device="cuda")], m_dtype="bf16", v_dtype="e4m3",
                v_scale=[3.0])
    with pytest.raises(ps.OptError):          # FP32 v takes no scale
        ps.Plan(x, [torch.zeros(8, device="cuda")], [torch.zeros(8, device="cuda")],
                [torch.zeros(8, device="cuda")], v_scale=[2.0])


def _lamb_run(w, seed, max_unorm, steps, with_oracle=True):
    gpu = GpuSide(w, seed=seed)
    orc = OracleSide(gpu, range(len(w.sizes))) if with_oracle else None
    ghp, ohp = hp_for(w)
    ratios = []
    for t in range(1, steps + 1):
        W.fill_grads(w, gpu.grads, t, seed)
        coef = 1.0
        d_norm = None
        if w.max_norm > 0:
            g_all = [W.to_numpy_codes(g) for g in gpu.grads]
            coef = oracle.grad_norm(g_all, w.max_norm)["clip_coef"]
            gpu.plan.grad_norm(w.max_norm, sync=False)
            d_norm = gpu.plan.norm_buffer()
        if orc is not None:
            g_np = orc.grads(gpu.grads)
            ratios.append([oracle.lamb_tensor(orc.p[k], g_np[k], orc.m[k], orc.v[k], ohp, t, max_unorm, coef)
                           for k in range(len(orc.samples))])
        gpu.plan.lamb_step(ghp, t, max_unorm, d_norm)
    torch.cuda.synchronize()
    return gpu, orc, ratios


@pytest.mark.parametrize("gdt", ["bf16", "f32"])
@pytest.mark.parametrize("max_unorm", [0.3, 100.0])
def test_lamb_matches_oracle(gdt, max_unorm):
    """Update-norm clipping ("Investigate SM103 bias-correction broadcast in
    32-bit optimizers", 'B300 result'): the GPU's fixed-slot norms give the
    oracle's ratios; p, m, v match within 1e-5 (1+|x|) after 5 steps."""
    w = W.workload("sweep", grad_dtype=gdt, hp=dict(lr=1e-2, weight_decay=0.1))
    gpu, orc, ratios = _lamb_run(w, 6, max_unorm, 5)
    flat = [r for rs in ratios for r in rs]
    if max_unorm < 1.0:
        assert all(r < 1.0 for r in flat)          # |u| ~ |g|/|g| >> 0.3 |p| everywhere
    else:
        assert any(r == 1.0 for r in flat) and any(r < 1.0 for r in flat)   # tiny tensors still clip
    orc.compare(gpu, 1e-5, False)


def test_lamb_bitwise_repeatable_and_zero_bound_is_adamw():
    w = W.workload("clip_740", steps=3)
    a, _, _ = _lamb_run(w, 7, 0.5, 3, with_oracle=False)
    b, _, _ = _lamb_run(w, 7, 0.5, 3, with_oracle=False)
    for x, y in zip(a.params + a.m + a.v, b.params + b.m + b.v):
        assert torch.equal(x, y)
    del a, b
    # max_unorm = 0: the AdamW step, bit for bit
    ws = W.workload("sweep")
    c, _, _ = _lamb_run(ws, 8, 0.0, 2, with_oracle=False)
    d = GpuSide(ws, seed=8)
    ghp, _ = hp_for(ws)
    for t in (1, 2):
        W.fill_grads(ws, d.grads, t, 8)
        d.step(t, ghp, clip=True)
    torch.cuda.synchronize()
    for x, y in zip(c.params + c.m + c.v, d.params + d.m + d.v):
        assert torch.equal(x, y)


def test_lamb_rejects_low_precision_states():
    w = W.workload("sweep", m_dtype="bf16", v_dtype="e4m3")
    gpu = GpuSide(w)
    with pytest.raises(ps.OptError) as e:
        gpu.plan.lamb_step(ps.hparams(), 1, 1.0)
    assert e.value.status == ps.OPT_EUNSUPPORTED


@pytest.mark.parametrize("v_dtype", ["f32", "bf16", "e4m3", "e2m2"])
def test_mixed_grad_dtypes_and_empty_tensors(v_dtype):
    """One plan over a list that mixes BF16 and FP32 gradients (two dtype
    buckets, one launch each) and holds zero-size and one-element tensors:
    three clipped steps with stochastic rounding, every value and code against
    the oracle.  Covers both step kernels (register-pipelined and staged) on
    both buckets, full and short tiles."""
    sizes = [4096, 0, 1, 2048 * 3 + 17, 5, 0, 8192, 333, 2048]
    m_dtype = "f32" if v_dtype == "f32" else "bf16"
    w = W.Workload("mixed", sizes, "bf16", m_dtype=m_dtype, v_dtype=v_dtype, steps=3, max_norm=1.0,
                   p_std=0.02, grad_std=1.0, hp=dict(lr=1e-2, weight_decay=0.1))
    gpu = GpuSide(w, seed=5)
    for i in (1, 2, 6, 7):
        gpu.grads[i] = torch.empty(sizes[i], dtype=torch.float32, device="cuda")
    gpu.plan.close()
    gpu.plan = ps.Plan(gpu.params, gpu.grads, gpu.m, gpu.v, m_dtype=m_dtype, v_dtype=v_dtype)
    _, _, counts = run_lockstep(w, 3, 1e-6, rounding="stochastic", count=v_dtype != "f32", gpu=gpu)
    for got, want in counts:
        assert got == want


def _offset16(t: torch.Tensor) -> torch.Tensor:
    """A copy of t that starts 16 bytes into a fresh allocation: 16-byte
    aligned (the ABI's rule) but not 32-byte aligned."""
    k = 16 // t.element_size()
    buf = torch.empty(t.numel() + k, dtype=t.dtype, device=t.device)
    assert buf.data_ptr() % 32 == 0
    view = buf[k:k + t.numel()]
    view.copy_(t)
    assert view.data_ptr() % 32 == 16
    return view


@pytest.mark.parametrize("algo", ["adamw", "ademamix"])
@pytest.mark.parametrize("gdt", ["bf16", "f32"])
def test_fp32_streams_without_32_byte_alignment(algo, gdt):
    """The AdamW step reads FP32 p, m and v 32 bytes at a time where the
    stream's base is 32-byte aligned and 16 bytes at a time where it is not;
    the choice is per tensor and per stream.  Here p, g, m, v and m2 of
    different tensors sit 16 bytes off a 32-byte boundary in different
    combinations, against the oracle (AdEMAMix, which always reads 16 bytes
    at a time, alongside)."""
    w = W.workload("sweep", algo=algo, grad_dtype=gdt, hp=dict(lr=0.1, weight_decay=0.1))
    gpu = GpuSide(w, seed=9)
    for i in range(len(w.sizes)):
        if w.sizes[i] == 0:
            continue
        if i % 2 == 0:
            gpu.params[i] = _offset16(gpu.params[i])
        if i % 3 == 0:
            gpu.grads[i] = _offset16(gpu.grads[i])
        if i % 4 == 1:
            gpu.m[i] = _offset16(gpu.m[i])
        if i % 5 != 2:
            gpu.v[i] = _offset16(gpu.v[i])
        if gpu.m2 is not None and i % 2 == 1:
            gpu.m2[i] = _offset16(gpu.m2[i])
    gpu.plan.close()
    gpu.plan = ps.Plan(gpu.params, gpu.grads, gpu.m, gpu.v, gpu.m2)
    run_lockstep(w, 2, 1e-6, gpu=gpu)


@pytest.mark.parametrize("case", ["lr0", "beta1_0", "beta2_0"])
@pytest.mark.parametrize("v_dtype", ["f32", "e4m3"])
def test_degenerate_hyperparameters(case, v_dtype):
    """Edge values of the hyperparameters, against the oracle: lr = 0 (the
    parameters stay bit-for-bit as they were while the moments move),
    beta1 = 0 (m is the clipped gradient) and beta2 = 0 (v is its square)."""
    hp = dict(lr=1e-2, weight_decay=0.1)
    hp.update({"lr0": dict(lr=0.0), "beta1_0": dict(beta1=0.0), "beta2_0": dict(beta2=0.0)}[case])
    m_dtype = "f32" if v_dtype == "f32" else "bf16"
    w = W.workload("sweep", m_dtype=m_dtype, v_dtype=v_dtype, hp=hp)
    gpu = GpuSide(w, seed=21)
    p0 = [p.clone() for p in gpu.params]
    run_lockstep(w, 3, 1e-6, rounding="stochastic" if v_dtype != "f32" else "nearest", gpu=gpu)
    if case == "lr0":
        for a, b in zip(gpu.params, p0):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_ademamix_without_slow_moment_is_adamw_bitwise():
    """AdEMAMix with alpha = 0 and beta3 = 1 keeps m2 at zero and adds
    nothing to the update, so it must leave p, m and v with exactly the bits
    AdamW leaves on the same inputs (the two run as different kernels)."""
    hp = dict(lr=1e-2, weight_decay=0.1, alpha=0.0, beta3=1.0)
    wa = W.workload("sweep", algo="adamw", hp=hp)
    we = W.workload("sweep", algo="ademamix", hp=hp)
    ga, ge = GpuSide(wa, seed=23), GpuSide(we, seed=23)
    hpa, _ = hp_for(wa)
    hpe, _ = hp_for(we)
    for t in range(1, 4):
        W.fill_grads(wa, ga.grads, t, 23)
        W.fill_grads(we, ge.grads, t, 23)
        ga.step(t, hpa, clip=True)
        ge.step(t, hpe, clip=True)
    torch.cuda.synchronize()
    for name in ("params", "m", "v"):
        for a, b in zip(getattr(ga, name), getattr(ge, name)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), name
    for m2 in ge.m2:
        assert not m2.any()


def _counted_lockstep(w, gpu, steps, seed, launch, first_step=1):
    """Steps first_step .. first_step + steps - 1 on the oracle beside the
    GPU's device-counted steps; `launch()` issues the GPU's norm and step."""
    orc = OracleSide(gpu, range(len(w.sizes)))
    _, ohp = hp_for(w)
    for t in range(first_step, first_step + steps):
        W.fill_grads(w, gpu.grads, t, seed)
        want = oracle.grad_norm([W.to_numpy_codes(g) for g in gpu.grads], w.max_norm)
        g_np = orc.grads(gpu.grads)
        launch()
        orc.step(t, g_np, ohp, want["clip_coef"], False, 0)
    torch.cuda.synchronize()
    orc.compare(gpu, 1e-5, False)


@pytest.mark.parametrize("algo", ["adamw", "ademamix"])
@pytest.mark.parametrize("gdt", ["bf16", "f32"])
def test_device_step_counter_matches_oracle(algo, gdt):
    """OPT_STEP_DEVICE_COUNTER: step argument 0, the step number taken from
    the plan's device counter (advanced by each call), the bias corrections
    formed on the device; five steps against the oracle's steps 1..5."""
    w = W.workload("sweep", algo=algo, grad_dtype=gdt, hp=dict(lr=1e-2, weight_decay=0.1))
    gpu = GpuSide(w, seed=31)
    ghp, _ = hp_for(w)
    ghp.flags |= ps.OPT_STEP_DEVICE_COUNTER
    fn = gpu.plan.ademamix_step if algo == "ademamix" else gpu.plan.adamw_step

    def launch():
        gpu.plan.grad_norm(w.max_norm, sync=False)
        fn(ghp, 0, gpu.plan.norm_buffer())
    _counted_lockstep(w, gpu, 5, 31, launch)


def test_device_step_counter_set_step():
    """opt_plan_set_step(7): the next counted steps are 7, 8, 9."""
    w = W.workload("sweep", hp=dict(lr=1e-2, weight_decay=0.1))
    gpu = GpuSide(w, seed=32)
    ghp, _ = hp_for(w)
    ghp.flags |= ps.OPT_STEP_DEVICE_COUNTER
    gpu.plan.set_step(7)

    def launch():
        gpu.plan.grad_norm(w.max_norm, sync=False)
        gpu.plan.adamw_step(ghp, 0, gpu.plan.norm_buffer())
    _counted_lockstep(w, gpu, 3, 32, launch, first_step=7)


def test_cuda_graph_replays_counted_steps():
    """The norm and a device-counted step captured once in a CUDA graph;
    each replay is the next step (1, 2, 3, 4), against the oracle."""
    w = W.workload("sweep", hp=dict(lr=1e-2, weight_decay=0.1))
    ghp, _ = hp_for(w)
    ghp.flags |= ps.OPT_STEP_DEVICE_COUNTER
    side = torch.cuda.Stream()
    # warm up (occupancy caches, first launches) on a throwaway plan
    warm = GpuSide(w, seed=98)
    with torch.cuda.stream(side):
        warm.plan.grad_norm(w.max_norm, sync=False)
        warm.plan.adamw_step(ghp, 0, warm.plan.norm_buffer())
    torch.cuda.synchronize()
    gpu = GpuSide(w, seed=34)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        gpu.plan.grad_norm(w.max_norm, sync=False)
        gpu.plan.adamw_step(ghp, 0, gpu.plan.norm_buffer())
    _counted_lockstep(w, gpu, 4, 34, graph.replay)
    assert gpu.plan.status() == 0


def test_device_step_counter_rejects():
    w = W.workload("sweep")
    gpu = GpuSide(w, seed=35)
    hp = ps.hparams(device_step=True)
    with pytest.raises(ps.OptError) as e:
        gpu.plan.adamw_step(hp, 1)                    # a step number with the counter
    assert e.value.status == ps.OPT_EINVAL
    with pytest.raises(ps.OptError) as e:
        gpu.plan.adamw_step(ps.hparams(), 0)          # step 0 without it
    assert e.value.status == ps.OPT_EINVAL
    with pytest.raises(ps.OptError) as e:
        gpu.plan.set_step(0)
    assert e.value.status == ps.OPT_EINVAL
    with pytest.raises(ps.OptError) as e:
        gpu.plan.lamb_step(hp, 0, 1.0)
    assert e.value.status == ps.OPT_EINVAL
    wl = W.workload("sweep", m_dtype="bf16", v_dtype="e4m3")
    low = GpuSide(wl, seed=36)
    with pytest.raises(ps.OptError) as e:
        low.plan.adamw_step(hp, 0)
    assert e.value.status == ps.OPT_EUNSUPPORTED


def test_grads_upload_copies_every_tensor_exactly():
    """opt_grads_upload: host gradients (pinned and pageable, BF16 and FP32,
    zero-size and one-element tensors) land in the plan's device gradients
    bit for bit, on a side stream; the norm over them equals the oracle's.
    The binding rejects a host list that does not match the plan."""
    sizes = [4096, 0, 1, 2048 * 3 + 17, 5]
    w = W.Workload("upload", sizes, "bf16", steps=1, max_norm=1.0, p_std=0.02, grad_std=1.0)
    gpu = GpuSide(w, seed=3)
    gpu.grads[2] = torch.empty(1, dtype=torch.float32, device="cuda")
    gpu.grads[4] = torch.empty(5, dtype=torch.float32, device="cuda")
    gpu.plan.close()
    gpu.plan = ps.Plan(gpu.params, gpu.grads, gpu.m, gpu.v)
    gen = torch.Generator().manual_seed(11)
    host = []
    for i, g in enumerate(gpu.grads):
        h = torch.randn(g.numel(), generator=gen).to(g.dtype)
        host.append(h.pin_memory() if i % 2 == 0 else h)
    side = torch.cuda.Stream()
    gpu.plan.grads_upload(host, stream=side)
    side.synchronize()
    for h, g in zip(host, gpu.grads):
        assert torch.equal(g.cpu().view(torch.int16 if g.dtype == torch.bfloat16 else torch.int32),
                           h.view(torch.int16 if h.dtype == torch.bfloat16 else torch.int32))
    got = gpu.plan.grad_norm(1.0)
    want = oracle.grad_norm([W.to_numpy_codes(h) for h in host], 1.0)
    assert abs(got.norm2 - want["norm2"]) <= 1e-12 * want["norm2"] and got.clip_coef == want["clip_coef"]
    with pytest.raises(ValueError):
        gpu.plan.grads_upload(host[:-1])
    with pytest.raises(ValueError):
        gpu.plan.grads_upload(host[:-1] + [torch.zeros(4, dtype=torch.float32)])
    with pytest.raises(ValueError):
        gpu.plan.grads_upload([host[0].float()] + host[1:])
    gpu.plan.close()


@pytest.mark.parametrize("max_unorm", [0.3, 100.0])
def test_lamb_tensors_over_several_segments_match_oracle(max_unorm):
    """The ratio pass cuts a tensor's tiles into segments of 2,048 and forms
    the ratio in the CTA that finishes the tensor's last segment: tensors of
    4 segments (the last one ragged), of exactly 1, of 2 (the second one
    tile), and a tiny one give the oracle's ratios and states after 3 steps,
    and the same bits twice."""
    seg = 2048 * 2048
    sizes = [3 * seg + 777, seg, seg + 1, 5]
    w = W.Workload("lamb_segments", sizes, "bf16", steps=3, max_norm=1.0, p_std=0.02, grad_std=1.0,
                   hp=dict(lr=1e-2, weight_decay=0.1))
    gpu, orc, ratios = _lamb_run(w, 9, max_unorm, 3)
    flat = [r for rs in ratios for r in rs]
    if max_unorm < 1.0:
        assert all(r < 1.0 for r in flat)
    orc.compare(gpu, 1e-5, False)
    again, _, _ = _lamb_run(w, 9, max_unorm, 3, with_oracle=False)
    for x, y in zip(gpu.params + gpu.m + gpu.v, again.params + again.m + again.v):
        assert torch.equal(x, y)
