"""Per-workload GPU parity at full size, in the launch configuration bench.py
times (whole tensor lists, one launch per dtype bucket).  The oracle computes
its own norm over every gradient each step and steps a seeded sample of
tensors and of slices of the large ones.

* clip_740: 740 tensors, 197M params, BF16 grads, clip 1.0, 20 steps.
* ademamix_gpt2: GPT-2-small list, 124M params, FP32 grads, 50 steps.
* lowp_gpt2: the same list with BF16 m and BF16 / E4M3 / E2M2 v, nearest
  and stochastic, plus the FP32 control, all 1,000 steps; unchanged-v counts
  exact.
* llama3_8b: the 8.03e9-parameter list, all 5 steps; each step the norm over
  all of it and the clipped step on 16 sampled tensors (always the embedding
  and a 4096-vector).  LAMB on the same list (the bench's LAMB run), 2 steps,
  8 sampled whole tensors.
"""
import numpy as np
import pytest
import torch

import oracle
import precision_states_gb300 as ps
import workloads as W
from harness import GpuSide, OracleSide, fp32_tol, hp_for, oracle_norm_parallel, rel_err, run_lockstep

pytestmark = pytest.mark.gpu


def free():
    import gc
    gc.collect()
    torch.cuda.empty_cache()


def sample_tensors(w, k, seed, always=()):
    rng = np.random.default_rng(seed)
    idx = set(always)
    while len(idx) < k:
        idx.add(int(rng.integers(0, len(w.sizes))))
    return sorted(idx)


def slices(w, seed, count, length, min_numel=1_000_000):
    """Seeded slices (index, even start, length) of the large tensors."""
    rng = np.random.default_rng(seed)
    big = [i for i, n in enumerate(w.sizes) if n >= min_numel]
    out = []
    for _ in range(count):
        i = int(rng.choice(big))
        start = int(rng.integers(0, (w.sizes[i] - length) // 2)) * 2
        out.append((i, start, length))
    return out


def test_clip740_twenty_steps():
    w = W.workload("clip_740")
    samples = sample_tensors(w, 24, seed=1, always=(int(np.argmax(w.sizes)), int(np.argmin(w.sizes))))
    run_lockstep(w, w.steps, 1e-5, samples=samples, checkpoints=(1,))
    free()


def test_ademamix_gpt2_fifty_steps():
    w = W.workload("ademamix_gpt2")
    small = [i for i, n in enumerate(w.sizes) if n < 1_000_000]
    samples = sorted(set(small[::9])) + slices(w, seed=2, count=4, length=65536)
    run_lockstep(w, w.steps, 1e-5, samples=samples, checkpoints=(1,))
    free()


@pytest.mark.parametrize("mode", ["f32", "bf16-nearest", "bf16-stochastic", "e4m3-nearest",
                                  "e4m3-stochastic", "e2m2-nearest", "e2m2-stochastic"])
def test_lowp_gpt2_modes(mode):
    """All seven state modes of the low-precision workload over all of its
    1,000 steps (the grad scale falls 10x linearly over them), full list on
    the GPU, codes compared on a sample at steps 1, 10, 100, 500 and 1,000,
    FP32 values within fp32_tol of the step count (p past 100 steps also
    within update_bound of the oracle's own moves).  The unchanged-v count is
    checked exactly on a second plan over the sampled tensors alone."""
    vd, _, rnd = mode.partition("-")
    w = W.workload("lowp_gpt2")
    assert w.steps == 1000 and w.sigma_decay_steps == 1000
    if vd == "f32":
        w.m_dtype = w.v_dtype = "f32"
    else:
        w.v_dtype = vd
    rounding = rnd or "nearest"
    small = [i for i, n in enumerate(w.sizes) if n < 10_000]
    samples = small[:6] + slices(w, seed=3, count=2, length=8192)
    run_lockstep(w, w.steps, fp32_tol, samples=samples, rounding=rounding, checkpoints=(1, 10, 100, 500),
                 track_moves=True)
    free()
    if vd == "f32":
        return   # FP32 v: the oracle forms v in double, so bitwise stalls need not match
    # exact unchanged counts on the small tensors alone (the pre-rounding fp32
    # values are bit-identical on both sides, so every code decision is too)
    ws = W.workload("lowp_gpt2", sigma_decay_steps=40, sizes=[w.sizes[i] for i in small[:8]])
    ws.m_dtype, ws.v_dtype = w.m_dtype, w.v_dtype
    _, _, counts = run_lockstep(ws, 40, 1e-5, rounding=rounding, count=True)
    assert all(got == want for got, want in counts), counts[:5]


def test_llama3_8b_five_steps():
    """All 5 steps of the Llama-3-8B workload on the whole list: every step
    the oracle's own norm over all 8.03e9 gradients (relative error <= 1e-12,
    identical clip coefficient) and the clipped step on 16 sampled tensors;
    p, m and v within 1e-6 (1+|x|) after step 1 and after step 5."""
    w = W.workload("llama3_8b")
    assert w.steps == 5
    gpu = GpuSide(w, seed=5)
    embed = 0
    vec = next(i for i, n in enumerate(w.sizes) if n == 4096)
    samples = sample_tensors(w, 16, seed=6, always=(embed, vec))
    got = gpu.plan.grad_norm(w.max_norm)
    assert got.clip_coef < 1.0          # the list's norm (~90) is clipped to 1.0
    gpu, orc, _ = run_lockstep(w, w.steps, 1e-6, samples=samples, checkpoints=(1,), gpu=gpu,
                               seed=5, step_threads=16)
    # repeatability of the norm at full size (the last step's gradients)
    first = gpu.plan.grad_norm(w.max_norm)
    again = gpu.plan.grad_norm(w.max_norm)
    assert again.as_dict() == first.as_dict()
    del gpu, orc
    free()


def test_llama3_8b_lamb_two_steps():
    """LAMB with max_unorm 1.0 on the whole Llama-3-8B list, as the bench
    times it (its three passes over every tile): each step the oracle's own
    norm over all 8.03e9 gradients gives the clip coefficient (relative error
    <= 1e-12, identical coefficient), and on 8 sampled whole tensors (always
    the embedding and a 4096-vector) the oracle's LAMB step, with that
    coefficient, gives p, m and v within 1e-5 (1+|x|) after 2 steps."""
    from concurrent.futures import ThreadPoolExecutor
    w = W.workload("llama3_8b")
    gpu = GpuSide(w, seed=5)
    vec = next(i for i, n in enumerate(w.sizes) if n == 4096)
    samples = sample_tensors(w, 8, seed=9, always=(0, vec))
    orc = OracleSide(gpu, samples)
    ghp, ohp = hp_for(w)
    ratios = []
    for t in (1, 2):
        W.fill_grads(w, gpu.grads, t, 5)
        g_all = [W.to_numpy_codes(g) for g in gpu.grads]
        want = oracle_norm_parallel(g_all, w.max_norm)
        del g_all
        got = gpu.plan.grad_norm(w.max_norm)
        assert rel_err(got.norm2, want["norm2"]) <= 1e-12, (t, got.norm2, want["norm2"])
        assert got.clip_coef == want["clip_coef"] and got.clip_coef < 1.0
        g_np = orc.grads(gpu.grads)
        with ThreadPoolExecutor(8) as ex:        # one whole tensor each; the C calls release the GIL
            ratios += list(ex.map(lambda k: oracle.lamb_tensor(orc.p[k], g_np[k], orc.m[k], orc.v[k], ohp, t, 1.0,
                                                               want["clip_coef"]), range(len(orc.samples))))
        gpu.plan.lamb_step(ghp, t, 1.0, gpu.plan.norm_buffer())
    torch.cuda.synchronize()
    assert any(r < 1.0 for r in ratios)          # the bound binds somewhere
    orc.compare(gpu, 1e-5, False)
    del gpu, orc
    free()


def test_single_tensor_beyond_32bit_indexing():
    """One tensor of 2^32 + 12 elements (BF16 grads, BF16 m and v, stochastic
    rounding, clipped): element offsets past 2^31 and 2^32, the high word of
    the Philox counter, and a ragged tail.  The oracle computes the full norm
    and steps slices at the start, across 2^31, across 2^32 and at the end."""
    n = (1 << 32) + 12
    w = W.Workload("huge", [n], "bf16", m_dtype="bf16", v_dtype="bf16", steps=1, max_norm=1.0,
                   p_std=0.02, grad_std=1e-3, hp=dict(lr=1e-3, weight_decay=0.1))
    gpu = GpuSide(w, seed=9)
    L = 4096
    samples = [(0, 0, L), (0, (1 << 31) - L // 2, L), (0, (1 << 32) - L // 2, L), (0, n - L, L)]
    orc = OracleSide(gpu, samples)
    ghp, ohp = hp_for(w, rounding="stochastic", seed=2024)
    got = gpu.plan.grad_norm(w.max_norm)
    g_all = W.to_numpy_codes(gpu.grads[0])
    want = oracle_norm_parallel([g_all[i:i + (1 << 28)] for i in range(0, n, 1 << 28)], w.max_norm)
    del g_all
    assert rel_err(got.norm2, want["norm2"]) <= 1e-12 and got.clip_coef == want["clip_coef"]
    g_np = orc.grads(gpu.grads)
    gpu.step(1, ghp, clip=True)
    orc.step(1, g_np, ohp, want["clip_coef"], True, 2024)
    torch.cuda.synchronize()
    orc.compare(gpu, 1e-6, True)
    del gpu, orc
    free()


def _omb(beta: float) -> np.float32:
    """(1 - beta) as the step forms it: in double from the fp32 beta, rounded once."""
    return np.float32(1.0 - float(np.float32(beta)))


@pytest.mark.parametrize("name,states", [("clip_740", "f32"), ("lowp_gpt2", "bf16"), ("llama3_8b", "f32")])
def test_every_element_updated_exactly_once(name, states):
    """One step from zero moments over a whole list: every element's new m
    and v must equal (1-b1) g' and (1-b2) g'^2 (g' = g times the clip
    coefficient), bit for bit, in every tensor -- an element skipped would
    keep 0, one updated twice would not match.  The 740-tensor list runs the
    register-pipelined FP32 kernel (about 317 tiles per CTA, 740 short
    tiles); the GPT-2 list with BF16 m and v (nearest) the staged kernel;
    the Llama-3-8B list (8.03e9 elements, the benchmark's launch) the FP32
    kernel again, with about 12,900 tiles per CTA.
    Reference values are torch fp32 operations (round to nearest, and for
    BF16 codes torch's nearest-even cast), the same operations in the same
    order."""
    w = W.workload(name)
    if states == "bf16":
        w.v_dtype = "bf16"
    gpu = GpuSide(w, seed=21)
    hp, _ = hp_for(w)
    clip = w.max_norm > 0
    gpu.step(1, hp, clip)
    coef = np.float32(gpu.plan.grad_norm(w.max_norm).clip_coef) if clip else np.float32(1.0)
    omb1, omb2 = _omb(0.9), _omb(w.hp.get("beta2", 0.999))
    for i, g in enumerate(gpu.grads):
        ge = g.float() * torch.tensor(coef, device="cuda")
        # + 0.0: the kernel adds b * 0 = +0 first, which turns a -0 into +0
        m_want = ge * torch.tensor(omb1, device="cuda") + 0.0
        v_want = (ge * ge) * torch.tensor(omb2, device="cuda") + 0.0
        if states == "f32":
            assert torch.equal(gpu.m[i].view(torch.int32), m_want.view(torch.int32)), f"m of tensor {i}"
            assert torch.equal(gpu.v[i].view(torch.int32), v_want.view(torch.int32)), f"v of tensor {i}"
        else:
            assert torch.equal(gpu.m[i], m_want.to(torch.bfloat16).view(torch.int16)), f"m of tensor {i}"
            assert torch.equal(gpu.v[i], v_want.to(torch.bfloat16).view(torch.int16)), f"v of tensor {i}"
    assert gpu.plan.status() == 0
    del gpu
    free()
