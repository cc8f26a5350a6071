"""Out-of-bounds writes, checked without a sanitizer: every device buffer a
call writes (parameters, moments, gradients, norm results, cast outputs) sits
inside a larger allocation whose bytes before and after it hold a fixed
pattern, and after the calls every pattern byte is still there.  The sizes
are odd and ragged (tile and chunk edges, single elements, odd E2M2 counts),
the calls every kernel of the library: the norm (plan and no-allocation),
the AdamW step in every state mode and rounding, the reset step, AdEMAMix,
the update-norm clipped (LAMB) step, and the standalone cast both ways."""
import ctypes

import numpy as np
import pytest
import torch

import precision_states_gb300 as ps
import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 512                      # pattern bytes before and after each buffer
PATTERN = 0xA5
SIZES = [1, 2, 3, 7, 9, 255, 257, 2047, 2049, 4097, 8193, 32767, 32769, 70001]
TORCH = {"f32": torch.float32, "bf16": torch.int16, "e4m3": torch.uint8, "e2m2": torch.uint8,
         "gbf16": torch.bfloat16}


class Guarded:
    """Buffers of given byte sizes, each inside a pattern-filled allocation."""

    def __init__(self):
        self.bufs = []

    def make(self, nbytes: int, dtype: torch.dtype, init: torch.Tensor | None = None) -> torch.Tensor:
        buf = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        view = buf[GUARD:GUARD + nbytes].view(dtype)
        assert view.data_ptr() % 256 == 0
        if init is not None:
            view.copy_(init.reshape(-1).view(dtype) if init.dtype != dtype else init.reshape(-1))
        else:
            view.zero_()
        self.bufs.append((buf, nbytes))
        return view

    def check(self, what: str):
        torch.cuda.synchronize()
        for k, (buf, nbytes) in enumerate(self.bufs):
            head = buf[:GUARD].cpu().numpy()
            tail = buf[GUARD + nbytes:].cpu().numpy()
            assert np.all(head == PATTERN), f"{what}: buffer {k}: bytes before it were written"
            assert np.all(tail == PATTERN), f"{what}: buffer {k}: bytes past its {nbytes} were written " \
                                            f"(first at +{int(np.argmax(tail != PATTERN))})"


def state_nbytes(dtype: str, n: int) -> int:
    return ps.state_nbytes(dtype, n)


def guarded_plan(g: Guarded, sizes, grad_dtypes, m_dtype, v_dtype, m2=False, seed=0):
    w = W.Workload("guard", list(sizes), "bf16", m_dtype=m_dtype, v_dtype=v_dtype, p_std=0.02, grad_std=1.0)
    params, grads, ms, vs, m2s = [], [], [], [], []
    src_p = W.make_params(w, "cuda", seed)
    for i, n in enumerate(sizes):
        params.append(g.make(4 * n, torch.float32, src_p[i]))
        gd = torch.bfloat16 if grad_dtypes[i] == "bf16" else torch.float32
        gr = g.make((2 if gd == torch.bfloat16 else 4) * n, gd)
        gr.copy_(torch.randn(n, device="cuda").to(gd))
        grads.append(gr)
        ms.append(g.make(state_nbytes(m_dtype, n), TORCH[m_dtype]))
        vs.append(g.make(state_nbytes(v_dtype, n), TORCH[v_dtype]))
        if m2:
            m2s.append(g.make(4 * n, torch.float32))
    plan = ps.Plan(params, grads, ms, vs, m2s if m2 else None, m_dtype=m_dtype, v_dtype=v_dtype)
    return plan


def mixed(sizes):
    return ["f32" if i % 3 == 1 else "bf16" for i in range(len(sizes))]


@pytest.mark.parametrize("v_dtype,rounding", [("f32", "nearest"), ("bf16", "nearest"), ("bf16", "stochastic"),
                                              ("e4m3", "nearest"), ("e4m3", "stochastic"),
                                              ("e2m2", "nearest"), ("e2m2", "stochastic")])
def test_step_writes_stay_inside(v_dtype, rounding):
    g = Guarded()
    m_dtype = "f32" if v_dtype == "f32" else "bf16"
    plan = guarded_plan(g, SIZES, mixed(SIZES), m_dtype, v_dtype)
    d_res = g.make(48, torch.uint8)
    hp = ps.hparams(lr=1e-2, weight_decay=0.1, rounding=rounding, seed=3, count_unchanged=v_dtype != "f32")
    for t in range(1, 4):
        plan.grad_norm(1.0, d_out=d_res.data_ptr(), sync=False)
        plan.adamw_step(hp, t, d_res.data_ptr())
    reset = ps.hparams(lr=1e-2, weight_decay=0.1, rounding=rounding, seed=3, reset_states=True)
    plan.adamw_step(reset, 1, None)
    if v_dtype != "f32":
        plan.unchanged_count()
    assert plan.status() == 0
    g.check(f"adamw {v_dtype} {rounding}")
    plan.close()


@pytest.mark.parametrize("v_dtype,rounding", [("f32", "nearest"), ("bf16", "stochastic"), ("e4m3", "nearest"),
                                              ("e2m2", "stochastic")])
def test_short_list_step_writes_stay_inside(v_dtype, rounding):
    """The short-list launch shape (at most eight tensors): ragged sizes."""
    g = Guarded()
    sizes = [1, 3, 2047, 2049, 2052, 4097, 32769, 70001]
    m_dtype = "f32" if v_dtype == "f32" else "bf16"
    plan = guarded_plan(g, sizes, ["bf16"] * len(sizes), m_dtype, v_dtype)
    d_res = g.make(48, torch.uint8)
    hp = ps.hparams(lr=1e-2, weight_decay=0.1, rounding=rounding, seed=3, count_unchanged=v_dtype != "f32")
    for t in range(1, 4):
        plan.grad_norm(1.0, d_out=d_res.data_ptr(), sync=False)
        plan.adamw_step(hp, t, d_res.data_ptr())
    if v_dtype != "f32":
        plan.unchanged_count()
    assert plan.status() == 0
    g.check(f"short list {v_dtype} {rounding}")
    plan.close()


def test_ademamix_and_lamb_writes_stay_inside():
    g = Guarded()
    plan = guarded_plan(g, SIZES, mixed(SIZES), "f32", "f32", m2=True)
    hp = ps.hparams(lr=1e-2, weight_decay=0.1)
    for t in range(1, 3):
        plan.ademamix_step(hp, t, None)
    g.check("ademamix")
    plan.close()
    g2 = Guarded()
    plan = guarded_plan(g2, SIZES, mixed(SIZES), "f32", "f32")
    for t in range(1, 3):
        plan.lamb_step(hp, t, 1.0, None)
    assert plan.status() == 0
    g2.check("lamb")
    plan.close()


def test_noalloc_norm_writes_stay_inside():
    g = Guarded()
    grads = []
    for i, n in enumerate(SIZES):
        gd = torch.bfloat16 if i % 2 else torch.float32
        t = g.make((2 if gd == torch.bfloat16 else 4) * n, gd)
        t.copy_(torch.randn(n, device="cuda").to(gd))
        grads.append(t)
    d_out = g.make(48, torch.uint8)
    n = len(grads)
    numel = (ctypes.c_int64 * n)(*[t.numel() for t in grads])
    ptrs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in grads])
    dts = (ctypes.c_int32 * n)(*[ps.OPT_BF16 if t.dtype == torch.bfloat16 else ps.OPT_F32 for t in grads])
    for _ in range(2):
        assert ps.lib().opt_grad_norm_noalloc(n, numel, ptrs, dts, 1.0, d_out.data_ptr(), None) == ps.OPT_OK
    g.check("noalloc norm")


@pytest.mark.parametrize("fmt", ["bf16", "e4m3", "e2m2"])
@pytest.mark.parametrize("rounding", ["nearest", "stochastic"])
def test_cast_writes_stay_inside(fmt, rounding):
    g = Guarded()
    for n in SIZES:
        x = g.make(4 * n, torch.float32)
        x.copy_(torch.randn(n, device="cuda"))
        codes = g.make(state_nbytes(fmt, n), TORCH[fmt])
        back = g.make(4 * n, torch.float32)
        ps.opt_encode(x, codes, fmt, rounding=rounding, seed=5)
        ps.opt_decode(codes, back, n, fmt)
    g.check(f"cast {fmt} {rounding}")


def test_guard_check_detects_a_stray_write():
    """The check itself: a byte written just past a buffer (by a plain torch
    write into the pattern region, not by a kernel) is reported."""
    g = Guarded()
    v = g.make(4 * 7, torch.float32)
    v.fill_(1.0)
    g.check("clean")
    g.bufs[0][0][GUARD + 4 * 7] = 0
    with pytest.raises(AssertionError, match="past its 28"):
        g.check("planted")
