"""GPU test of opt_grad_norm_noalloc, the norm entry point for callers that
cannot allocate device memory (their device memory belongs to a framework's
caching allocator or a fixed budget reserved up front, so they cannot build a
plan, which allocates a workspace).  It is called through the C ABI and its
result is compared bit for bit with opt_grad_norm's on the same gradients
(both sum the same slot spans in the same order: the plan's are built on the
host, the no-allocation call's by a kernel), on two calls
in a row with different lists, so that anything the first call leaves in the
shared scratch array would show up in the second.  Collected last on purpose
(file name) so a failure here does not hide the other tests."""
import ctypes
import math

import numpy as np
import pytest
import torch

import precision_states_gb300 as ps
import workloads as W

pytestmark = pytest.mark.gpu

def via_plan(grads, max_norm):
    params = [torch.zeros(g.numel(), device="cuda") for g in grads]
    m = [torch.zeros(g.numel(), device="cuda") for g in grads]
    v = [torch.zeros(g.numel(), device="cuda") for g in grads]
    plan = ps.Plan(params, grads, m, v)
    r = plan.grad_norm(max_norm)
    plan.close()
    return r


def via_noalloc(grads, max_norm, d_out):
    n = len(grads)
    numel = (ctypes.c_int64 * max(n, 1))(*[g.numel() for g in grads])
    ptrs = (ctypes.c_void_p * max(n, 1))(*[g.data_ptr() for g in grads])
    dts = (ctypes.c_int32 * max(n, 1))(*[ps.OPT_BF16 if g.dtype == torch.bfloat16 else ps.OPT_F32
                                          for g in grads])
    stream = torch.cuda.current_stream().cuda_stream
    st = ps.lib().opt_grad_norm_noalloc(n, numel, ptrs, dts, max_norm, d_out.data_ptr(), stream)
    assert st == ps.OPT_OK, ps.opt_strerror(st)
    torch.cuda.synchronize()
    raw = d_out.cpu().numpy().tobytes()
    return ps.opt_norm_result.from_buffer_copy(raw)


def same(a, b):
    assert a.status == b.status and a.nan_count == b.nan_count and a.inf_count == b.inf_count
    for k in ("norm2", "norm_inf", "sumsq"):
        x, y = getattr(a, k), getattr(b, k)
        if math.isnan(y):
            assert math.isnan(x)
        else:
            assert x == y, (k, x, y)
    assert a.clip_coef == b.clip_coef


def test_noalloc_matches_plan_norm_twice():
    d_out = torch.zeros(6, dtype=torch.float64, device="cuda")      # 48 bytes
    # first call: the size sweep with both gradient dtypes
    w = W.workload("sweep")
    g16 = W.make_grads(w, "cuda", step=1, seed=31)
    g32 = W.make_grads(W.workload("sweep", grad_dtype="f32"), "cuda", step=1, seed=32)
    first = [g16[i] if i % 3 else g32[i] for i in range(len(g16))]
    a = via_noalloc(first, 1.0, d_out)
    same(a, via_plan(first, 1.0))
    # second call, a different and larger list on the same scratch
    w2 = W.workload("clip_740")
    second = W.make_grads(w2, "cuda", step=2, seed=33)
    second[5] = second[5].float()
    b = via_noalloc(second, 1.0, d_out)
    same(b, via_plan(second, 1.0))
    assert a.norm2 != b.norm2
    # a list with fewer elements than slots, most slots empty
    gen = torch.Generator(device="cuda").manual_seed(34)
    third = [torch.randn(n, device="cuda", generator=gen).to(torch.bfloat16) for n in (3, 0, 5, 900)]
    third[2] = third[2].float()
    same(via_noalloc(third, 1.0, d_out), via_plan(third, 1.0))


def test_noalloc_rejects_lists_beyond_its_limits():
    n = ps.OPT_NOALLOC_MAX_TENSORS + 1
    numel = (ctypes.c_int64 * n)(*([1] * n))
    ptrs = (ctypes.c_void_p * n)(*([0x1000] * n))
    dts = (ctypes.c_int32 * n)(*([ps.OPT_BF16] * n))
    d_out = torch.zeros(6, dtype=torch.float64, device="cuda")
    assert ps.lib().opt_grad_norm_noalloc(n, numel, ptrs, dts, 1.0, d_out.data_ptr(), None) == ps.OPT_ELIMIT
    big = ps.OPT_NOALLOC_MAX_CHUNKS * ps.OPT_CHUNK_ELEMS + 1
    numel1 = (ctypes.c_int64 * 1)(big)
    assert ps.lib().opt_grad_norm_noalloc(1, numel1, ptrs, dts, 1.0, d_out.data_ptr(), None) == ps.OPT_ELIMIT
