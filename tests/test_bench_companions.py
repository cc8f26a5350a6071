"""The default bench run also times every other workload briefly: the list
covers each workload and every low-precision state mode, and only the
default single-GPU invocation runs it."""
import sys

import pytest

import bench
import workloads as W


def test_companions_cover_every_workload_and_state_mode():
    names = {c[0] for c in bench.COMPANIONS}
    assert names == {"adamw_1m", "clip_740", "ademamix_gpt2", "lowp_gpt2", "llama3_8b"}
    lowp = {(v, r) for n, v, r, _ in bench.COMPANIONS if n == "lowp_gpt2" and v != "f32"}
    assert lowp == {(v, r) for v in ("bf16", "e4m3", "e2m2") for r in ("nearest", "stochastic")}
    assert ("lowp_gpt2", "f32", "nearest", None) in bench.COMPANIONS      # the fp32 control
    assert any(lamb is not None for *_, lamb in bench.COMPANIONS)          # the LAMB step
    for n, v, r, lamb in bench.COMPANIONS:
        import argparse
        w = bench.apply_overrides(W.workload(n), argparse.Namespace(v_dtype=v, lamb=lamb))
        assert w.numel > 0
        if v is not None and v != "f32":
            assert (w.m_dtype, w.v_dtype) == ("bf16", v)


@pytest.mark.parametrize("argv,world,want", [
    ([], 1, True),
    ([], 2, False),
    (["--no-companions"], 1, False),
    (["--workload", "clip_740"], 1, False),
    (["--v-dtype", "e4m3"], 1, False),
    (["--lamb", "1.0"], 1, False),
    (["--graph"], 1, False),
])
def test_companions_only_in_the_default_single_gpu_run(monkeypatch, argv, world, want):
    monkeypatch.setattr(sys, "argv", ["bench.py", *argv])
    assert bench.companions_wanted(bench.parse(), world) is want


def test_step_kernel_labels_follow_the_dispatch():
    """The roofline's kernel label names what the library launches for each
    list: the short-list shapes, the warp-dynamic FP32 step, the staged and
    register-pipelined low-precision steps, LAMB's passes."""
    import bench
    import workloads as W
    one = W.workload("adamw_1m")
    assert bench.step_kernel_name(one, "nearest").startswith("step_small4_kernel<")
    lowp_short = W.workload("sweep", sizes=[4097, 5], m_dtype="bf16", v_dtype="e4m3")
    assert bench.step_kernel_name(lowp_short, "nearest").startswith("step_small_kernel<")
    assert bench.step_kernel_name(W.workload("clip_740"), "nearest").startswith("step_dyn_kernel<")
    assert bench.step_kernel_name(W.workload("ademamix_gpt2"), "nearest").startswith("step_dyn_kernel<")
    lowp = W.workload("lowp_gpt2", v_dtype="e2m2")
    assert bench.step_kernel_name(lowp, "stochastic").startswith("step_bulk_kernel<")
    assert bench.step_kernel_name(lowp, "nearest").startswith("step_kernel<")
