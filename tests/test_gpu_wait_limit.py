"""The staged step kernel's bounded waits, made to run out on purpose.

Low-precision states with stochastic rounding (and BF16 v with nearest
rounding) take their tiles through shared memory: a producer warp issues
bulk copies and consumer warps wait for them.  Every such wait gives up
after the plan's wait limit and raises OPT_FLAG_WAIT_TIMEOUT instead of
hanging.  A wait drill (OPT_STEP_WAIT_DRILL) makes that happen with no fault:
each thread block's producer withholds its first tile, so nothing ever
completes the stage the consumers wait on first -- a flag that nothing
sets.  The consumers give up, let the copies that were issued land, and
leave (OPT_FLAG_DRAIN_TIMEOUT stays clear); no tile is processed.

Checked: the flag is reported and then cleared; the step changed nothing
(p and both states are bitwise as before); nothing outside the buffers was
written (pattern bytes around each one); the same plan then takes a step
equal to the oracle's, and so does a fresh plan."""
import time

import pytest
import torch

import oracle
import precision_states_gb300 as ps
import workloads as W
from harness import assert_close_scaled, compare_codes
from test_gpu_guard_bands import TORCH, Guarded

pytestmark = pytest.mark.gpu

# Ragged sizes with many 2048-element tiles per thread block of the
# persistent grid (about 8.4M elements, 4,100 tiles).
SIZES = [4 * 2 ** 20 + 3, 2 * 2 ** 20 + 1, 2 ** 20, 777_777, 2049, 3]
STAGED = [("bf16", "nearest"), ("bf16", "stochastic"), ("e4m3", "stochastic"), ("e2m2", "stochastic")]
SEED = 21
DRILL_LIMIT_NS = 1_000_000          # 1 ms


def make_lists(g: Guarded, v_dtype: str, seed: int):
    w = W.Workload("waits", list(SIZES), "bf16", m_dtype="bf16", v_dtype=v_dtype, p_std=0.02, grad_std=1.0)
    src_p = W.make_params(w, "cuda", seed)
    src_g = W.make_grads(w, "cuda", 1, seed)
    params, grads, ms, vs = [], [], [], []
    for i, n in enumerate(SIZES):
        params.append(g.make(4 * n, torch.float32, src_p[i]))
        grads.append(g.make(2 * n, torch.bfloat16, src_g[i]))
        ms.append(g.make(ps.state_nbytes("bf16", n), TORCH["bf16"]))
        vs.append(g.make(ps.state_nbytes(v_dtype, n), TORCH[v_dtype]))
    return params, grads, ms, vs


def host(ts):
    return [W.to_numpy_codes(t) for t in ts]


def oracle_step(p, g, m, v, v_dtype, rounding):
    """The oracle's step 1 over the whole list, on host copies."""
    hp = oracle.hparams(lr=1e-2, weight_decay=0.1)
    for i in range(len(SIZES)):
        oracle.adam_tensor(oracle.ADAMW, p[i], g[i], m[i], v[i], hp, 1, m_dtype="bf16", v_dtype=v_dtype,
                           stochastic=rounding == "stochastic", seed=SEED, tensor_index=i)


def check_against_oracle(params, ms, vs, want_p, want_m, want_v, v_dtype, rounding):
    exact = rounding == "stochastic"
    for i, n in enumerate(SIZES):
        assert_close_scaled(W.to_numpy_codes(params[i]), want_p[i], 1e-6, f"p {i}")
        compare_codes(W.to_numpy_codes(ms[i]), want_m[i], "bf16", n, exact, f"m {i}")
        compare_codes(W.to_numpy_codes(vs[i]), want_v[i], v_dtype, n, exact, f"v {i}")


@pytest.mark.parametrize("v_dtype,rounding", STAGED)
def test_wait_drill_runs_out_reports_and_recovers(v_dtype, rounding):
    g = Guarded()
    params, grads, ms, vs = make_lists(g, v_dtype, seed=3)
    plan = ps.Plan(params, grads, ms, vs, m_dtype="bf16", v_dtype=v_dtype)
    hp = ps.hparams(lr=1e-2, weight_decay=0.1, rounding=rounding, seed=SEED)
    drill = ps.hparams(lr=1e-2, weight_decay=0.1, rounding=rounding, seed=SEED, wait_drill=True)
    before = [t.clone() for t in params + ms + vs]
    want_p, want_m, want_v = host(params), host(ms), host(vs)
    oracle_step(want_p, host(grads), want_m, want_v, v_dtype, rounding)

    plan.set_wait_limit(DRILL_LIMIT_NS)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    plan.adamw_step(drill, 1)
    flags = plan.status()
    took = time.perf_counter() - t0
    assert flags & ps.OPT_FLAG_WAIT_TIMEOUT, "the drill's waits did not run out"
    assert not flags & ps.OPT_FLAG_DRAIN_TIMEOUT, "issued copies did not land before the kernel left"
    assert plan.status() == 0, "opt_plan_status did not clear the flags"
    assert took < 5.0, f"the drill took {took:.2f} s with a 1 ms wait limit"
    for k, (now, was) in enumerate(zip(params + ms + vs, before)):
        assert torch.equal(now.view(torch.uint8), was.view(torch.uint8)), f"buffer {k} changed in the drill"
    g.check(f"drill ({v_dtype} {rounding})")

    # the same plan, its limit back to the default: a complete step that
    # equals the oracle's
    plan.set_wait_limit(2_000_000_000)
    plan.adamw_step(hp, 1)
    assert plan.status() == 0
    check_against_oracle(params, ms, vs, want_p, want_m, want_v, v_dtype, rounding)
    g.check(f"step after the drill ({v_dtype} {rounding})")
    plan.close()

    # a fresh plan over fresh buffers: the same step, the same result
    g2 = Guarded()
    params, grads, ms, vs = make_lists(g2, v_dtype, seed=3)
    plan = ps.Plan(params, grads, ms, vs, m_dtype="bf16", v_dtype=v_dtype)
    plan.adamw_step(hp, 1)
    assert plan.status() == 0
    check_against_oracle(params, ms, vs, want_p, want_m, want_v, v_dtype, rounding)
    g2.check(f"fresh plan ({v_dtype} {rounding})")
    plan.close()


def test_wait_limit_and_drill_rejections():
    """Limits above 10 s are rejected; the drill only exists for the steps
    that run the staged kernel."""
    g = Guarded()
    params, grads, ms, vs = make_lists(g, "e4m3", seed=4)
    plan = ps.Plan(params, grads, ms, vs, m_dtype="bf16", v_dtype="e4m3")
    plan.set_wait_limit(10_000_000_000)
    with pytest.raises(ps.OptError) as e:
        plan.set_wait_limit(10_000_000_001)
    assert e.value.status == ps.OPT_EINVAL
    with pytest.raises(ps.OptError) as e:        # nearest E4M3 v: register-pipelined kernel
        plan.adamw_step(ps.hparams(rounding="nearest", wait_drill=True), 1)
    assert e.value.status == ps.OPT_EUNSUPPORTED
    plan.close()
