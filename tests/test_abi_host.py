"""CPU tests of the C ABI: the library loads and exports every function that
include/opt.h declares; the host-only logic (chunk table, per-step scalars,
cross-rank combine, argument validation) is correct.  No GPU compute."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import precision_states_gb300 as ps
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "opt.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(opt_[a-z0-9_]+)\s*\(", src)))


def test_header_declarations_exported():
    lib = ps.lib()
    names = declared_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(lib, name), f"{name} declared in opt.h but not exported"
    assert sorted(ps.EXPORTED) == names, "binding and header disagree"


def test_exports_via_nm():
    import shutil
    import subprocess
    if shutil.which("nm") is None:
        pytest.skip("nm not available")
    out = subprocess.run(["nm", "-D", "--defined-only", ps.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (opt_\w+)", out))
    assert set(declared_functions()) <= exported


def test_version_and_strerror():
    assert ps.opt_version() == 2
    for code in (0, 1, -1, -2, -3, -4, -5, 99):
        assert isinstance(ps.opt_strerror(code), str) and ps.opt_strerror(code)


def test_struct_sizes_match_header_layout():
    assert ctypes.sizeof(ps.opt_norm_result) == 48
    assert ctypes.sizeof(ps.opt_chunk) == 16
    assert ctypes.sizeof(ps.opt_step_scalars) == 48
    assert ctypes.sizeof(ps.opt_hparams) == 48


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_chunk_table_covers_each_tensor_once(seed):
    rng = np.random.default_rng(seed)
    numel = [int(x) for x in rng.choice([0, 1, 7, 32767, 32768, 32769, 100000, 262144 + 5], 40)]
    gd = [int(x) for x in rng.choice([ps.OPT_F32, ps.OPT_BF16], 40)]
    table, bb = ps.opt_chunk_table(numel, gd)
    ch = [ps.opt_norm_chunk_elems(numel, gd, b) for b in (0, 1)]
    assert ch == [ps.OPT_NORM_CHUNK_MIN] * 2          # small buckets: the smallest chunks
    CH = {ps.OPT_F32: ch[0], ps.OPT_BF16: ch[1]}
    assert bb[0] == 0 and bb[2] == len(table)
    assert len(table) == sum((n + CH[d] - 1) // CH[d] for n, d in zip(numel, gd))
    for k, (t, ln, start) in enumerate(table):
        bucket = 0 if k < bb[1] else 1
        assert gd[t] == (ps.OPT_F32 if bucket == 0 else ps.OPT_BF16)
        c = CH[gd[t]]
        assert 1 <= ln <= c and start % c == 0 and start + ln <= numel[t]
    covered = {}
    for t, ln, start in table:
        covered.setdefault(t, []).append((start, ln))
    for t, n in enumerate(numel):
        segs = covered.get(t, [])
        assert [s for s, _ in segs] == list(range(0, n, CH[gd[t]]))       # in element order
        assert sum(ln for _, ln in segs) == n
    # tensors appear in list order within a bucket
    for lo, hi in ((0, bb[1]), (bb[1], bb[2])):
        ts = [table[k][0] for k in range(lo, hi)]
        assert ts == sorted(ts)


def test_norm_chunk_size_rule():
    """The norm's chunk size comes from a bucket's size alone: 4K elements
    below 2^28, 8K below 2^29, 16K below 2^31, 32K above, doubled while a
    slot would own more than OPT_NORM_MAX_PART chunks; the other bucket does
    not matter."""
    f = ps.opt_norm_chunk_elems
    B, F = ps.OPT_BF16, ps.OPT_F32
    assert f([], [], 0) == f([], [], 1) == ps.OPT_NORM_CHUNK_MIN
    assert ps.OPT_NORM_CHUNK_MIN == 4096
    assert f([(1 << 28) - 1], [B], 1) == 4096
    assert f([1 << 28], [B], 1) == 8192
    assert f([197_281_486], [B], 1) == 4096                # the 740-tensor list's size
    assert f([(1 << 29) - 1], [B], 1) == 8192
    assert f([1 << 29], [B], 1) == 16384
    assert f([(1 << 31) - 1], [B], 1) == 16384
    assert f([1 << 31], [B], 1) == 32768
    assert f([8_030_261_248], [B], 1) == 32768             # the Llama-3-8B list's size
    assert f([1 << 31, 5], [F, B], 1) == 4096              # buckets apart
    assert f([1 << 31, 5], [F, B], 0) == 32768
    # 32K chunks would give a slot more than OPT_NORM_MAX_PART: doubled
    lim = ps.OPT_NORM_SLOTS * ps.OPT_NORM_MAX_PART * 32768
    assert f([lim], [B], 1) == 32768
    assert f([lim + 1], [B], 1) == 65536
    # tensors beyond what the slots can hold, one chunk each at least
    many = ps.OPT_NORM_SLOTS * ps.OPT_NORM_MAX_PART + 1
    with pytest.raises(ps.OptError) as e:
        f([1] * many, [B] * many, 1)
    assert e.value.status == ps.OPT_ELIMIT
    with pytest.raises(ps.OptError):
        f([5], [B], 2)


def test_chunk_table_errors():
    assert ps.lib().opt_chunk_table(-1, None, None, None, 0, None) == ps.OPT_EINVAL
    with pytest.raises(ps.OptError):
        ps.opt_chunk_table([5, -1], [0, 0])
    with pytest.raises(ps.OptError) as e:
        ps.opt_chunk_table([5], [ps.OPT_E4M3])
    assert e.value.status == ps.OPT_EUNSUPPORTED


@pytest.mark.parametrize("step", [1, 2, 10, 1000])
def test_step_scalars_are_the_definitions(step):
    """Bias corrections and (1 - beta) formed once in double ("Investigate SM103
    bias-correction broadcast in 32-bit optimizers", 'Problem')."""
    hp = ps.hparams(lr=3e-4, beta1=0.9, beta2=0.999, beta3=0.9999, alpha=5.0, eps=1e-8, weight_decay=0.1)
    s = ps.opt_step_scalars_compute(hp, step)
    f = lambda x: float(np.float32(x))
    b1, b2, b3, lr, wd = f(0.9), f(0.999), f(0.9999), f(3e-4), f(0.1)
    assert s["inv_bc1"] == f(1.0 / (1.0 - b1 ** step))
    assert s["inv_bc2"] == f(1.0 / (1.0 - b2 ** step))
    assert s["omb1"] == f(1.0 - b1) and s["omb2"] == f(1.0 - b2) and s["omb3"] == f(1.0 - b3)
    assert s["decay"] == f(1.0 - lr * wd)
    assert s["lr"] == lr and s["alpha"] == 5.0 and s["eps"] == f(1e-8)


def test_step_scalars_reject_step_zero():
    with pytest.raises(ps.OptError):
        ps.opt_step_scalars_compute(ps.hparams(), 0)


def _nr(sumsq, ninf, nan=0, inf=0):
    r = ps.opt_norm_result()
    r.sumsq, r.norm2, r.norm_inf, r.nan_count, r.inf_count = sumsq, math.sqrt(sumsq), ninf, nan, inf
    return r


def test_norm_combine_rank_order_and_policy():
    parts = [_nr(4.0, 1.5), _nr(5.0, 2.0), _nr(0.0, 0.0)]
    out = ps.opt_norm_combine(parts, 1.0)
    assert out.sumsq == 9.0 and out.norm2 == 3.0 and out.norm_inf == 2.0 and out.status == 0
    assert out.clip_coef == np.float32(1.0 / (3.0 + 1e-6))
    assert ps.opt_norm_combine(parts, 0.0).clip_coef == 1.0
    nan = ps.opt_norm_combine(parts + [_nr(0.0, 0.0, nan=2, inf=1)], 1.0)
    assert math.isnan(nan.norm2) and nan.status == ps.OPT_ENONFINITE and nan.nan_count == 2
    inf = ps.opt_norm_combine(parts + [_nr(0.0, 0.0, inf=3)], 1.0)
    assert inf.norm2 == math.inf and inf.status == ps.OPT_ENONFINITE
    empty = ps.opt_norm_combine([], 1.0)
    assert empty.norm2 == 0.0 and empty.clip_coef == 1.0


def _tensor_list(n=1, numel=(8,), ptr=0x10000, dtype_p=0, m_dt=0, v_dt=0, gd=0):
    a = dict(numel=(ctypes.c_int64 * n)(*numel), ptrs=(ctypes.c_void_p * n)(*([ptr] * n)),
             gd=(ctypes.c_int32 * n)(*([gd] * n)))
    tl = ps.opt_tensor_list(n, a["numel"], a["ptrs"], a["ptrs"], a["ptrs"], a["ptrs"], None, a["gd"],
                            dtype_p, m_dt, v_dt, None)
    return tl, a


@pytest.mark.parametrize("kw,want", [
    (dict(numel=(-1,)), ps.OPT_EINVAL),
    (dict(ptr=0), ps.OPT_EINVAL),
    (dict(ptr=0x10008), ps.OPT_EALIGN),
    (dict(dtype_p=ps.OPT_BF16), ps.OPT_EUNSUPPORTED),
    (dict(m_dt=ps.OPT_F32, v_dt=ps.OPT_BF16), ps.OPT_EUNSUPPORTED),
    (dict(m_dt=ps.OPT_E4M3, v_dt=ps.OPT_E4M3), ps.OPT_EUNSUPPORTED),
    (dict(gd=ps.OPT_E4M3), ps.OPT_EUNSUPPORTED),
])
def test_plan_create_validates_before_any_cuda_call(kw, want):
    """Invalid descriptors are rejected on the host (the pointers here are
    fake and never dereferenced)."""
    tl, keep = _tensor_list(**kw)
    h = ctypes.c_void_p()
    assert ps.lib().opt_plan_create(ctypes.byref(tl), ctypes.byref(h)) == want
    assert not h.value


def test_plan_create_null_arguments():
    h = ctypes.c_void_p()
    assert ps.lib().opt_plan_create(None, ctypes.byref(h)) == ps.OPT_EINVAL
    tl, keep = _tensor_list()
    assert ps.lib().opt_plan_create(ctypes.byref(tl), None) == ps.OPT_EINVAL


def test_calls_on_null_plan():
    L = ps.lib()
    hp = ps.hparams()
    assert L.opt_grad_norm(None, 1.0, None, None, None) == ps.OPT_EINVAL
    assert L.opt_adamw_step(None, ctypes.byref(hp), 1, None, None) == ps.OPT_EINVAL
    assert L.opt_ademamix_step(None, ctypes.byref(hp), 1, None, None) == ps.OPT_EINVAL
    out = ctypes.c_uint64()
    assert L.opt_unchanged_count(None, ctypes.byref(out), None) == ps.OPT_EINVAL
    assert L.opt_grads_upload(None, None, None) == ps.OPT_EINVAL
    assert L.opt_plan_info(None, None, None, None) == ps.OPT_EINVAL
    L.opt_plan_destroy(None)


def test_codec_entry_validation():
    L = ps.lib()
    assert L.opt_encode(None, None, -1, ps.OPT_BF16, 0, 0, 0, 0, None) == ps.OPT_EINVAL
    assert L.opt_encode(None, None, 4, ps.OPT_F32, 0, 0, 0, 0, None) == ps.OPT_EUNSUPPORTED
    assert L.opt_encode(None, None, 4, ps.OPT_BF16, 3, 0, 0, 0, None) == ps.OPT_EINVAL
    assert L.opt_encode(0x10004, 0x10000, 4, ps.OPT_BF16, 0, 0, 0, 0, None) == ps.OPT_EALIGN
    assert L.opt_encode(None, None, 0, ps.OPT_BF16, 0, 0, 0, 0, None) == ps.OPT_OK
    assert L.opt_decode(None, None, 4, 9, None) == ps.OPT_EUNSUPPORTED


@pytest.mark.parametrize("scale", [3.0, 0.0, -2.0, float("inf"), float("nan"), 2.0 ** -120])
def test_plan_create_rejects_bad_v_scale(scale):
    tl, keep = _tensor_list(m_dt=ps.OPT_BF16, v_dt=ps.OPT_E4M3)
    sc = (ctypes.c_float * 1)(scale)
    tl.v_scale = sc
    h = ctypes.c_void_p()
    assert ps.lib().opt_plan_create(ctypes.byref(tl), ctypes.byref(h)) == ps.OPT_EINVAL


def test_plan_status_null_arguments():
    L = ps.lib()
    out = ctypes.c_int32()
    assert L.opt_plan_status(None, ctypes.byref(out), None) == ps.OPT_EINVAL
    assert ps.OPT_FLAG_WAIT_TIMEOUT == 1 and ps.OPT_FLAG_DRAIN_TIMEOUT == 2


def test_set_wait_limit_rejects_a_missing_plan():
    assert ps.lib().opt_plan_set_wait_limit(None, 0) == ps.OPT_EINVAL
    assert ps.lib().opt_plan_set_wait_limit(None, 2_000_000_000) == ps.OPT_EINVAL
    assert ps.OPT_STEP_WAIT_DRILL == 4 and ps.hparams(wait_drill=True).flags == 4


def test_set_step_and_step_flags_on_the_host():
    """opt_plan_set_step rejects a missing plan before any CUDA call, and
    the device-counter flag is the bit the header defines."""
    assert ps.lib().opt_plan_set_step(None, 1, None) == ps.OPT_EINVAL
    assert ps.OPT_STEP_DEVICE_COUNTER == 2 and ps.OPT_STEP_RESET_STATES == 1
    assert ps.hparams(device_step=True, reset_states=True).flags == 3


@pytest.mark.parametrize("field,value", [
    ("beta1", 1.0), ("beta1", -0.1), ("beta2", 1.0), ("beta3", 1.5), ("lr", -1e-3), ("eps", -1e-8),
    ("weight_decay", -0.1), ("lr", float("nan")), ("alpha", float("inf")), ("beta2", float("nan")),
])
def test_step_scalars_reject_out_of_range_hparams(field, value):
    """The ranges torch.optim.AdamW accepts, and finite."""
    hp = ps.hparams()
    setattr(hp, field, value)
    with pytest.raises(ps.OptError) as e:
        ps.opt_step_scalars_compute(hp, 1)
    assert e.value.status == ps.OPT_EINVAL
    L = ps.lib()
    assert L.opt_adamw_step(None, ctypes.byref(hp), 1, None, None) == ps.OPT_EINVAL


def test_step_scalars_accept_edge_hparams():
    hp = ps.hparams(lr=0.0, eps=0.0, weight_decay=0.0, beta1=0.0, beta2=0.0, beta3=1.0)
    s = ps.opt_step_scalars_compute(hp, 3)
    assert s["omb3"] == 0.0 and s["inv_bc1"] == 1.0 and s["inv_bc2"] == 1.0
