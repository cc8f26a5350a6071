"""Plain CPU oracle for the fused optimizer step -- TEST INFRASTRUCTURE ONLY.

This package is the slow, obviously-correct definition that the CUDA library
is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the product path
(``precision_states_gb300``) never does, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, scalar loops, built with
``-O2 -ffp-contract=off``); this module compiles it with gcc and wraps it for
numpy arrays.  What each function computes, and the passage it follows, is
documented in ``oracle.h``/``oracle.c``.

Parity pins (tests/test_oracle_*.py): codecs against torch casts, brute force
and the carry rule of "When Small Updates Disappear" sec. 6.1; the norm
against exact rational arithmetic; the step against the one-step closed form
of bitsandbytes PR #2040 and against torch.optim.AdamW in float64; Philox
against the independent host-side Philox4_32_10 generator of cuRAND.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_SRC = [os.path.join(_HERE, "oracle.c")]
_HDR = os.path.join(_HERE, "oracle.h")

F32, BF16, E4M3, E2M2, F64 = 0, 1, 2, 3, 4
ADAMW, ADEMAMIX = 0, 1
# planted mistakes (ORC_MUT_* in oracle.h), for tests that show a pin is not vacuous
MUT_DECAY_AFTER, MUT_U_FROM_CODES, MUT_NO_BIAS_CORR, MUT_SCALE_IN_SQRT = 1, 2, 4, 8

_DT = {"f32": F32, "bf16": BF16, "e4m3": E4M3, "e2m2": E2M2, "f64": F64}


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (the checker, not the product)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(p) for p in _SRC + [_HDR])
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp] + _SRC + ["-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _SO)
    return _SO


_lib = None
_lock = threading.Lock()


class SumSq(ctypes.Structure):
    _fields_ = [("sum", ctypes.c_double), ("comp", ctypes.c_double),
                ("maxabs", ctypes.c_float), ("nan_count", ctypes.c_uint64),
                ("inf_count", ctypes.c_uint64)]


class Norm(ctypes.Structure):
    _fields_ = [("sumsq", ctypes.c_double), ("norm2", ctypes.c_double),
                ("norm_inf", ctypes.c_double), ("nan_count", ctypes.c_uint64),
                ("inf_count", ctypes.c_uint64), ("clip_coef", ctypes.c_float),
                ("status", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


class HParams(ctypes.Structure):
    _fields_ = [(k, ctypes.c_float) for k in
                ("lr", "beta1", "beta2", "beta3", "alpha", "eps", "weight_decay")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u8, u16, u32, f32, f64 = (ctypes.c_uint8, ctypes.c_uint16, ctypes.c_uint32,
                                      ctypes.c_float, ctypes.c_double)
            i32, i64, u64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
            L.oracle_bf16_decode.argtypes, L.oracle_bf16_decode.restype = [u16], f32
            L.oracle_bf16_encode.argtypes, L.oracle_bf16_encode.restype = [f32, ctypes.c_int, u32], u16
            L.oracle_e4m3_decode.argtypes, L.oracle_e4m3_decode.restype = [u8], f32
            L.oracle_e4m3_encode.argtypes, L.oracle_e4m3_encode.restype = [f32, ctypes.c_int, u32], u8
            L.oracle_e2m2_decode.argtypes, L.oracle_e2m2_decode.restype = [u8], f32
            L.oracle_e2m2_encode.argtypes, L.oracle_e2m2_encode.restype = [f32, ctypes.c_int, u32], u8
            L.oracle_philox4x32_10.argtypes = [ctypes.POINTER(u32)] * 3
            L.oracle_philox4x32_10.restype = None
            L.oracle_draws.argtypes = [u64, i64, u32, i64, ctypes.POINTER(u32), ctypes.POINTER(u32)]
            L.oracle_draws.restype = None
            L.oracle_cast_draw.argtypes = [u64, i64, u32, i64]
            L.oracle_cast_draw.restype = u32
            L.oracle_tensor_sumsq.argtypes = [i64, vp, ctypes.c_int, ctypes.POINTER(SumSq)]
            L.oracle_tensor_sumsq.restype = None
            L.oracle_norm_finish.argtypes = [i32, ctypes.POINTER(SumSq), f64, ctypes.POINTER(Norm)]
            L.oracle_norm_finish.restype = None
            L.oracle_grad_norm.argtypes = [i32, ctypes.POINTER(i64), ctypes.POINTER(vp),
                                           ctypes.POINTER(i32), f64, ctypes.POINTER(Norm)]
            L.oracle_grad_norm.restype = None
            L.oracle_clip_coef.argtypes, L.oracle_clip_coef.restype = [f64, f64], f32
            L.oracle_adam_tensor.argtypes = [
                ctypes.c_int, i64, vp, ctypes.c_int, vp, ctypes.c_int, vp, vp, ctypes.c_int,
                vp, ctypes.c_int, ctypes.POINTER(HParams), i64, f32, ctypes.c_int, u64, u32,
                i64, f64, ctypes.c_int, ctypes.POINTER(i64)]
            L.oracle_adam_tensor.restype = ctypes.c_int
            L.oracle_lamb_tensor.argtypes = [i64, vp, vp, ctypes.c_int, vp, vp, ctypes.POINTER(HParams),
                                             i64, f32, f32, ctypes.POINTER(f64)]
            L.oracle_lamb_tensor.restype = ctypes.c_int
            _lib = L
    return _lib


# ---------------------------------------------------------------- codecs
def bf16_decode(code: int) -> float:
    return lib().oracle_bf16_decode(code)


def bf16_encode(x: float, stochastic: bool = False, r16: int = 0) -> int:
    return lib().oracle_bf16_encode(x, int(stochastic), r16)


def e4m3_decode(code: int) -> float:
    return lib().oracle_e4m3_decode(code)


def e4m3_encode(x: float, stochastic: bool = False, r16: int = 0) -> int:
    return lib().oracle_e4m3_encode(x, int(stochastic), r16)


def e2m2_decode(code: int) -> float:
    return lib().oracle_e2m2_decode(code)


def e2m2_encode(x: float, stochastic: bool = False, r16: int = 0) -> int:
    return lib().oracle_e2m2_encode(x, int(stochastic), r16)


def philox4x32_10(ctr, key):
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    o = (ctypes.c_uint32 * 4)()
    lib().oracle_philox4x32_10(c, k, o)
    return tuple(o)


def draws(seed: int, step: int, tensor_index: int, index: int):
    a, b = ctypes.c_uint32(), ctypes.c_uint32()
    lib().oracle_draws(seed, step, tensor_index, index, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def cast_draw(seed: int, step: int, tensor_index: int, index: int) -> int:
    """The standalone cast's 16-bit draw for element `index`."""
    return lib().oracle_cast_draw(seed, step, tensor_index, index)


# ------------------------------------------------------------------ norm
def _grad_dtype(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:       # BF16 codes
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"gradient array dtype {a.dtype} (use float32, uint16 BF16 codes, float64)")


def tensor_sumsq(g: np.ndarray) -> SumSq:
    g = np.ascontiguousarray(g)
    out = SumSq()
    lib().oracle_tensor_sumsq(g.size, g.ctypes.data, _grad_dtype(g), ctypes.byref(out))
    return out


def norm_finish(parts, max_norm: float) -> dict:
    arr = (SumSq * len(parts))(*parts)
    out = Norm()
    lib().oracle_norm_finish(len(parts), arr, float(max_norm), ctypes.byref(out))
    return out.as_dict()


def grad_norm(grads, max_norm: float = 0.0) -> dict:
    """Global norm over a list of gradient arrays (float32, float64, or uint16
    BF16 codes).  Returns the oracle_norm fields as a dict."""
    grads = [np.ascontiguousarray(g) for g in grads]
    n = len(grads)
    numel = (ctypes.c_int64 * max(n, 1))(*[g.size for g in grads])
    ptrs = (ctypes.c_void_p * max(n, 1))(*[g.ctypes.data for g in grads])
    dts = (ctypes.c_int32 * max(n, 1))(*[_grad_dtype(g) for g in grads])
    out = Norm()
    lib().oracle_grad_norm(n, numel, ptrs, dts, float(max_norm), ctypes.byref(out))
    return out.as_dict()


def clip_coef(norm2: float, max_norm: float) -> float:
    return lib().oracle_clip_coef(norm2, max_norm)


# ------------------------------------------------------------------ step
def hparams(lr=1e-3, beta1=0.9, beta2=0.999, beta3=0.9999, alpha=5.0, eps=1e-8,
            weight_decay=0.0) -> HParams:
    return HParams(lr, beta1, beta2, beta3, alpha, eps, weight_decay)


def adam_tensor(algo: int, p: np.ndarray, g: np.ndarray, m: np.ndarray, v: np.ndarray,
                hp: HParams, step: int, *, m2: np.ndarray | None = None, m_dtype="f32",
                v_dtype="f32", coef: float = 1.0, stochastic: bool = False, seed: int = 0,
                tensor_index: int = 0, index_base: int = 0, v_scale: float = 1.0,
                decay_after: bool = False, mutation: int = 0) -> int:
    """One step on one tensor, in place.  p: float32 (or float64 with every
    other array float64).  g: float32 or uint16 BF16 codes.  m/m2: float32 or
    uint16 BF16 codes.  v: float32, uint16 BF16, uint8 E4M3 codes, or uint8
    packed E2M2 (ceil(n/2) bytes).  Element i of the arrays is element
    index_base + i of the tensor (selects the stochastic-rounding draws).
    `mutation` (MUT_* bits, 0 = the oracle) plants a mistake for tests that
    show the pins catch it.  Returns the count of v codes unchanged."""
    for a in (p, g, m, v) + ((m2,) if m2 is not None else ()):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays must be C-contiguous")
    n = p.size
    p_dt = F64 if p.dtype == np.float64 else F32
    g_dt = _grad_dtype(g)
    unchanged = ctypes.c_int64()
    rc = lib().oracle_adam_tensor(
        algo, n, p.ctypes.data, p_dt, g.ctypes.data, g_dt, m.ctypes.data,
        None if m2 is None else m2.ctypes.data, _DT[m_dtype] if p_dt != F64 else F64,
        v.ctypes.data, _DT[v_dtype] if p_dt != F64 else F64, ctypes.byref(hp), int(step),
        float(coef), int(stochastic), int(seed), int(tensor_index), int(index_base), float(v_scale),
        int(mutation) | (MUT_DECAY_AFTER if decay_after else 0),
        ctypes.byref(unchanged))
    if rc != 0:
        raise ValueError("unsupported oracle combination")
    return unchanged.value


def lamb_tensor(p: np.ndarray, g: np.ndarray, m: np.ndarray, v: np.ndarray, hp: HParams, step: int,
                max_unorm: float, coef: float = 1.0) -> float:
    """LAMB-style update-norm clipping step on one tensor (FP32 p, m, v; g
    float32 or uint16 BF16 codes), in place.  Returns the ratio applied."""
    for a in (p, m, v):
        if a.dtype != np.float32 or not a.flags["C_CONTIGUOUS"]:
            raise ValueError("p, m, v must be contiguous float32")
    ratio = ctypes.c_double()
    rc = lib().oracle_lamb_tensor(p.size, p.ctypes.data, g.ctypes.data, _grad_dtype(g), m.ctypes.data,
                                  v.ctypes.data, ctypes.byref(hp), int(step), float(coef),
                                  float(max_unorm), ctypes.byref(ratio))
    if rc != 0:
        raise ValueError("unsupported oracle combination")
    return ratio.value
