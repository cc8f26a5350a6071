"""Python binding of the GB300 fused optimizer-step library (libpsopt.so).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels, reached through the C ABI declared in include/opt.h.  The functions
below carry the C names; ``Plan`` is a convenience that builds an
``opt_tensor_list`` from torch tensors (torch is used only for device memory
and streams).  There is no fallback: if the shared library is missing or was
built without its kernels, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpsopt.so")

# ------------------------------------------------------------------ constants
OPT_OK, OPT_ENONFINITE = 0, 1
OPT_EINVAL, OPT_EUNSUPPORTED, OPT_EALIGN, OPT_ECUDA, OPT_ENOMEM, OPT_ELIMIT = -1, -2, -3, -4, -5, -6
OPT_NOALLOC_MAX_TENSORS, OPT_NOALLOC_MAX_CHUNKS = 8192, 262144
OPT_F32, OPT_BF16, OPT_E4M3, OPT_E2M2 = 0, 1, 2, 3
OPT_ROUND_NEAREST, OPT_ROUND_STOCHASTIC = 0, 1
OPT_STEP_RESET_STATES = 1
OPT_STEP_DEVICE_COUNTER = 2
OPT_STEP_WAIT_DRILL = 4
OPT_FLAG_WAIT_TIMEOUT, OPT_FLAG_DRAIN_TIMEOUT = 1, 2
OPT_NORM_CHUNK_MIN, OPT_CHUNK_ELEMS = 4096, 32768
OPT_NORM_SLOTS, OPT_NORM_MAX_PART = 152, 4096

DTYPES = {"f32": OPT_F32, "bf16": OPT_BF16, "e4m3": OPT_E4M3, "e2m2": OPT_E2M2}

_c = ctypes
_vp = _c.c_void_p


class opt_tensor_list(_c.Structure):
    _fields_ = [("n", _c.c_int32), ("numel", _c.POINTER(_c.c_int64)),
                ("param", _c.POINTER(_vp)), ("grad", _c.POINTER(_vp)),
                ("m", _c.POINTER(_vp)), ("v", _c.POINTER(_vp)), ("m2", _c.POINTER(_vp)),
                ("grad_dtype", _c.POINTER(_c.c_int32)), ("param_dtype", _c.c_int32),
                ("m_dtype", _c.c_int32), ("v_dtype", _c.c_int32), ("v_scale", _c.POINTER(_c.c_float))]


class opt_hparams(_c.Structure):
    _fields_ = [("lr", _c.c_float), ("beta1", _c.c_float), ("beta2", _c.c_float),
                ("beta3", _c.c_float), ("alpha", _c.c_float), ("eps", _c.c_float),
                ("weight_decay", _c.c_float), ("rounding", _c.c_int32), ("seed", _c.c_uint64),
                ("count_unchanged", _c.c_int32), ("flags", _c.c_int32)]


class opt_norm_result(_c.Structure):
    _fields_ = [("sumsq", _c.c_double), ("norm2", _c.c_double), ("norm_inf", _c.c_double),
                ("nan_count", _c.c_uint64), ("inf_count", _c.c_uint64),
                ("clip_coef", _c.c_float), ("status", _c.c_int32)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


class opt_chunk(_c.Structure):
    _fields_ = [("tensor", _c.c_uint32), ("len", _c.c_uint32), ("start", _c.c_int64)]


class opt_step_scalars(_c.Structure):
    _fields_ = [(k, _c.c_float) for k in ("lr", "decay", "beta1", "omb1", "beta2", "omb2",
                                          "beta3", "omb3", "alpha", "eps", "inv_bc1", "inv_bc2")]


# the C ABI: name -> (restype, argtypes)
_SIGS = {
    "opt_version": (_c.c_int, []),
    "opt_strerror": (_c.c_char_p, [_c.c_int]),
    "opt_plan_create": (_c.c_int, [_c.POINTER(opt_tensor_list), _c.POINTER(_vp)]),
    "opt_plan_destroy": (None, [_vp]),
    "opt_plan_info": (_c.c_int, [_vp, _c.POINTER(_c.c_int64), _c.POINTER(_c.c_int64),
                                 _c.POINTER(_c.c_int64)]),
    "opt_plan_norm_buffer": (_vp, [_vp]),
    "opt_grad_norm": (_c.c_int, [_vp, _c.c_double, _vp, _c.POINTER(opt_norm_result), _vp]),
    "opt_grad_norm_noalloc": (_c.c_int, [_c.c_int32, _c.POINTER(_c.c_int64), _c.POINTER(_vp),
                                         _c.POINTER(_c.c_int32), _c.c_double, _vp, _vp]),
    "opt_adamw_step": (_c.c_int, [_vp, _c.POINTER(opt_hparams), _c.c_int64, _vp, _vp]),
    "opt_ademamix_step": (_c.c_int, [_vp, _c.POINTER(opt_hparams), _c.c_int64, _vp, _vp]),
    "opt_lamb_step": (_c.c_int, [_vp, _c.POINTER(opt_hparams), _c.c_int64, _c.c_float, _vp, _vp]),
    "opt_unchanged_count": (_c.c_int, [_vp, _c.POINTER(_c.c_uint64), _vp]),
    "opt_plan_status": (_c.c_int, [_vp, _c.POINTER(_c.c_int32), _vp]),
    "opt_plan_set_step": (_c.c_int, [_vp, _c.c_int64, _vp]),
    "opt_plan_set_wait_limit": (_c.c_int, [_vp, _c.c_uint64]),
    "opt_grads_upload": (_c.c_int, [_vp, _c.POINTER(_vp), _vp]),
    "opt_encode": (_c.c_int, [_vp, _vp, _c.c_int64, _c.c_int32, _c.c_int32, _c.c_uint64,
                              _c.c_uint32, _c.c_int64, _vp]),
    "opt_decode": (_c.c_int, [_vp, _vp, _c.c_int64, _c.c_int32, _vp]),
    "opt_chunk_table": (_c.c_int64, [_c.c_int32, _c.POINTER(_c.c_int64), _c.POINTER(_c.c_int32),
                                     _c.POINTER(opt_chunk), _c.c_int64, _c.POINTER(_c.c_int64)]),
    "opt_norm_chunk_elems": (_c.c_int64, [_c.c_int32, _c.POINTER(_c.c_int64), _c.POINTER(_c.c_int32),
                                          _c.c_int32]),
    "opt_step_scalars_compute": (_c.c_int, [_c.POINTER(opt_hparams), _c.c_int64,
                                            _c.POINTER(opt_step_scalars)]),
    "opt_norm_combine": (_c.c_int, [_c.POINTER(opt_norm_result), _c.c_int32, _c.c_double,
                                    _c.POINTER(opt_norm_result)]),
}
EXPORTED = tuple(_SIGS)

_lib = None
_lock = threading.Lock()


def lib():
    """Load libpsopt.so (built by ``precision_states_gb300.build``).  Raises if
    it is missing: the library has no CPU fallback."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: run precision_states_gb300.build.build() "
                                   "(needs nvcc); there is no fallback path")
            L = _c.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


class OptError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {opt_strerror(status)} ({status})")
        self.status = status


def _check(status: int, what: str) -> int:
    if status < 0:
        raise OptError(status, what)
    return status


# ------------------------------------------------------------ thin wrappers
def opt_version() -> int:
    return lib().opt_version()


def opt_strerror(status: int) -> str:
    return lib().opt_strerror(status).decode()


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, beta3=0.9999, alpha=5.0, eps=1e-8, weight_decay=0.0,
            rounding="nearest", seed=0, count_unchanged=False, reset_states=False,
            device_step=False, wait_drill=False) -> opt_hparams:
    r = OPT_ROUND_STOCHASTIC if rounding in ("stochastic", "sr", OPT_ROUND_STOCHASTIC) else OPT_ROUND_NEAREST
    return opt_hparams(lr, beta1, beta2, beta3, alpha, eps, weight_decay, r, seed,
                       1 if count_unchanged else 0,
                       (OPT_STEP_RESET_STATES if reset_states else 0) |
                       (OPT_STEP_DEVICE_COUNTER if device_step else 0) |
                       (OPT_STEP_WAIT_DRILL if wait_drill else 0))


def opt_chunk_table(numel, grad_dtype):
    """Host-only chunk table: returns (list of (tensor, len, start), bucket_begin)."""
    n = len(numel)
    ne = (_c.c_int64 * max(n, 1))(*numel)
    gd = (_c.c_int32 * max(n, 1))(*grad_dtype)
    bb = (_c.c_int64 * 3)()
    cnt = _check(lib().opt_chunk_table(n, ne, gd, None, 0, bb), "opt_chunk_table")
    out = (opt_chunk * max(cnt, 1))()
    lib().opt_chunk_table(n, ne, gd, out, cnt, bb)
    return [(out[i].tensor, out[i].len, out[i].start) for i in range(cnt)], list(bb)


def opt_norm_chunk_elems(numel, grad_dtype, bucket: int) -> int:
    """Host-only: the norm's chunk size for gradient-dtype bucket 0 (FP32) or 1 (BF16)."""
    n = len(numel)
    ne = (_c.c_int64 * max(n, 1))(*numel)
    gd = (_c.c_int32 * max(n, 1))(*grad_dtype)
    return _check(lib().opt_norm_chunk_elems(n, ne, gd, bucket), "opt_norm_chunk_elems")


def opt_step_scalars_compute(hp: opt_hparams, step: int) -> dict:
    out = opt_step_scalars()
    _check(lib().opt_step_scalars_compute(_c.byref(hp), step, _c.byref(out)), "opt_step_scalars_compute")
    return {k: getattr(out, k) for k, _ in out._fields_}


def opt_norm_combine(parts, max_norm: float) -> opt_norm_result:
    arr = (opt_norm_result * max(len(parts), 1))(*parts)
    out = opt_norm_result()
    _check(lib().opt_norm_combine(arr, len(parts), max_norm, _c.byref(out)), "opt_norm_combine")
    return out


def _stream_ptr(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def opt_encode(x, out, dtype: str, rounding="nearest", seed=0, tensor_index=0, step=0, stream=None):
    """x: float32 CUDA tensor; out: uint8/int16 CUDA tensor of the encoded size."""
    r = OPT_ROUND_STOCHASTIC if rounding in ("stochastic", "sr") else OPT_ROUND_NEAREST
    _check(lib().opt_encode(x.data_ptr(), out.data_ptr(), x.numel(), DTYPES[dtype], r, seed,
                            tensor_index, step, _stream_ptr(stream)), "opt_encode")


def opt_decode(codes, out, n: int, dtype: str, stream=None):
    _check(lib().opt_decode(codes.data_ptr(), out.data_ptr(), n, DTYPES[dtype], _stream_ptr(stream)),
           "opt_decode")


def state_nbytes(dtype: str, n: int) -> int:
    return {"f32": 4 * n, "bf16": 2 * n, "e4m3": n, "e2m2": (n + 1) // 2}[dtype]


class Plan:
    """A plan over lists of CUDA torch tensors (kept alive by the plan).

    params: float32; grads: bfloat16 or float32 (per tensor); m, v, m2: the
    storage of the chosen state dtypes (float32, or raw code tensors such as
    int16/uint8 for BF16/E4M3/E2M2 -- only their data pointers are used)."""

    def __init__(self, params, grads, m, v, m2=None, m_dtype="f32", v_dtype="f32", v_scale=None):
        import torch
        n = len(params)
        if not (len(grads) == len(m) == len(v) == n) or (m2 is not None and len(m2) != n):
            raise ValueError("tensor lists differ in length")
        for t in list(params) + list(grads) + list(m) + list(v) + (list(m2) if m2 else []):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError("every tensor must be a contiguous CUDA tensor")
        self._keep = (params, grads, m, v, m2)
        gd = []
        for g in grads:
            if g.dtype == torch.bfloat16:
                gd.append(OPT_BF16)
            elif g.dtype == torch.float32:
                gd.append(OPT_F32)
            else:
                raise OptError(OPT_EUNSUPPORTED, f"gradient dtype {g.dtype}")
        self.numel = [p.numel() for p in params]
        self.grad_dtype = gd
        arr = lambda ts: (_vp * max(n, 1))(*[t.data_ptr() for t in ts])
        self._arrays = dict(numel=(_c.c_int64 * max(n, 1))(*self.numel), param=arr(params),
                            grad=arr(grads), m=arr(m), v=arr(v), m2=arr(m2) if m2 else None,
                            gd=(_c.c_int32 * max(n, 1))(*gd),
                            vs=(_c.c_float * max(n, 1))(*v_scale) if v_scale is not None else None)
        a = self._arrays
        tl = opt_tensor_list(n, a["numel"], a["param"], a["grad"], a["m"], a["v"], a["m2"], a["gd"],
                             OPT_F32, DTYPES[m_dtype], DTYPES[v_dtype], a["vs"])
        h = _vp()
        _check(lib().opt_plan_create(_c.byref(tl), _c.byref(h)), "opt_plan_create")
        self.handle = h
        self.m_dtype, self.v_dtype = m_dtype, v_dtype

    def close(self):
        if getattr(self, "handle", None):
            lib().opt_plan_destroy(self.handle)
            self.handle = None
        self._keep = None          # the tensors are free to go with the plan

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def info(self) -> dict:
        a, b, c = _c.c_int64(), _c.c_int64(), _c.c_int64()
        _check(lib().opt_plan_info(self.handle, _c.byref(a), _c.byref(b), _c.byref(c)), "opt_plan_info")
        return {"n_chunks": a.value, "total_numel": b.value, "workspace_bytes": c.value}

    def norm_buffer(self) -> int:
        return lib().opt_plan_norm_buffer(self.handle)

    def grad_norm(self, max_norm: float = 0.0, d_out: int | None = None, sync: bool = True,
                  stream=None) -> opt_norm_result | None:
        h = opt_norm_result() if sync else None
        st = lib().opt_grad_norm(self.handle, max_norm, d_out, _c.byref(h) if sync else None,
                                 _stream_ptr(stream))
        _check(st, "opt_grad_norm")
        return h

    def adamw_step(self, hp: opt_hparams, step: int, d_norm: int | None = None, stream=None):
        _check(lib().opt_adamw_step(self.handle, _c.byref(hp), step, d_norm, _stream_ptr(stream)),
               "opt_adamw_step")

    def ademamix_step(self, hp: opt_hparams, step: int, d_norm: int | None = None, stream=None):
        _check(lib().opt_ademamix_step(self.handle, _c.byref(hp), step, d_norm, _stream_ptr(stream)),
               "opt_ademamix_step")

    def lamb_step(self, hp: opt_hparams, step: int, max_unorm: float, d_norm: int | None = None,
                  stream=None):
        _check(lib().opt_lamb_step(self.handle, _c.byref(hp), step, max_unorm, d_norm, _stream_ptr(stream)),
               "opt_lamb_step")

    def unchanged_count(self, stream=None) -> int:
        out = _c.c_uint64()
        _check(lib().opt_unchanged_count(self.handle, _c.byref(out), _stream_ptr(stream)),
               "opt_unchanged_count")
        return out.value

    def set_step(self, next_step: int, stream=None):
        """Set the device step counter: the next step taken with
        device_step=True (step argument 0) is `next_step`."""
        _check(lib().opt_plan_set_step(self.handle, next_step, _stream_ptr(stream)), "opt_plan_set_step")

    def status(self, stream=None) -> int:
        """Kernel error flags since the last call (0: all ran to completion)."""
        out = _c.c_int32()
        _check(lib().opt_plan_status(self.handle, _c.byref(out), _stream_ptr(stream)), "opt_plan_status")
        return out.value

    def set_wait_limit(self, ns: int):
        """Limit of each wait of the staged step kernel, in ns (0 .. 10 s)."""
        _check(lib().opt_plan_set_wait_limit(self.handle, ns), "opt_plan_set_wait_limit")

    def grads_upload(self, host_grads, stream=None):
        """Copy host gradients (one tensor per list entry, the plan's sizes and
        gradient dtypes) into the plan's device gradients on `stream`."""
        if len(host_grads) != len(self.numel):
            raise ValueError("host gradient list differs in length from the plan's")
        for i, t in enumerate(host_grads):
            want = 2 if self.grad_dtype[i] == OPT_BF16 else 4
            if t.numel() != self.numel[i] or t.element_size() != want or not t.is_contiguous():
                raise ValueError(f"host gradient {i}: expected {self.numel[i]} contiguous elements of "
                                 f"{want} bytes")
        arr = (_vp * max(len(host_grads), 1))(*[t.data_ptr() for t in host_grads])
        _check(lib().opt_grads_upload(self.handle, arr, _stream_ptr(stream)), "opt_grads_upload")
