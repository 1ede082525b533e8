"""ctypes front end of the FP64 oracle in ``gdn_oracle.c``.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA path: it builds and loads its own C library and takes plain
NumPy arrays (bit patterns for bf16 / fp16 data).

What the oracle computes, and the pages each step follows, is stated in the
header comment of ``gdn_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdn_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libgdn_oracle.so")

F32, BF16, F16, F64 = 0, 1, 2, 3
ERRORS = {
    -1: "null argument",
    -2: "bad shape",
    -3: "num_accepted > spec_stride",
    -4: "q_len > spec_stride",
    -5: "slot index >= num_slots",
    -6: "token row out of range",
    -7: "slot or token row shared between sequences",
    -8: "out of memory",
}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available).  Returns the path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    base = ["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", SRC, "-o", LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


class Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int64), ("num_tokens", ctypes.c_int64),
        ("H_k", ctypes.c_int64), ("H_v", ctypes.c_int64),
        ("K", ctypes.c_int64), ("V", ctypes.c_int64),
        ("spec_stride", ctypes.c_int64), ("num_slots", ctypes.c_int64),
        ("state_dtype", ctypes.c_int32), ("num_threads", ctypes.c_int32),
        ("scale", ctypes.c_double), ("eps", ctypes.c_double),
        ("qk_eps", ctypes.c_double), ("softplus_threshold", ctypes.c_double),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p), ("norm_w", ctypes.c_void_p),
        ("state_indices", ctypes.c_void_p), ("num_accepted", ctypes.c_void_p),
        ("cu_seqlens", ctypes.c_void_p), ("spec_token_indx", ctypes.c_void_p),
        ("pool", ctypes.c_void_p),
        ("out_f64", ctypes.c_void_p), ("out_bf16", ctypes.c_void_p),
        ("states_f64", ctypes.c_void_p), ("states_T", ctypes.c_int64),
        ("q64", ctypes.c_void_p), ("k64", ctypes.c_void_p), ("v64", ctypes.c_void_p),
    ]


class Conv(ctypes.Structure):
    """Mirror of gdn_oracle_conv."""
    _fields_ = [
        ("conv_dim", ctypes.c_int64), ("width", ctypes.c_int64),
        ("state_len", ctypes.c_int64), ("num_conv_slots", ctypes.c_int64),
        ("x", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("bias", ctypes.c_void_p),
        ("conv_pool", ctypes.c_void_p), ("conv_in", ctypes.c_void_p), ("conv_out", ctypes.c_void_p),
    ]


def load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.gdn_oracle_spec_decode.argtypes = [ctypes.POINTER(Problem)]
            lib.gdn_oracle_spec_decode.restype = ctypes.c_int
            lib.gdn_oracle_decode_nonspec.argtypes = [ctypes.POINTER(Problem)]
            lib.gdn_oracle_decode_nonspec.restype = ctypes.c_int
            lib.gdn_oracle_prefill.argtypes = [ctypes.POINTER(Problem), ctypes.c_void_p, ctypes.c_void_p]
            lib.gdn_oracle_prefill.restype = ctypes.c_int
            lib.gdn_oracle_spec_decode_conv.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(Conv)]
            lib.gdn_oracle_spec_decode_conv.restype = ctypes.c_int
            for name in ("gdn_oracle_round_bf16", "gdn_oracle_round_f16", "gdn_oracle_round_f32",
                         "gdn_oracle_value_bf16", "gdn_oracle_value_f16"):
                getattr(lib, name).argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
                getattr(lib, name).restype = None
            _lib = lib
        return _lib


class OracleError(RuntimeError):
    pass


def _ptr(x):
    return None if x is None else x.ctypes.data


def _c(x, dtype):
    if x is None:
        return None
    x = np.ascontiguousarray(x)
    if x.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {x.dtype}")
    return x


_POOL_DTYPES = {F32: np.float32, BF16: np.uint16, F16: np.uint16, F64: np.float64}


def spec_decode(*, q, k, v, a, b, z, A_log, dt_bias, norm_w, pool, state_dtype,
                state_indices, num_accepted, cu_seqlens, spec_token_indx=None,
                num_tokens=None, scale=128 ** -0.5, eps=1e-5, qk_eps=1e-6,
                softplus_threshold=20.0, states_T=0, num_threads=1):
    """Run the step.  ``pool`` ([num_slots, H_v, K, V], state dtype bits) is
    updated in place.  Returns a dict with ``out_f64`` and ``out_bf16``
    ([num_tokens, H_v, V]; rows the step does not write are NaN / 0xFFFF) and,
    when states_T > 0, ``states`` ([batch, H_v, states_T, K, V] FP64 state
    after each token, NaN where no token ran)."""
    lib = load()
    q = _c(q, np.uint16); k = _c(k, np.uint16); v = _c(v, np.uint16)
    a = _c(a, np.uint16); b = _c(b, np.uint16); z = _c(z, np.uint16)
    A_log = _c(A_log, np.float32); dt_bias = _c(dt_bias, np.uint16); norm_w = _c(norm_w, np.uint16)
    idx = _c(state_indices, np.int32); acc = _c(num_accepted, np.int32)
    cu = _c(cu_seqlens, np.int32); sti = _c(spec_token_indx, np.int32)
    if pool.dtype != _POOL_DTYPES[state_dtype] or not pool.flags.c_contiguous:
        raise TypeError("pool must be a contiguous array of the state dtype's storage type")
    N = q.shape[0] if num_tokens is None else num_tokens
    H_k, K = q.shape[1], q.shape[2]
    H_v, V = v.shape[1], v.shape[2]
    batch, stride = idx.shape
    out_f64 = np.full((N, H_v, V), np.nan)
    out_bf16 = np.full((N, H_v, V), 0xFFFF, dtype=np.uint16)
    states = np.full((batch, H_v, states_T, K, V), np.nan) if states_T > 0 else None
    p = Problem(
        batch=batch, num_tokens=N, H_k=H_k, H_v=H_v, K=K, V=V, spec_stride=stride,
        num_slots=pool.shape[0], state_dtype=state_dtype, num_threads=num_threads,
        scale=scale, eps=eps, qk_eps=qk_eps, softplus_threshold=softplus_threshold,
        q=_ptr(q), k=_ptr(k), v=_ptr(v), a=_ptr(a), b=_ptr(b), z=_ptr(z),
        A_log=_ptr(A_log), dt_bias=_ptr(dt_bias), norm_w=_ptr(norm_w),
        state_indices=_ptr(idx), num_accepted=_ptr(acc), cu_seqlens=_ptr(cu),
        spec_token_indx=_ptr(sti), pool=pool.ctypes.data,
        out_f64=out_f64.ctypes.data, out_bf16=out_bf16.ctypes.data,
        states_f64=_ptr(states), states_T=states_T,
    )
    rc = lib.gdn_oracle_spec_decode(ctypes.byref(p))
    if rc != 0:
        raise OracleError(f"oracle rejected the problem: {ERRORS.get(rc, rc)}")
    return {"out_f64": out_f64, "out_bf16": out_bf16, "states": states}


def decode_nonspec(*, q, k, v, a, b, z, A_log, dt_bias, norm_w, pool, state_dtype,
                   slots, scale=128 ** -0.5, eps=1e-5, qk_eps=1e-6, softplus_threshold=20.0):
    """Ordinary one-token-per-sequence decode; sequence i is token row i and
    updates slot ``slots[i]`` in place."""
    lib = load()
    q = _c(q, np.uint16); k = _c(k, np.uint16); v = _c(v, np.uint16)
    a = _c(a, np.uint16); b = _c(b, np.uint16); z = _c(z, np.uint16)
    A_log = _c(A_log, np.float32); dt_bias = _c(dt_bias, np.uint16); norm_w = _c(norm_w, np.uint16)
    slots = _c(slots, np.int32)
    N, H_k, K = q.shape
    H_v, V = v.shape[1], v.shape[2]
    out_f64 = np.full((N, H_v, V), np.nan)
    out_bf16 = np.full((N, H_v, V), 0xFFFF, dtype=np.uint16)
    p = Problem(
        batch=slots.shape[0], num_tokens=N, H_k=H_k, H_v=H_v, K=K, V=V, spec_stride=1,
        num_slots=pool.shape[0], state_dtype=state_dtype, num_threads=1,
        scale=scale, eps=eps, qk_eps=qk_eps, softplus_threshold=softplus_threshold,
        q=_ptr(q), k=_ptr(k), v=_ptr(v), a=_ptr(a), b=_ptr(b), z=_ptr(z),
        A_log=_ptr(A_log), dt_bias=_ptr(dt_bias), norm_w=_ptr(norm_w),
        state_indices=_ptr(slots), pool=pool.ctypes.data,
        out_f64=out_f64.ctypes.data, out_bf16=out_bf16.ctypes.data,
    )
    rc = lib.gdn_oracle_decode_nonspec(ctypes.byref(p))
    if rc != 0:
        raise OracleError(f"oracle rejected the problem: {ERRORS.get(rc, rc)}")
    return {"out_f64": out_f64, "out_bf16": out_bf16}


def prefill(*, q, k, v, a, b, z, A_log, dt_bias, norm_w, pool, state_dtype, cu_seqlens,
            read_slots, write_slots, scale=128 ** -0.5, eps=1e-5, qk_eps=1e-6,
            softplus_threshold=20.0, final_states=False, num_threads=1):
    """Prefill over whole prompts: sequence i is rows cu_seqlens[i] ..
    cu_seqlens[i+1]-1, starts from slot read_slots[i] (zero state when < 0)
    and stores its final state in write_slots[i] (skipped when < 0).
    ``pool`` is updated in place.  Returns out_f64 / out_bf16 and, with
    final_states, the FP64 final state [batch, H_v, K, V]."""
    lib = load()
    q = _c(q, np.uint16); k = _c(k, np.uint16); v = _c(v, np.uint16)
    a = _c(a, np.uint16); b = _c(b, np.uint16); z = _c(z, np.uint16)
    A_log = _c(A_log, np.float32); dt_bias = _c(dt_bias, np.uint16); norm_w = _c(norm_w, np.uint16)
    cu = _c(cu_seqlens, np.int32)
    rd = _c(read_slots, np.int32); wr = _c(write_slots, np.int32)
    N, H_k, K = q.shape
    H_v, V = v.shape[1], v.shape[2]
    batch = rd.shape[0]
    out_f64 = np.full((N, H_v, V), np.nan)
    out_bf16 = np.full((N, H_v, V), 0xFFFF, dtype=np.uint16)
    states = np.full((batch, H_v, 1, K, V), np.nan) if final_states else None
    p = Problem(
        batch=batch, num_tokens=N, H_k=H_k, H_v=H_v, K=K, V=V, spec_stride=1,
        num_slots=pool.shape[0], state_dtype=state_dtype, num_threads=num_threads,
        scale=scale, eps=eps, qk_eps=qk_eps, softplus_threshold=softplus_threshold,
        q=_ptr(q), k=_ptr(k), v=_ptr(v), a=_ptr(a), b=_ptr(b), z=_ptr(z),
        A_log=_ptr(A_log), dt_bias=_ptr(dt_bias), norm_w=_ptr(norm_w),
        cu_seqlens=_ptr(cu), pool=pool.ctypes.data,
        out_f64=out_f64.ctypes.data, out_bf16=out_bf16.ctypes.data,
        states_f64=_ptr(states), states_T=1 if final_states else 0,
    )
    rc = lib.gdn_oracle_prefill(ctypes.byref(p), rd.ctypes.data, wr.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle rejected the problem: {ERRORS.get(rc, rc)}")
    return {"out_f64": out_f64, "out_bf16": out_bf16,
            "states": None if states is None else states[:, :, 0]}


def _unary(name, x, in_dtype, out_dtype):
    lib = load()
    x = np.ascontiguousarray(x, dtype=in_dtype)
    y = np.empty(x.shape, dtype=out_dtype)
    getattr(lib, name)(x.ctypes.data, y.ctypes.data, x.size)
    return y


def round_bf16(x):
    """float64 -> bf16 bits, round to nearest even."""
    return _unary("gdn_oracle_round_bf16", x, np.float64, np.uint16)


def round_f16(x):
    """float64 -> fp16 bits, round to nearest even, gradual underflow."""
    return _unary("gdn_oracle_round_f16", x, np.float64, np.uint16)


def round_f32(x):
    """float64 -> float32, round to nearest even."""
    return _unary("gdn_oracle_round_f32", x, np.float64, np.float32)


def value_bf16(bits):
    return _unary("gdn_oracle_value_bf16", bits, np.uint16, np.float64)


def value_f16(bits):
    return _unary("gdn_oracle_value_f16", bits, np.uint16, np.float64)


def run_case(case, pool, **kw):
    """Convenience: run a ``synth.Case``-shaped object against ``pool``."""
    return spec_decode(
        q=case.q, k=case.k, v=case.v, a=case.a, b=case.b, z=case.z, A_log=case.A_log,
        dt_bias=case.dt_bias, norm_w=case.norm_w, pool=pool, state_dtype=case.state_dtype,
        state_indices=case.state_indices, num_accepted=case.num_accepted,
        cu_seqlens=case.cu_seqlens, spec_token_indx=case.spec_token_indx,
        num_tokens=case.num_tokens, scale=case.scale, eps=case.eps, **kw)


def spec_decode_conv(*, x, conv_weight, conv_bias, conv_pool, conv_in, conv_out, H_k, K, a, b, z, A_log,
                     dt_bias, norm_w, pool, state_dtype, state_indices, num_accepted, cu_seqlens,
                     spec_token_indx=None, scale=128 ** -0.5, eps=1e-5, qk_eps=1e-6,
                     softplus_threshold=20.0, num_threads=1):
    """The short causal convolution with rewind, then the step on its output
    (see ``gdn_oracle_spec_decode_conv``).  ``x`` [num_tokens, conv_dim] are the
    projection rows (bf16 bits, channels q | k | v); ``conv_weight``
    [conv_dim, width], ``conv_bias`` [conv_dim] or None; ``conv_pool``
    [num_conv_slots, state_len, conv_dim] bf16 bits, updated in place, like
    ``pool``.  Returns out_f64 / out_bf16 as ``spec_decode`` does."""
    lib = load()
    x = _c(x, np.uint16); w = _c(conv_weight, np.uint16); cb = _c(conv_bias, np.uint16)
    a = _c(a, np.uint16); b = _c(b, np.uint16); z = _c(z, np.uint16)
    A_log = _c(A_log, np.float32); dt_bias = _c(dt_bias, np.uint16); norm_w = _c(norm_w, np.uint16)
    idx = _c(state_indices, np.int32); acc = _c(num_accepted, np.int32)
    cu = _c(cu_seqlens, np.int32); sti = _c(spec_token_indx, np.int32)
    cin = _c(conv_in, np.int32); cout = _c(conv_out, np.int32)
    if pool.dtype != _POOL_DTYPES[state_dtype] or not pool.flags.c_contiguous:
        raise TypeError("pool must be a contiguous array of the state dtype's storage type")
    if conv_pool.dtype != np.uint16 or not conv_pool.flags.c_contiguous:
        raise TypeError("conv_pool must be a contiguous uint16 (bf16 bits) array")
    N, D = x.shape
    H_v, V = a.shape[1], pool.shape[3]
    batch, stride = idx.shape
    out_f64 = np.full((N, H_v, V), np.nan)
    out_bf16 = np.full((N, H_v, V), 0xFFFF, dtype=np.uint16)
    p = Problem(
        batch=batch, num_tokens=N, H_k=H_k, H_v=H_v, K=K, V=V, spec_stride=stride,
        num_slots=pool.shape[0], state_dtype=state_dtype, num_threads=num_threads,
        scale=scale, eps=eps, qk_eps=qk_eps, softplus_threshold=softplus_threshold,
        a=_ptr(a), b=_ptr(b), z=_ptr(z),
        A_log=_ptr(A_log), dt_bias=_ptr(dt_bias), norm_w=_ptr(norm_w),
        state_indices=_ptr(idx), num_accepted=_ptr(acc), cu_seqlens=_ptr(cu),
        spec_token_indx=_ptr(sti), pool=pool.ctypes.data,
        out_f64=out_f64.ctypes.data, out_bf16=out_bf16.ctypes.data,
    )
    c = Conv(conv_dim=D, width=w.shape[1], state_len=conv_pool.shape[1], num_conv_slots=conv_pool.shape[0],
             x=_ptr(x), weight=_ptr(w), bias=_ptr(cb), conv_pool=conv_pool.ctypes.data,
             conv_in=_ptr(cin), conv_out=_ptr(cout))
    rc = lib.gdn_oracle_spec_decode_conv(ctypes.byref(p), ctypes.byref(c))
    if rc != 0:
        raise OracleError(f"oracle rejected the problem: {ERRORS.get(rc, rc)}")
    return {"out_f64": out_f64, "out_bf16": out_bf16}
