"""Python binding of libgdnspec (include/gdnspec.h): argument marshalling only.

PyTorch provides device memory and streams; every step of the computation
runs in the library's CUDA kernel.  There is no fallback: if the library has
not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

F32, BF16, F16 = 0, 1, 2
_STATE_DTYPES = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}

GDN_FLAG_SLOT_RANGE = 1
GDN_FLAG_ACCEPTED = 2
GDN_FLAG_QLEN = 4
GDN_FLAG_TOKEN_ROW = 8
GDN_FLAG_TIMEOUT = 16
GDN_FLAG_DRAIN = 32
GDN_SPLIT_NARROW = 0x100     # dims.split flag: 8 V columns per warp (small batches)
GDN_SPLIT_HALFK = 0x200      # dims.split flag (with 2): half of the K rows per warp (small batches)
GDN_PRE_INDEX = 0x1          # dims.flags: the index tables were not written by the preceding kernel
GDN_PRE_TOKENS = 0x2         # dims.flags (with GDN_PRE_INDEX): nor were the token inputs
GDN_PRE_STATE = 0x4          # dims.flags (with GDN_PRE_INDEX): nor were the state slots this call reads


class gdn_dims(ctypes.Structure):
    """Mirror of gdn_dims in include/gdnspec.h."""

    _fields_ = [
        ("batch", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
        ("H_k", ctypes.c_int32), ("H_v", ctypes.c_int32),
        ("K", ctypes.c_int32), ("V", ctypes.c_int32),
        ("spec_stride", ctypes.c_int32), ("max_T", ctypes.c_int32),
        ("num_slots", ctypes.c_int64),
        ("q_stride", ctypes.c_int64), ("k_stride", ctypes.c_int64), ("v_stride", ctypes.c_int64),
        ("a_stride", ctypes.c_int64), ("b_stride", ctypes.c_int64), ("z_stride", ctypes.c_int64),
        ("out_stride", ctypes.c_int64),
        ("split", ctypes.c_int32), ("flags", ctypes.c_int32),
    ]


class gdn_conv_dims(ctypes.Structure):
    """Mirror of gdn_conv_dims in include/gdnspec.h."""

    _fields_ = [
        ("width", ctypes.c_int32), ("state_len", ctypes.c_int32),
        ("num_conv_slots", ctypes.c_int64), ("x_stride", ctypes.c_int64),
        ("reserved", ctypes.c_int32 * 2),
    ]


class GdnError(RuntimeError):
    def __init__(self, status: int, text: str):
        super().__init__(f"gdn_spec_decode failed: {text} (status {status})")
        self.status = status


class LibraryMissing(RuntimeError):
    pass


_lock = threading.Lock()
_lib = None

# the C functions and their signatures, as declared in include/gdnspec.h
_VP = ctypes.c_void_p
EXPORTS = {
    "gdn_spec_decode": (ctypes.c_int, [_VP] * 15 + [ctypes.POINTER(gdn_dims), ctypes.c_float, ctypes.c_float,
                                                   ctypes.c_int, _VP, _VP]),
    "gdn_prefill": (ctypes.c_int, [_VP] * 14 + [ctypes.POINTER(gdn_dims), ctypes.c_float, ctypes.c_float,
                                               ctypes.c_int, _VP, _VP]),
    "gdn_prefill_chunked": (ctypes.c_int, [_VP] * 14 + [ctypes.POINTER(gdn_dims), ctypes.c_float,
                                                       ctypes.c_float, ctypes.c_int, _VP, _VP]),
    "gdn_spec_decode_conv": (ctypes.c_int, [_VP] * 6 + [ctypes.POINTER(gdn_conv_dims)] + [_VP] * 12 +
                             [ctypes.POINTER(gdn_dims), ctypes.c_float, ctypes.c_float, ctypes.c_int, _VP, _VP]),
    "gdn_spec_decode_split": (ctypes.c_int32, [ctypes.POINTER(gdn_dims), ctypes.c_int]),
    "gdn_set_wait_limit": (None, [ctypes.c_uint32]),
    "gdn_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "gdn_version": (ctypes.c_int32, []),
}


def library_path() -> str:
    return _build.LIB


def load_library() -> ctypes.CDLL:
    """Load the in-tree libgdnspec.so (built by __graft_entry__.build() or
    ``python -m gated_deltanet_linear_sm_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise LibraryMissing(f"{path} is not built; run `python -m gated_deltanet_linear_sm_gb300.build`")
            lib = ctypes.CDLL(path)
            for name, (res, args) in EXPORTS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def status_str(status: int) -> str:
    return load_library().gdn_status_str(status).decode()


def version() -> int:
    return int(load_library().gdn_version())


def set_wait_limit(polls: int) -> None:
    """Bound on each tensor-core wait of gdn_prefill_chunked, in polls (0: the
    default); process-wide, for exercising the timeout path."""
    load_library().gdn_set_wait_limit(int(polls))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _row_stride(t, name, inner):
    """Elements between token rows; the rest of a row must be dense."""
    if t.dim() < 2:
        raise ValueError(f"{name}: expected [tokens, ...]")
    if t.dim() == 3 and (t.stride(2) != 1 or t.stride(1) != t.shape[2]):
        raise ValueError(f"{name}: heads and head dim must be contiguous within a row")
    if t.dim() == 2 and t.stride(1) != 1:
        raise ValueError(f"{name}: the head dim must be contiguous")
    return t.stride(0) if t.shape[0] > 1 else inner


def _check(t, name, dtype, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")


def check_shapes(q, k, v, a, b, z, A_log, dt_bias, norm_w, out=None):
    """Sizes of the token and parameter tensors against each other, checked
    before anything else (device, dtype) so that no call with a short buffer
    reaches the library: q, k [N, H_k, K]; v (and z, out) [N, H_v, V]; a, b
    [N, H_v]; A_log, dt_bias [H_v]; norm_w [V].  Raises ValueError."""
    if q.dim() != 3 or k.shape != q.shape:
        raise ValueError(f"expected q, k [N, H_k, K]; got q {tuple(q.shape)}, k {tuple(k.shape)}")
    N = q.shape[0]
    if v.dim() != 3 or v.shape[0] != N:
        raise ValueError(f"expected v [N={N}, H_v, V]; got {tuple(v.shape)}")
    H_v, V = v.shape[1], v.shape[2]
    for t, n in ((a, "a"), (b, "b")):
        if tuple(t.shape) != (N, H_v):
            raise ValueError(f"expected {n} [N={N}, H_v={H_v}]; got {tuple(t.shape)}")
    for t, n in ((A_log, "A_log"), (dt_bias, "dt_bias")):
        if tuple(t.shape) != (H_v,):
            raise ValueError(f"expected {n} [H_v={H_v}]; got {tuple(t.shape)}")
    if z is not None and tuple(z.shape) != tuple(v.shape):
        raise ValueError(f"expected z {tuple(v.shape)} (the shape of v); got {tuple(z.shape)}")
    if norm_w is not None and tuple(norm_w.shape) != (V,):
        raise ValueError(f"expected norm_w [V={V}]; got {tuple(norm_w.shape)}")
    if out is not None and tuple(out.shape) != tuple(v.shape):
        raise ValueError(f"expected out {tuple(v.shape)} (the shape of v); got {tuple(out.shape)}")


def make_dims(q, v, state_pool, state_indices, *, k=None, a=None, b=None, z=None, out=None,
              max_T=None, split=0, flags=0) -> gdn_dims:
    N, H_k, K = q.shape
    H_v, V = v.shape[1], v.shape[2]
    batch, stride = state_indices.shape
    d = gdn_dims()
    d.batch, d.num_tokens, d.H_k, d.H_v, d.K, d.V = batch, N, H_k, H_v, K, V
    d.spec_stride = stride
    d.max_T = min(stride, 8) if max_T is None else max_T
    d.num_slots = state_pool.shape[0]
    d.q_stride = _row_stride(q, "q", H_k * K)
    d.k_stride = _row_stride(k, "k", H_k * K) if k is not None else 0
    d.v_stride = _row_stride(v, "v", H_v * V)
    d.a_stride = _row_stride(a, "a", H_v) if a is not None else 0
    d.b_stride = _row_stride(b, "b", H_v) if b is not None else 0
    d.z_stride = _row_stride(z, "z", H_v * V) if z is not None else 0
    d.out_stride = _row_stride(out, "out", H_v * V) if out is not None else 0
    d.split = split
    d.flags = flags
    return d


def gdn_spec_decode(q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, state_indices,
                    num_accepted, cu_seqlens, out, *, spec_token_indx=None, scale=128 ** -0.5,
                    eps=1e-5, max_T=None, split=0, flags=0, status=None, stream=None):
    """One speculative decode step (see include/gdnspec.h).  Tensors are CUDA
    tensors on one device: q, k [N, H_k, 128], v, z, out [N, H_v, 128], a, b
    [N, H_v], dt_bias [H_v], norm_w [128] in bf16; A_log [H_v] fp32;
    state_pool [num_slots, H_v, 128, 128] fp32 / bf16 / fp16 (updated in
    place); state_indices [B, spec_stride], num_accepted [B], cu_seqlens
    [B+1], spec_token_indx [sum q_len] (optional) and status [1] (optional)
    int32.  ``flags``: GDN_PRE_INDEX [| GDN_PRE_TOKENS] [| GDN_PRE_STATE] when
    those inputs were not written by the kernel launched just before on the
    stream.  Launches on
    ``stream`` (default: the current stream) and returns ``out``."""
    call = prepare(q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, state_indices,
                   num_accepted, cu_seqlens, out, spec_token_indx=spec_token_indx, scale=scale,
                   eps=eps, max_T=max_T, split=split, flags=flags, status=status)
    call(stream)
    return out


class PreparedCall:
    """A marshalled gdn_spec_decode call; invoking it launches on the given
    stream (default: the current stream), so it can be replayed in a loop or
    captured in a CUDA graph without re-checking the arguments."""

    def __init__(self, args, dims, scale, eps, state_dtype, device, keep, status_ptr=None):
        self._fn = load_library().gdn_spec_decode
        self._args = args
        self._dims = dims
        self._scale = scale
        self._eps = eps
        self._state_dtype = state_dtype
        self._device = device
        self._keep = keep          # the tensors stay alive as long as the call
        self._status_ptr = status_ptr
        # converted once: a call only adds the stream handle
        self._cargs = tuple(ctypes.c_void_p(x) for x in args) + (
            ctypes.byref(dims), ctypes.c_float(scale), ctypes.c_float(eps), ctypes.c_int(state_dtype),
            ctypes.c_void_p(status_ptr))

    @property
    def dims(self) -> gdn_dims:
        return self._dims

    @property
    def state_dtype(self) -> int:
        return self._state_dtype

    def __call__(self, stream=None):
        """Launch on `stream`: a torch.cuda.Stream, a raw cudaStream_t handle
        (int), or None for the current stream."""
        if stream is None:
            stream = torch.cuda.current_stream(self._device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
        rc = self._fn(*self._cargs, handle)
        if rc != 0:
            raise GdnError(rc, status_str(rc))


def prepare(q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, state_indices, num_accepted,
            cu_seqlens, out, *, spec_token_indx=None, scale=128 ** -0.5, eps=1e-5, max_T=None,
            split=0, flags=0, status=None) -> PreparedCall:
    check_shapes(q, k, v, a, b, z, A_log, dt_bias, norm_w, out)
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("gdn_spec_decode runs on CUDA tensors only")
    bf = torch.bfloat16
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (a, "a"), (b, "b"), (dt_bias, "dt_bias"), (out, "out")):
        _check(t, n, bf, dev)
    if (z is None) != (norm_w is None):
        raise ValueError("z and norm_w must both be given or both be None")
    if z is not None:
        _check(z, "z", bf, dev)
        _check(norm_w, "norm_w", bf, dev)
        if not norm_w.is_contiguous():
            raise ValueError("norm_w must be contiguous")
    _check(A_log, "A_log", torch.float32, dev)
    for t, n in ((state_indices, "state_indices"), (num_accepted, "num_accepted"), (cu_seqlens, "cu_seqlens")):
        _check(t, n, torch.int32, dev)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if spec_token_indx is not None:
        _check(spec_token_indx, "spec_token_indx", torch.int32, dev)
        if not spec_token_indx.is_contiguous():
            raise ValueError("spec_token_indx must be contiguous")
    if status is not None:
        _check(status, "status", torch.int32, dev)
    if state_pool.dtype not in _STATE_DTYPES:
        raise TypeError(f"state_pool: dtype {state_pool.dtype} not in fp32 / bf16 / fp16")
    if state_pool.device != dev or not state_pool.is_contiguous():
        raise ValueError("state_pool must be a contiguous tensor on the same device")
    if not (A_log.is_contiguous() and dt_bias.is_contiguous()):
        raise ValueError("A_log and dt_bias must be contiguous")
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or out.shape != v.shape:
        raise ValueError("expected q, k [N, H_k, K] and v, out [N, H_v, V]")
    if state_indices.dim() != 2 or num_accepted.shape[0] != state_indices.shape[0] or \
            cu_seqlens.shape[0] != state_indices.shape[0] + 1:
        raise ValueError("expected state_indices [B, S], num_accepted [B], cu_seqlens [B+1]")
    if state_pool.dim() != 4 or state_pool.shape[1] != v.shape[1] or state_pool.shape[2] != q.shape[2] or \
            state_pool.shape[3] != v.shape[2]:
        raise ValueError("expected state_pool [num_slots, H_v, K, V]")
    dims = make_dims(q, v, state_pool, state_indices, k=k, a=a, b=b, z=z, out=out, max_T=max_T, split=split,
                     flags=flags)
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(z), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w),
            _ptr(state_pool), _ptr(state_indices), _ptr(num_accepted), _ptr(cu_seqlens),
            _ptr(spec_token_indx), _ptr(out)]
    return PreparedCall(args, dims, float(scale), float(eps), _STATE_DTYPES[state_pool.dtype], dev,
                        keep=(q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, state_indices,
                              num_accepted, cu_seqlens, spec_token_indx, out, status),
                        status_ptr=_ptr(status))


def chosen_split(dims: gdn_dims, state_dtype: int = BF16) -> int:
    """The split code gdn_spec_decode uses for these sizes and state dtype
    (F32 / BF16 / F16)."""
    return int(load_library().gdn_spec_decode_split(ctypes.byref(dims), int(state_dtype)))


def gdn_prefill(q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, read_slots, write_slots,
                cu_seqlens, out, *, scale=128 ** -0.5, eps=1e-5, status=None, stream=None):
    """Prefill over whole prompts (see include/gdnspec.h): sequence i is rows
    cu_seqlens[i] .. cu_seqlens[i+1]-1 of q, k, v, a, b, z, starts from slot
    read_slots[i] (zero state when < 0) and stores its final state in slot
    write_slots[i] (none when < 0).  Tensors as for gdn_spec_decode;
    read_slots, write_slots [B] int32.  Returns ``out``."""
    return _prefill("gdn_prefill", q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, read_slots,
                    write_slots, cu_seqlens, out, scale, eps, status, stream)


def gdn_prefill_chunked(q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, read_slots, write_slots,
                        cu_seqlens, out, *, scale=128 ** -0.5, eps=1e-5, status=None, stream=None):
    """The same prefill as gdn_prefill, computed chunk by chunk on the tensor
    cores at FP32 accuracy (hi / lo bf16 operand parts, FP32 accumulation; see
    include/gdnspec.h).  Same arguments; returns ``out``."""
    return _prefill("gdn_prefill_chunked", q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, read_slots,
                    write_slots, cu_seqlens, out, scale, eps, status, stream)


def _prefill(entry, q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, read_slots, write_slots,
             cu_seqlens, out, scale, eps, status, stream):
    check_shapes(q, k, v, a, b, z, A_log, dt_bias, norm_w, out)
    dev = q.device
    if dev.type != "cuda":
        raise ValueError(f"{entry} runs on CUDA tensors only")
    bf = torch.bfloat16
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (a, "a"), (b, "b"), (dt_bias, "dt_bias"), (out, "out")):
        _check(t, n, bf, dev)
    if (z is None) != (norm_w is None):
        raise ValueError("z and norm_w must both be given or both be None")
    if z is not None:
        _check(z, "z", bf, dev)
        _check(norm_w, "norm_w", bf, dev)
    _check(A_log, "A_log", torch.float32, dev)
    for t, n in ((read_slots, "read_slots"), (write_slots, "write_slots"), (cu_seqlens, "cu_seqlens")):
        _check(t, n, torch.int32, dev)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if read_slots.shape != write_slots.shape or read_slots.dim() != 1 or \
            cu_seqlens.shape[0] != read_slots.shape[0] + 1:
        raise ValueError("expected read_slots, write_slots [B] and cu_seqlens [B+1]")
    if status is not None:
        _check(status, "status", torch.int32, dev)
    if state_pool.dtype not in _STATE_DTYPES or state_pool.device != dev or not state_pool.is_contiguous():
        raise ValueError("state_pool must be a contiguous fp32 / bf16 / fp16 tensor on the same device")
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or out.shape != v.shape:
        raise ValueError("expected q, k [N, H_k, K] and v, out [N, H_v, V]")
    # the decode-only size fields are not used by the prefill entry points
    dims = make_dims(q, v, state_pool, read_slots.view(-1, 1), k=k, a=a, b=b, z=z, out=out, max_T=1)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    rc = getattr(load_library(), entry)(
        _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(z), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w),
        _ptr(state_pool), _ptr(read_slots), _ptr(write_slots), _ptr(cu_seqlens), _ptr(out),
        ctypes.byref(dims), float(scale), float(eps), _STATE_DTYPES[state_pool.dtype], _ptr(status), handle)
    if rc != 0:
        raise GdnError(rc, status_str(rc))
    return out


def gdn_spec_decode_conv(x, conv_weight, conv_bias, conv_pool, conv_in, conv_out, a, b, z, A_log, dt_bias,
                         norm_w, state_pool, state_indices, num_accepted, cu_seqlens, out, *, H_k, K=128,
                         spec_token_indx=None, scale=128 ** -0.5, eps=1e-5, max_T=None, flags=0, status=None,
                         stream=None):
    """The speculative step with the short causal convolution fused in front
    (see include/gdnspec.h): x [N, conv_dim] bf16 projection rows (channels
    q | k | v), conv_weight [conv_dim, W] bf16, conv_bias [conv_dim] bf16 or
    None, conv_pool [num_conv_slots, state_len, conv_dim] bf16 (updated in
    place), conv_in / conv_out [B] int32; the other tensors as for
    gdn_spec_decode.  Returns ``out``."""
    if x.dim() != 2 or state_pool.dim() != 4:
        raise ValueError("expected x [N, conv_dim] and state_pool [num_slots, H_v, K, V]")
    N, H_v, V = x.shape[0], state_pool.shape[1], state_pool.shape[3]
    for t, n, shape in ((a, "a", (N, H_v)), (b, "b", (N, H_v)), (A_log, "A_log", (H_v,)),
                        (dt_bias, "dt_bias", (H_v,)), (out, "out", (N, H_v, V))):
        if tuple(t.shape) != shape:
            raise ValueError(f"expected {n} {shape}; got {tuple(t.shape)}")
    if z is not None and tuple(z.shape) != (N, H_v, V):
        raise ValueError(f"expected z {(N, H_v, V)}; got {tuple(z.shape)}")
    if norm_w is not None and tuple(norm_w.shape) != (V,):
        raise ValueError(f"expected norm_w [V={V}]; got {tuple(norm_w.shape)}")
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("gdn_spec_decode_conv runs on CUDA tensors only")
    bf = torch.bfloat16
    for t, n in ((x, "x"), (conv_weight, "conv_weight"), (conv_pool, "conv_pool"), (a, "a"), (b, "b"),
                 (dt_bias, "dt_bias"), (out, "out")):
        _check(t, n, bf, dev)
    if conv_bias is not None:
        _check(conv_bias, "conv_bias", bf, dev)
    if (z is None) != (norm_w is None):
        raise ValueError("z and norm_w must both be given or both be None")
    if z is not None:
        _check(z, "z", bf, dev)
        _check(norm_w, "norm_w", bf, dev)
    _check(A_log, "A_log", torch.float32, dev)
    for t, n in ((state_indices, "state_indices"), (num_accepted, "num_accepted"), (cu_seqlens, "cu_seqlens"),
                 (conv_in, "conv_in"), (conv_out, "conv_out")):
        _check(t, n, torch.int32, dev)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if spec_token_indx is not None:
        _check(spec_token_indx, "spec_token_indx", torch.int32, dev)
    if status is not None:
        _check(status, "status", torch.int32, dev)
    if not (conv_weight.is_contiguous() and conv_pool.is_contiguous() and
            (conv_bias is None or conv_bias.is_contiguous())):
        raise ValueError("conv_weight, conv_bias and conv_pool must be contiguous")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be [N, conv_dim] with contiguous channels")
    if state_pool.dtype not in _STATE_DTYPES or state_pool.device != dev or not state_pool.is_contiguous():
        raise ValueError("state_pool must be a contiguous fp32 / bf16 / fp16 tensor on the same device")
    N, D = x.shape
    H_v, V = state_pool.shape[1], state_pool.shape[3]
    if D != 2 * H_k * K + H_v * V or conv_weight.shape[0] != D or conv_pool.shape[2] != D:
        raise ValueError("conv_dim must be 2 H_k K + H_v V for x, conv_weight and conv_pool")
    d = gdn_dims()
    d.batch, d.num_tokens, d.H_k, d.H_v, d.K, d.V = state_indices.shape[0], N, H_k, H_v, K, V
    d.spec_stride = state_indices.shape[1]
    d.max_T = min(d.spec_stride, 8) if max_T is None else max_T
    d.num_slots = state_pool.shape[0]
    d.a_stride = _row_stride(a, "a", H_v)
    d.b_stride = _row_stride(b, "b", H_v)
    d.z_stride = _row_stride(z, "z", H_v * V) if z is not None else 0
    d.out_stride = _row_stride(out, "out", H_v * V)
    d.flags = flags
    cd = gdn_conv_dims()
    cd.width = conv_weight.shape[1]
    cd.state_len = conv_pool.shape[1]
    cd.num_conv_slots = conv_pool.shape[0]
    cd.x_stride = x.stride(0) if N > 1 else D
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    rc = load_library().gdn_spec_decode_conv(
        _ptr(x), _ptr(conv_weight), _ptr(conv_bias), _ptr(conv_pool), _ptr(conv_in), _ptr(conv_out),
        ctypes.byref(cd), _ptr(a), _ptr(b), _ptr(z), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w), _ptr(state_pool),
        _ptr(state_indices), _ptr(num_accepted), _ptr(cu_seqlens), _ptr(spec_token_indx), _ptr(out),
        ctypes.byref(d), float(scale), float(eps), _STATE_DTYPES[state_pool.dtype], _ptr(status), handle)
    if rc != 0:
        raise GdnError(rc, status_str(rc))
    return out
