"""Kimi Delta Attention (KDA) forward pass for GB300 (sm_103a).

Thin ctypes binding over the C ABI in ``include/kda.h`` (library
``_lib/libkda.so``, built by ``gated_delta_rule_39_gb300._build``).  The
functions here only check and marshal arguments: every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if
the library is missing, every call raises.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["KdaError", "kda_fwd", "kda_fwd_segments", "kda_fwd_host", "kda_fwd_noalloc",
           "kda_decode", "kda_bwd", "kda_bwd_workspace_bytes",
           "kda_fwd_get_error", "kda_status_string",
           "kda_last_cuda_error",
           "kda_fwd_workspace_bytes", "kda_profile_enable", "kda_profile_read",
           "kda_kernel_name", "lib_path", "load_library", "KDA_BF16", "KDA_F32",
           "KERNEL_NAMES"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libkda.so")

KDA_BF16 = 0
KDA_F32 = 1
KDA_NUM_KERNELS = 9
KERNEL_NAMES = ("seqmap_kernel", "fused_kernel", "decode_kernel", "combine_kernel",
                "segprep_kernel", "segfinal_kernel", "bwd_kernel", "bwd_finish_kernel",
                "bwd_reduce_kernel")

_lib = None
_vp = ctypes.c_void_p


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str = "kda_fwd"):
        self.status = status
        self.cuda_error = 0
        msg = f"{where} failed: {kda_status_string(status)} ({status})"
        if status in (-6, -10, -11):   # KDA_ERR_LAUNCH, KDA_ERR_ALLOC, KDA_ERR_CUDA
            self.cuda_error = kda_last_cuda_error()
            msg += f"; cudaError_t {self.cuda_error}"
        super().__init__(msg)


def lib_path() -> str:
    return _LIB_PATH


def load_library():
    """Load ``libkda.so``; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"CUDA library {_LIB_PATH} is missing; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    _lib = declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def declare(lib):
    """Set the argument and result types of the C ABI's functions on a loaded library
    (this package's build, or a variant of it built with other flags)."""
    fwd_args = [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, ctypes.c_float, _vp,
                ctypes.c_int, _vp, ctypes.c_int, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp]
    lib.kda_fwd.argtypes = fwd_args
    lib.kda_fwd.restype = ctypes.c_int
    lib.kda_fwd_host.argtypes = fwd_args
    lib.kda_fwd_host.restype = ctypes.c_int
    lib.kda_fwd_noalloc.argtypes = fwd_args
    lib.kda_fwd_noalloc.restype = ctypes.c_int
    lib.kda_fwd_segments.argtypes = fwd_args[:-1] + [ctypes.c_int, _vp]
    lib.kda_fwd_segments.restype = ctypes.c_int
    lib.kda_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp,
                               ctypes.c_float, _vp, ctypes.c_int, _vp, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp]
    lib.kda_decode.restype = ctypes.c_int
    lib.kda_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, ctypes.c_float,
                            _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                            _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                            ctypes.c_int, ctypes.c_int, _vp]
    lib.kda_bwd.restype = ctypes.c_int
    lib.kda_bwd_workspace_bytes.argtypes = [ctypes.c_int] * 5
    lib.kda_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.kda_fwd_get_error.argtypes = [_vp]
    lib.kda_fwd_get_error.restype = ctypes.c_int
    lib.kda_last_cuda_error.argtypes = []
    lib.kda_last_cuda_error.restype = ctypes.c_int
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_fwd_workspace_bytes.argtypes = [ctypes.c_int] * 5
    lib.kda_fwd_workspace_bytes.restype = ctypes.c_size_t
    lib.kda_profile_enable.argtypes = [ctypes.c_int]
    lib.kda_profile_enable.restype = ctypes.c_int
    lib.kda_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(ctypes.c_longlong)]
    lib.kda_profile_read.restype = ctypes.c_int
    lib.kda_kernel_name.argtypes = [ctypes.c_int]
    lib.kda_kernel_name.restype = ctypes.c_char_p
    return lib


def kda_status_string(status: int) -> str:
    return load_library().kda_status_string(int(status)).decode()


def kda_last_cuda_error() -> int:
    """cudaError_t value behind the calling thread's last LAUNCH / ALLOC / CUDA status."""
    return int(load_library().kda_last_cuda_error())


def kda_kernel_name(kernel_id: int) -> str:
    return load_library().kda_kernel_name(int(kernel_id)).decode()


def kda_fwd_workspace_bytes(B: int, T: int, H: int, num_seqs: int = 0,
                            varlen: bool = False) -> int:
    return int(load_library().kda_fwd_workspace_bytes(B, T, H, num_seqs, int(varlen)))


def _state_dtype(t):
    import torch
    if t is None:
        return 0
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"state dtype must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def _marshal(q, k, v, g, beta, out, A_log, dt_bias, initial_state, final_state, cu_seqlens,
             device):
    import torch
    B, T, H, K = q.shape
    V = v.shape[-1]
    for name, t in (("q", q), ("k", k), ("g", g)):
        _check(t, name, torch.bfloat16, (B, T, H, K), device)
    _check(v, "v", torch.bfloat16, (B, T, H, V), device)
    _check(out, "out", torch.bfloat16, (B, T, H, V), device)
    _check(beta, "beta", torch.bfloat16, (B, T, H), device)
    _check(A_log, "A_log", torch.float32, (H,), device)
    _check(dt_bias, "dt_bias", torch.float32, (H, K), device)
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
            raise ValueError("cu_seqlens must be a contiguous 1-D int32 tensor")
        if device is not None and cu_seqlens.device != device:
            raise ValueError(f"cu_seqlens must be on {device}")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    for name, t in (("initial_state", initial_state), ("final_state", final_state)):
        if t is not None:
            if t.dtype not in (torch.bfloat16, torch.float32):
                raise TypeError(f"{name} must be bfloat16 or float32")
            _check(t, name, t.dtype, (N, H, K, V), device)
    return B, T, H, K, V, N


def kda_fwd(q, k, v, g, beta, scale: float, out, A_log, dt_bias, lower_bound: float,
            initial_state=None, final_state=None, cu_seqlens=None, stream=None) -> None:
    """KDA forward on CUDA tensors (asynchronous on ``stream``; default: current stream).

    q, k, g: bf16 [B, T, H, 128]; v, out: bf16 [B, T, H, 128]; beta: bf16 [B, T, H] (logits);
    A_log: fp32 [H]; dt_bias: fp32 [H, 128]; initial_state / final_state: optional
    bf16 or fp32 [N, H, 128, 128]; cu_seqlens: optional int32 [N + 1] (then B == 1).
    Long fixed-length calls with few (sequence, head) recurrences are split into
    segments automatically (``kda_fwd_segments`` with ``num_segments=0``).
    Raises KdaError on a rejected call.
    """
    _fwd_call("kda_fwd", None, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
              initial_state, final_state, cu_seqlens, stream)


def kda_fwd_segments(q, k, v, g, beta, scale: float, out, A_log, dt_bias, lower_bound: float,
                     initial_state=None, final_state=None, cu_seqlens=None, stream=None,
                     num_segments: int = 0) -> None:
    """``kda_fwd`` with the sequence split chosen by the caller: ``num_segments`` 0 picks
    it (as kda_fwd), 1 runs one pass, s >= 2 cuts every sequence of a fixed-length call
    into s segments that run side by side (two windows and a combine step)."""
    _fwd_call("kda_fwd_segments", int(num_segments), q, k, v, g, beta, scale, out, A_log,
              dt_bias, lower_bound, initial_state, final_state, cu_seqlens, stream)


def _fwd_call(name, segments, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
              initial_state, final_state, cu_seqlens, stream):
    import torch
    dev = q.device
    if dev.type != "cuda":
        raise ValueError(f"{name} takes CUDA tensors; use kda_fwd_host for host buffers")
    B, T, H, K, V, N = _marshal(q, k, v, g, beta, out, A_log, dt_bias, initial_state,
                                final_state, cu_seqlens, dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    s = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
            _ptr(A_log), _ptr(dt_bias), float(lower_bound), _ptr(initial_state),
            _state_dtype(initial_state), _ptr(final_state), _state_dtype(final_state),
            _ptr(cu_seqlens), N if cu_seqlens is not None else 0, B, T, H, K, V]
    if segments is not None:
        args.append(segments)
    with torch.cuda.device(dev):
        rc = getattr(load_library(), name)(*args, s)
    if rc != 0:
        raise KdaError(rc, name)


def kda_decode(q, k, v, g, beta, scale: float, out, A_log, dt_bias, lower_bound: float,
               state_in=None, state_out=None, stream=None) -> None:
    """One decode step on CUDA tensors (asynchronous on ``stream``): a single token per
    sequence applied to the states.

    q, k, g: bf16 [N, H, 128]; v, out: bf16 [N, H, 128]; beta: bf16 [N, H] (logits);
    A_log: fp32 [H]; dt_bias: fp32 [H, 128]; state_in / state_out: optional bf16 or
    fp32 [N, H, 128, 128] (the same tensor updates the states in place).
    Raises KdaError on a rejected call.
    """
    import torch
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda_decode takes CUDA tensors")
    N, H, K = q.shape
    V = v.shape[-1]
    for name, t in (("q", q), ("k", k), ("g", g)):
        _check(t, name, torch.bfloat16, (N, H, K), dev)
    _check(v, "v", torch.bfloat16, (N, H, V), dev)
    _check(out, "out", torch.bfloat16, (N, H, V), dev)
    _check(beta, "beta", torch.bfloat16, (N, H), dev)
    _check(A_log, "A_log", torch.float32, (H,), dev)
    _check(dt_bias, "dt_bias", torch.float32, (H, K), dev)
    for name, t in (("state_in", state_in), ("state_out", state_out)):
        if t is not None:
            if t.dtype not in (torch.bfloat16, torch.float32):
                raise TypeError(f"{name} must be bfloat16 or float32")
            _check(t, name, t.dtype, (N, H, K, V), dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    s = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    with torch.cuda.device(dev):
        rc = load_library().kda_decode(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
            _ptr(A_log), _ptr(dt_bias), float(lower_bound), _ptr(state_in),
            _state_dtype(state_in), _ptr(state_out), _state_dtype(state_out), N, H, K, V, s)
    if rc != 0:
        raise KdaError(rc, "kda_decode")


def kda_fwd_noalloc(q, k, v, g, beta, scale: float, out, A_log, dt_bias, lower_bound: float,
                    initial_state=None, final_state=None, cu_seqlens=None, stream=None) -> None:
    """kda_fwd without any device allocation, for callers that cannot allocate.

    Same arguments and results as ``kda_fwd``.  Varlen calls keep their
    scratch in a fixed array inside the library (at most KDA_NOALLOC_MAX_SEQS =
    65536 sequences); calls that overlap on the GPU share that array and race.
    """
    import torch
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda_fwd_noalloc takes CUDA tensors")
    B, T, H, K, V, N = _marshal(q, k, v, g, beta, out, A_log, dt_bias, initial_state,
                                final_state, cu_seqlens, dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    s = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    with torch.cuda.device(dev):
        rc = load_library().kda_fwd_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
            _ptr(A_log), _ptr(dt_bias), float(lower_bound), _ptr(initial_state),
            _state_dtype(initial_state), _ptr(final_state), _state_dtype(final_state),
            _ptr(cu_seqlens), N if cu_seqlens is not None else 0, B, T, H, K, V, s)
    if rc != 0:
        raise KdaError(rc, "kda_fwd_noalloc")


def kda_fwd_host(q, k, v, g, beta, scale: float, out, A_log, dt_bias, lower_bound: float,
                 initial_state=None, final_state=None, cu_seqlens=None, stream=None,
                 device=None) -> None:
    """The same operation on HOST (CPU, ideally pinned) torch tensors; synchronous.

    The library copies inputs to the GPU, runs, and copies ``out`` and
    ``final_state`` back before returning.
    """
    import torch
    for t in (q, k, v, g, beta, out, A_log, dt_bias, initial_state, final_state, cu_seqlens):
        if t is not None and t.device.type != "cpu":
            raise ValueError("kda_fwd_host takes host (CPU) tensors")
    B, T, H, K, V, N = _marshal(q, k, v, g, beta, out, A_log, dt_bias, initial_state,
                                final_state, cu_seqlens, None)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    s = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    with torch.cuda.device(dev):
        rc = load_library().kda_fwd_host(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
            _ptr(A_log), _ptr(dt_bias), float(lower_bound), _ptr(initial_state),
            _state_dtype(initial_state), _ptr(final_state), _state_dtype(final_state),
            _ptr(cu_seqlens), N if cu_seqlens is not None else 0, B, T, H, K, V, s)
    if rc != 0:
        raise KdaError(rc, "kda_fwd_host")


def kda_bwd(q, k, v, g, beta, scale: float, A_log, dt_bias, lower_bound: float, d_out,
            initial_state=None, d_final_state=None, cu_seqlens=None, stream=None,
            d_initial_state: bool = True) -> dict:
    """Gradients of a loss with respect to the forward pass's inputs, on CUDA tensors
    (asynchronous on ``stream``).  d_out: bf16 [B, T, H, 128] = dL/d(out);
    d_final_state: optional fp32 [N, H, 128, 128] = dL/d(final state).  Other arguments
    as ``kda_fwd``.  Returns fp32 tensors: dq, dk, dg [B, T, H, 128], dv [B, T, H, 128],
    dbeta [B, T, H], dA_log [H], ddt_bias [H, 128] and (unless d_initial_state is
    False) d_initial_state [N, H, 128, 128]."""
    import torch
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda_bwd takes CUDA tensors")
    B, T, H, K, V, N = _marshal(q, k, v, g, beta, d_out, A_log, dt_bias, initial_state, None,
                                cu_seqlens, dev)
    if d_final_state is not None:
        _check(d_final_state, "d_final_state", torch.float32, (N, H, K, V), dev)
    f32 = dict(dtype=torch.float32, device=dev)
    r = {"dq": torch.empty((B, T, H, K), **f32), "dk": torch.empty((B, T, H, K), **f32),
         "dv": torch.empty((B, T, H, V), **f32), "dg": torch.empty((B, T, H, K), **f32),
         "dbeta": torch.empty((B, T, H), **f32), "dA_log": torch.empty((H,), **f32),
         "ddt_bias": torch.empty((H, K), **f32)}
    if d_initial_state:
        r["d_initial_state"] = torch.empty((N, H, K, V), **f32)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    s = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    with torch.cuda.device(dev):
        rc = load_library().kda_bwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(A_log),
            _ptr(dt_bias), float(lower_bound), _ptr(initial_state), _state_dtype(initial_state),
            _ptr(d_out), _ptr(d_final_state), _ptr(r["dq"]), _ptr(r["dk"]), _ptr(r["dv"]),
            _ptr(r["dg"]), _ptr(r["dbeta"]), _ptr(r["dA_log"]), _ptr(r["ddt_bias"]),
            _ptr(r.get("d_initial_state")), _ptr(cu_seqlens),
            N if cu_seqlens is not None else 0, B, T, H, K, V, s)
    if rc != 0:
        raise KdaError(rc, "kda_bwd")
    return r


def kda_bwd_workspace_bytes(B: int, T: int, H: int, num_seqs: int = 0,
                            varlen: bool = False) -> int:
    return int(load_library().kda_bwd_workspace_bytes(B, T, H, num_seqs, int(varlen)))


def kda_fwd_get_error(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device error word."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    s = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    return int(load_library().kda_fwd_get_error(s))


def kda_profile_enable(on: bool = True) -> None:
    load_library().kda_profile_enable(int(bool(on)))


def kda_profile_read() -> dict:
    """{kernel name: (summed milliseconds, launches)} since the last enable."""
    ms = (ctypes.c_double * KDA_NUM_KERNELS)()
    n = (ctypes.c_longlong * KDA_NUM_KERNELS)()
    rc = load_library().kda_profile_read(ms, n)
    if rc != 0:
        raise KdaError(rc, "kda_profile_read")
    return {KERNEL_NAMES[i]: (float(ms[i]), int(n[i])) for i in range(KDA_NUM_KERNELS)}
