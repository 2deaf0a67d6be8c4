"""fp64 CPU oracle for the Kimi Delta Attention (KDA) forward pass.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports this package; only the test suite, the smoke check
and the benchmark's CPU-baseline leg do.  It shares no code with the CUDA
path: the arithmetic lives in ``kda_oracle.c`` (plain C, double precision,
no fast-math, no FMA contraction), and this module only converts inputs to
float64 arrays and calls it through ctypes.

Parity status of each function (what pins it, see ``tests/test_oracle_pins.py``):
  * ``kda_recurrence`` -- pinned: brute-force equality with an independent
    chunked (WY) evaluation and with explicit K x K transition matrices,
    one-token closed forms, delta-rule retrieval, pure decay (beta = 0),
    causal linear attention for orthogonal keys, state carry, varlen
    independence, linearity.
  * ``kda_gate`` -- pinned by value at the sigmoid midpoint, its limits, its
    point symmetry and its monotonicity.
  * ``kda_fwd`` -- ``kda_gate`` + sigmoid(beta) + ``kda_recurrence``; pinned by
    equality with those pieces called separately.
  * ``kda_bwd`` (``kda_oracle_bwd.c``, a library of its own) -- the reverse
    pass of ``kda_fwd``; pinned by central finite differences of ``kda_fwd``
    along random directions of every input, element-wise differences on small
    sizes, and equality with PyTorch autograd through an independently written
    fp64 token recurrence (``tests/test_oracle_bwd.py``).
  * equality of the oracle's numbers with FlashKDA's own kernel outputs:
    parity unpinned (the pages print no output values).

Sources: "Moonshot AI Rilis FlashKDA" (captivela.com) -- the forward pass's
inputs, sigmoid on beta, optional states, cu_seqlens; "Moonshot AI
Open-Sources FlashKDA" (alphasignal.ai), "Why KDA?" -- channel-wise gating.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libkda_oracle.so")
_BWD_SRC = os.path.join(_HERE, "kda_oracle_bwd.c")
_BWD_LIB_PATH = os.path.join(_HERE, "_build", "libkda_oracle_bwd.so")
_lib = None
_bwd_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (plain C, -O2, no FMA contraction)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _f64(x):
    """float64 contiguous copy; uint16 arrays are read as bf16 bit patterns."""
    if x is None:
        return None
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a, t=_dp):
    return None if a is None else a.ctypes.data_as(t)


def _seq_start(rows: int, cu_seqlens, B: int | None):
    if cu_seqlens is not None:
        s = np.ascontiguousarray(cu_seqlens, dtype=np.int64).astype(np.int_)
        return s, len(s) - 1
    assert B is not None and B > 0 and rows % B == 0
    T = rows // B
    return (np.arange(B + 1, dtype=np.int_) * T), B


def _heads(heads, H):
    if heads is None:
        return None, H
    h = np.ascontiguousarray(heads, dtype=np.intc)
    assert h.ndim == 1 and np.all((h >= 0) & (h < H))
    return h, len(h)


class Oracle:
    """ctypes view of one compiled copy of ``kda_oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.kda_oracle_fwd.restype = ctypes.c_int
        lib.kda_oracle_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_double, _dp, _dp,
                                       ctypes.c_double, _dp, _dp, _dp, _lp, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, _ip,
                                       ctypes.c_int, ctypes.c_int]
        lib.kda_oracle_recurrence.restype = ctypes.c_int
        lib.kda_oracle_recurrence.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_double,
                                              _dp, _dp, _dp, _lp, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, _ip,
                                              ctypes.c_int, ctypes.c_int]
        lib.kda_oracle_gate.restype = None
        lib.kda_oracle_gate.argtypes = [_dp, _dp, _dp, ctypes.c_double, _dp, ctypes.c_long,
                                        ctypes.c_int, ctypes.c_int]
        self.lib = lib
        self.path = lib_path

    def kda_gate(self, g, A_log, dt_bias, lower_bound: float) -> np.ndarray:
        """Per-channel natural-log decay lower_bound*sigmoid(exp(A_log)*(g+dt_bias)).

        g: [..., H, K]; A_log: [H]; dt_bias: [H, K].  Returns float64 shaped like g.
        """
        g64 = _f64(g)
        A = _f64(A_log)
        dtb = _f64(dt_bias)
        H, K = dtb.shape
        assert g64.shape[-2:] == (H, K) and A.shape == (H,)
        out = np.empty_like(g64)
        rows = g64.size // (H * K)
        self.lib.kda_oracle_gate(_ptr(g64), _ptr(A), _ptr(dtb), float(lower_bound),
                                 _ptr(out), rows, H, K)
        return out

    def kda_fwd(self, q, k, v, g, beta, scale: float, A_log, dt_bias, lower_bound: float,
                initial_state=None, cu_seqlens=None, heads=None, n_threads=None):
        """Full KDA forward in fp64.

        q, k, g: [B, T, H, K]; v: [B, T, H, V]; beta: [B, T, H] (logits).
        uint16 arrays are bf16 bit patterns; anything else is read as real numbers.
        cu_seqlens: optional [N+1] token offsets (then B must be 1).
        initial_state: optional [N, H, K, V].  heads: optional subset of head indices.
        Returns (out [B, T, H, V], final_state [N, H, K, V]), both float64; entries
        of heads outside ``heads`` are NaN.
        """
        q64, k64, v64, g64, b64 = (_f64(x) for x in (q, k, v, g, beta))
        B, T, H, K = q64.shape
        V = v64.shape[-1]
        assert k64.shape == q64.shape and g64.shape == q64.shape
        assert v64.shape == (B, T, H, V) and b64.shape == (B, T, H)
        if cu_seqlens is not None:
            assert B == 1
        ss, N = _seq_start(B * T, cu_seqlens, B)
        hsel, nsel = _heads(heads, H)
        S0 = _f64(initial_state)
        if S0 is not None:
            assert S0.shape == (N, H, K, V)
        out = np.full((B, T, H, V), np.nan)
        Sf = np.full((N, H, K, V), np.nan)
        A = _f64(A_log)
        dtb = _f64(dt_bias)
        rc = self.lib.kda_oracle_fwd(
            _ptr(q64), _ptr(k64), _ptr(v64), _ptr(g64), _ptr(b64), float(scale), _ptr(A),
            _ptr(dtb), float(lower_bound), _ptr(S0), _ptr(Sf), _ptr(out), _ptr(ss, _lp), N,
            H, K, V, _ptr(hsel, _ip), nsel, n_threads or default_threads())
        if rc != 0:
            raise ValueError(f"kda_oracle_fwd rejected its arguments (code {rc})")
        return out, Sf

    def kda_recurrence(self, q, k, v, log_alpha, beta, scale: float, initial_state=None,
                       cu_seqlens=None, heads=None, n_threads=None):
        """Raw recurrence in fp64 with a given natural-log decay and post-activation beta.

        q, k, log_alpha: [B, T, H, K]; v: [B, T, H, V]; beta: [B, T, H] (used as is).
        Returns (out [B, T, H, V], final_state [N, H, K, V]).
        """
        q64, k64, v64, la64, b64 = (_f64(x) for x in (q, k, v, log_alpha, beta))
        B, T, H, K = q64.shape
        V = v64.shape[-1]
        assert k64.shape == q64.shape and la64.shape == q64.shape
        assert v64.shape == (B, T, H, V) and b64.shape == (B, T, H)
        if cu_seqlens is not None:
            assert B == 1
        ss, N = _seq_start(B * T, cu_seqlens, B)
        hsel, nsel = _heads(heads, H)
        S0 = _f64(initial_state)
        if S0 is not None:
            assert S0.shape == (N, H, K, V)
        out = np.full((B, T, H, V), np.nan)
        Sf = np.full((N, H, K, V), np.nan)
        rc = self.lib.kda_oracle_recurrence(
            _ptr(q64), _ptr(k64), _ptr(v64), _ptr(la64), _ptr(b64), float(scale), _ptr(S0),
            _ptr(Sf), _ptr(out), _ptr(ss, _lp), N, H, K, V, _ptr(hsel, _ip), nsel,
            n_threads or default_threads())
        if rc != 0:
            raise ValueError(f"kda_oracle_recurrence rejected its arguments (code {rc})")
        return out, Sf


def build_bwd(force: bool = False) -> str:
    """Compile the backward oracle ``kda_oracle_bwd.c`` (same flags as the forward)."""
    return build(force=force, src=_BWD_SRC, out=_BWD_LIB_PATH)


def kda_bwd(q, k, v, g, beta, scale: float, A_log, dt_bias, lower_bound: float, dout,
            initial_state=None, dfinal=None, cu_seqlens=None, heads=None, n_threads=None):
    """Gradients of a loss L = sum(dout * out) + sum(dfinal * final_state) of ``kda_fwd``
    in fp64.  Shapes as ``kda_fwd``; dout [B, T, H, V]; dfinal optional [N, H, K, V].
    Returns a dict: dq, dk, dg [B, T, H, K]; dv [B, T, H, V]; dbeta [B, T, H];
    dA_log [H]; dt_bias [H, K] (as "ddt_bias"); d_initial_state [N, H, K, V] (the
    gradient with respect to the initial state, also when none was given: zero).
    Entries of heads outside ``heads`` are NaN (dA_log, ddt_bias: 0)."""
    global _bwd_lib
    if _bwd_lib is None:
        lib = ctypes.CDLL(build_bwd())
        lib.kda_oracle_bwd.restype = ctypes.c_int
        lib.kda_oracle_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_double, _dp, _dp,
                                       ctypes.c_double, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                       _dp, _dp, _dp, _dp, _lp, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, _ip, ctypes.c_int,
                                       ctypes.c_int]
        _bwd_lib = lib
    q64, k64, v64, g64, b64, do64 = (_f64(x) for x in (q, k, v, g, beta, dout))
    B, T, H, K = q64.shape
    V = v64.shape[-1]
    assert k64.shape == q64.shape and g64.shape == q64.shape
    assert v64.shape == (B, T, H, V) and b64.shape == (B, T, H) and do64.shape == v64.shape
    if cu_seqlens is not None:
        assert B == 1
    ss, N = _seq_start(B * T, cu_seqlens, B)
    hsel, nsel = _heads(heads, H)
    S0 = _f64(initial_state)
    dST = _f64(dfinal)
    for x in (S0, dST):
        if x is not None:
            assert x.shape == (N, H, K, V)
    r = {"dq": np.full((B, T, H, K), np.nan), "dk": np.full((B, T, H, K), np.nan),
         "dg": np.full((B, T, H, K), np.nan), "dv": np.full((B, T, H, V), np.nan),
         "dbeta": np.full((B, T, H), np.nan), "d_initial_state": np.full((N, H, K, V), np.nan)}
    dA_u = np.zeros((N, H))
    ddt_u = np.zeros((N, H, K))
    A = _f64(A_log)
    dtb = _f64(dt_bias)
    rc = _bwd_lib.kda_oracle_bwd(
        _ptr(q64), _ptr(k64), _ptr(v64), _ptr(g64), _ptr(b64), float(scale), _ptr(A), _ptr(dtb),
        float(lower_bound), _ptr(S0), _ptr(do64), _ptr(dST), _ptr(r["dq"]), _ptr(r["dk"]),
        _ptr(r["dv"]), _ptr(r["dg"]), _ptr(r["dbeta"]), _ptr(dA_u), _ptr(ddt_u),
        _ptr(r["d_initial_state"]), _ptr(ss, _lp), N, H, K, V, _ptr(hsel, _ip), nsel,
        n_threads or default_threads())
    if rc != 0:
        raise ValueError(f"kda_oracle_bwd rejected its arguments (code {rc})")
    r["dA_log"] = dA_u.sum(axis=0)
    r["ddt_bias"] = ddt_u.sum(axis=0)
    return r


def get() -> Oracle:
    """The oracle compiled from this directory's ``kda_oracle.c``."""
    global _lib
    if _lib is None:
        _lib = Oracle(build())
    return _lib


def kda_gate(*a, **kw):
    return get().kda_gate(*a, **kw)


def kda_fwd(*a, **kw):
    return get().kda_fwd(*a, **kw)


def kda_recurrence(*a, **kw):
    return get().kda_recurrence(*a, **kw)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
