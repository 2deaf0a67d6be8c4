"""Seeded synthetic inputs for the KDA forward pass.

This module is shared by the CUDA-path tests, the benchmark and the oracle
tests.  It holds no arithmetic of the method itself: it only draws random
numbers, L2-normalises q and k (an input property of the workloads, not a
step of the kernel), rounds to bf16 bit patterns and builds cu_seqlens.

Workloads follow the shapes of the FlashKDA benchmarks reported on the
pages ("Moonshot AI Rilis FlashKDA", benchmark paragraph: T=8192, head
dimension 128, H in {96, 64}, fixed length, mixed variable length, and
uniform 1024 x 8 variable length; "Moonshot AI Open-Sources FlashKDA",
section "The performance gap FlashKDA closes").  No dataset is involved.

Value distributions (every workload):
  q, k ~ N(0,1) in fp32, L2-normalised per (token, head), rounded to bf16
  v, g (pre-activation gate), beta logits ~ N(0,1), rounded to bf16
  A_log[H] ~ U(0, ln 16) fp32; dt_bias[H,K] ~ N(0, 0.1) fp32
  lower_bound = -5.0; scale = 1/sqrt(K)
  initial states (where present) ~ N(0, 0.02) (standard deviation 0.02)
Draw order from one numpy PCG64 generator: q, k, v, g, beta, A_log, dt_bias,
initial state, then sequence lengths.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

LOWER_BOUND = -5.0


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    r = ((u.astype(np.uint64) + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[np.isnan(f)] = 0x7FC0
    return r


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int                      # total tokens (packed) per call
    H: int
    B: int = 1
    K: int = 128
    V: int = 128
    lengths: str | None = None  # None = fixed length; "mixed12", "uniform8x1024", "short20000"
    init_dtype: str | None = None   # None, "bf16" or "f32"
    final_dtype: str | None = "f32"
    carry_calls: int = 1        # >1: the sequence is processed in this many calls
    description: str = ""


WORKLOADS = {
    "tiny_t64_h1": Workload(
        "tiny_t64_h1", T=64, H=1,
        description="B=1 T=64 H=1 K=V=128, no initial state, fp32 final state"),
    "prefill_t8192_h64": Workload(
        "prefill_t8192_h64", T=8192, H=64,
        description="fixed-length prefill B=1 T=8192 H=64, no initial state, fp32 final state"),
    "prefill_t8192_h96": Workload(
        "prefill_t8192_h96", T=8192, H=96, init_dtype="bf16",
        description="fixed-length prefill B=1 T=8192 H=96, bf16 initial state, "
                    "fp32 final state"),
    "varlen_mixed_t8192_h96": Workload(
        "varlen_mixed_t8192_h96", T=8192, H=96, lengths="mixed12", init_dtype="f32",
        description="12 sequences of mixed length packed to T=8192, H=96, fp32 states"),
    "varlen_uniform_8x1024_h96": Workload(
        "varlen_uniform_8x1024_h96", T=8192, H=96, lengths="uniform8x1024",
        init_dtype="f32",
        description="8 sequences x 1024 tokens packed, H=96, fp32 states"),
    "carry_t65536_h32": Workload(
        "carry_t65536_h32", T=65536, H=32, carry_calls=2,
        description="B=1 T=65536 H=32 as two 32768-token calls carrying an fp32 state"),
    "varlen_short_20000_h16": Workload(
        "varlen_short_20000_h16", T=160000, H=16, lengths="short20000", final_dtype=None,
        description="20,000 sequences of 0-16 tokens (uniform, summing to 160,000) "
                    "packed, H=16, no states: many short prompts in one call"),
}


def short_lengths(rng: np.random.Generator, n: int = 20000, total: int = 160000,
                  hi: int = 16) -> np.ndarray:
    """n lengths uniform in [0, hi], then moved one token at a time (a random sequence
    that still has room) until they sum to ``total``."""
    lens = rng.integers(0, hi + 1, size=n).astype(np.int64)
    while lens.sum() != total:
        i = int(rng.integers(n))
        if lens.sum() < total and lens[i] < hi:
            lens[i] += 1
        elif lens.sum() > total and lens[i] > 0:
            lens[i] -= 1
    return lens


def mixed_lengths(rng: np.random.Generator, n: int = 12, total: int = 8192,
                  lo: int = 64, hi: int = 2048) -> np.ndarray:
    """n lengths drawn uniform in [lo, hi], rescaled to sum to ``total``.

    Floors the rescaled lengths and gives the remainder to the longest one.
    Returns None-equivalent (empty array) if fewer than 3 lengths are not
    multiples of 16, so that the caller redraws from the next seed.
    """
    raw = rng.integers(lo, hi + 1, size=n)
    lens = np.floor(raw * (total / raw.sum())).astype(np.int64)
    lens = np.maximum(lens, 1)
    lens[np.argmax(lens)] += total - lens.sum()
    assert lens.sum() == total and lens.min() >= 1
    if np.count_nonzero(lens % 16) < 3:
        return np.zeros(0, np.int64)
    return lens


def cu_from_lengths(lengths) -> np.ndarray:
    lens = np.asarray(lengths, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def _normal_bf16(rng, shape):
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _unit_rows_bf16(rng, shape):
    x = rng.standard_normal(shape, dtype=np.float32)
    x /= np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True)).astype(np.float32)
    return f32_to_bf16_bits(x)


def make_inputs(B: int, T: int, H: int, K: int = 128, V: int = 128, seed: int = 0,
                lengths=None, init_dtype: str | None = None,
                lower_bound: float = LOWER_BOUND, scale: float | None = None) -> dict:
    """Draw one set of inputs.

    lengths: None (fixed length, B sequences of T tokens), an explicit list of
    sequence lengths (B must be 1 and the lengths must sum to T), or the
    strings "mixed12" / "uniform8x1024" (drawn / fixed after the tensors).
    Returns a dict of numpy arrays: bf16 tensors as uint16 bit patterns.
    """
    rng = np.random.default_rng(seed)
    out = {
        "q": _unit_rows_bf16(rng, (B, T, H, K)),
        "k": _unit_rows_bf16(rng, (B, T, H, K)),
        "v": _normal_bf16(rng, (B, T, H, V)),
        "g": _normal_bf16(rng, (B, T, H, K)),
        "beta": _normal_bf16(rng, (B, T, H)),
        "A_log": rng.uniform(0.0, math.log(16.0), size=H).astype(np.float32),
        "dt_bias": (0.1 * rng.standard_normal((H, K))).astype(np.float32),
        "lower_bound": float(lower_bound),
        "scale": float(1.0 / math.sqrt(K)) if scale is None else float(scale),
    }
    # number of sequences is fixed by the recipe before any length is drawn
    if lengths is None:
        N = B
    elif isinstance(lengths, str):
        assert B == 1
        N = {"mixed12": 12, "uniform8x1024": 8, "short20000": 20000}[lengths]
    else:
        assert B == 1
        N = len(lengths)
    if init_dtype is not None:
        s0 = (0.02 * rng.standard_normal((N, H, K, V), dtype=np.float32)).astype(np.float32)
        out["initial_state"] = f32_to_bf16_bits(s0) if init_dtype == "bf16" else s0
    else:
        out["initial_state"] = None
    cu = None
    lengths_seed = None
    if lengths == "mixed12":
        s = seed
        lens = mixed_lengths(rng, n=N, total=T)
        while lens.size == 0:   # redraw from the next seed, recorded below
            s += 1
            lens = mixed_lengths(np.random.default_rng(s), n=N, total=T)
        lengths_seed = s
        cu = cu_from_lengths(lens)
    elif lengths == "uniform8x1024":
        assert T % N == 0
        cu = cu_from_lengths(np.full(N, T // N, np.int64))
    elif lengths == "short20000":
        cu = cu_from_lengths(short_lengths(rng, n=N, total=T))
    elif lengths is not None:
        cu = cu_from_lengths(lengths)
        assert int(cu[-1]) == T
    out["cu_seqlens"] = cu
    out["N"] = N
    out["lengths_seed"] = lengths_seed
    return out


def make_inputs_device(T: int, H: int, seed: int = 0, device="cuda:0",
                       lower_bound: float = LOWER_BOUND) -> dict:
    """The recipe of make_inputs (B = 1, fixed length, no initial state) drawn on the
    device with torch's generator, for sizes too large to draw on the host.

    q, k: N(0,1) rows normalised in fp32, rounded to bf16; v, g, beta: N(0,1) in bf16;
    torch tensors [1, T, H, 128] ([1, T, H] for beta).  A_log, dt_bias and the scalars
    come from numpy as in make_inputs.  A token window of the result is handed to a
    host-side consumer with ``window_bits``.
    """
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def normal(shape):
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)

    def unit_rows():
        x = normal((1, T, H, 128))
        x /= torch.linalg.vector_norm(x, dim=-1, keepdim=True)
        return x.to(torch.bfloat16)

    out = {"q": unit_rows(), "k": unit_rows()}
    for name in ("v", "g"):
        out[name] = normal((1, T, H, 128)).to(torch.bfloat16)
    out["beta"] = normal((1, T, H)).to(torch.bfloat16)
    rng = np.random.default_rng(seed)
    out["A_log"] = rng.uniform(0.0, math.log(16.0), size=H).astype(np.float32)
    out["dt_bias"] = (0.1 * rng.standard_normal((H, 128))).astype(np.float32)
    out["lower_bound"] = float(lower_bound)
    out["scale"] = float(1.0 / math.sqrt(128))
    out["N"] = 1
    return out


def window_bits(t, start: int, stop: int) -> np.ndarray:
    """Tokens start .. stop - 1 of a bf16 torch tensor [1, T, ...] as host uint16 bits."""
    import torch
    w = t[:, start:stop].contiguous().cpu().view(torch.int16).numpy()
    return w.view(np.uint16)


def make_workload(name: str, seed: int = 0) -> dict:
    w = WORKLOADS[name]
    d = make_inputs(w.B, w.T, w.H, w.K, w.V, seed=seed, lengths=w.lengths,
                    init_dtype=w.init_dtype)
    d["workload"] = w
    return d
