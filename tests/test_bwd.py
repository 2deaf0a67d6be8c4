"""kda_bwd (the backward pass) against the fp64 backward oracle, which is pinned by finite
differences and autograd (``tests/test_oracle_bwd.py``).

Tolerance: the CUDA pass runs the token recurrence and its reverse in fp32 from the
same bf16 inputs as the oracle (which widens them exactly), so the differences are
fp32 rounding, accumulated over the tokens: every gradient tensor must satisfy
max|gpu - ref| <= 1e-3 * RMS(ref) + 1e-6 element-wise; dA_log and ddt_bias, sums over
all tokens, in the Frobenius norm (<= 1e-3 * ||ref||).  A dropped or wrong term
gives errors of the order of the gradient itself.
"""
import ctypes

import numpy as np
import pytest

import synth
from gpu_harness import upload

GRADS = ("dq", "dk", "dv", "dg", "dbeta")


def _bf16(torch, x, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)


def _run(d, dout_bits, dfinal, heads=None):
    import torch
    import oracle
    import gated_delta_rule_39_gb300 as kda
    x = upload(d)
    do = _bf16(torch, dout_bits)
    dF = None if dfinal is None else torch.from_numpy(dfinal.astype(np.float32)).cuda()
    g = kda.kda_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], d["scale"], x["A_log"],
                    x["dt_bias"], d["lower_bound"], do, initial_state=x["initial_state"],
                    d_final_state=dF, cu_seqlens=x["cu_seqlens"])
    torch.cuda.synchronize()
    assert kda.kda_fwd_get_error() == 0
    ref = oracle.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["A_log"],
                         d["dt_bias"], d["lower_bound"], dout_bits,
                         initial_state=d["initial_state"],
                         dfinal=None if dfinal is None else dfinal.astype(np.float32),
                         cu_seqlens=d["cu_seqlens"], heads=heads)
    return {n: t.cpu().numpy().astype(np.float64) for n, t in g.items()}, ref


def _compare(gpu, ref, heads=None):
    sel = (lambda a, ax: a if heads is None else np.take(a, heads, axis=ax))
    for n in GRADS:
        a, r = sel(gpu[n], 2), sel(ref[n], 2)
        rms = np.sqrt(np.mean(r ** 2)) if r.size else 0.0
        err = np.max(np.abs(a - r)) if r.size else 0.0
        assert err <= 1e-3 * rms + 1e-6, (n, err, rms)
    a, r = sel(gpu["d_initial_state"], 1), sel(ref["d_initial_state"], 1)
    assert np.linalg.norm(a - r) <= 1e-3 * np.linalg.norm(r) + 1e-6, "d_initial_state"
    for n, ax in (("dA_log", 0), ("ddt_bias", 0)):
        a, r = sel(gpu[n], ax), sel(ref[n], ax)
        assert np.linalg.norm(a - r) <= 1e-3 * np.linalg.norm(r) + 1e-6, (n, a, r)


def _dout(shape, seed):
    return synth.f32_to_bf16_bits(np.random.default_rng(seed).standard_normal(shape, dtype=np.float32))


@pytest.mark.gpu
@pytest.mark.parametrize("init", ["f32", "bf16", None])
@pytest.mark.parametrize("with_dfinal", [True, False])
def test_bwd_fixed_length(init, with_dfinal):
    d = synth.make_inputs(2, 50, 2, seed=81, init_dtype=init)
    N, H = 2, 2
    dfinal = (np.random.default_rng(3).standard_normal((N, H, 128, 128)) if with_dfinal else None)
    gpu, ref = _run(d, _dout(d["v"].shape, 4), dfinal)
    _compare(gpu, ref)


@pytest.mark.gpu
def test_bwd_varlen_ragged_and_empty():
    lens = [17, 0, 33, 5, 16, 1]
    d = synth.make_inputs(1, sum(lens), 3, seed=82, lengths=lens, init_dtype="f32")
    dfinal = np.random.default_rng(5).standard_normal((len(lens), 3, 128, 128))
    gpu, ref = _run(d, _dout(d["v"].shape, 6), dfinal)
    _compare(gpu, ref)


@pytest.mark.gpu
@pytest.mark.parametrize("lower_bound", [0.0, -5.4])
def test_bwd_decay_range(lower_bound):
    """No decay (the state gradient carries the whole sequence) and gates at the bound."""
    d = synth.make_inputs(1, 300, 2, seed=83, init_dtype="f32", lower_bound=lower_bound)
    gpu, ref = _run(d, _dout(d["v"].shape, 7), None)
    _compare(gpu, ref)


@pytest.mark.gpu
def test_bwd_full_size_every_head():
    """prefill_t8192_h96 against the oracle on every one of the 96 heads (the fp64
    backward oracle takes about 8 s for them on 16 host cores)."""
    d = synth.make_workload("prefill_t8192_h96")
    dfinal = np.random.default_rng(8).standard_normal((1, 96, 128, 128))
    gpu, ref = _run(d, _dout(d["v"].shape, 9), dfinal)
    _compare(gpu, ref)


def test_bwd_argument_errors():
    """Checked on the host before anything runs: an output overlapping an input, a NULL
    output, a misaligned dv."""
    import gated_delta_rule_39_gb300 as kda
    from gated_delta_rule_39_gb300 import _build
    _build.build()
    lib = kda.load_library()
    vp = ctypes.c_void_p
    base = 0x10000000
    T, H = 64, 2
    row = T * H * 128

    def call(dq=base + 8 * row * 4, dv=base + 10 * row * 4, dA=base + 20 * row * 4):
        return lib.kda_bwd(vp(base), vp(base + row * 2), vp(base + 2 * row * 2), vp(base + 3 * row * 2),
                           vp(base + 4 * row * 2), 0.1, vp(base + 6 * row * 2), vp(base + 7 * row * 2),
                           -5.0, None, 0, vp(base + 5 * row * 2), None, vp(dq),
                           vp(base + 9 * row * 4), vp(dv), vp(base + 11 * row * 4),
                           vp(base + 12 * row * 4), None if dA is None else vp(dA),
                           vp(base + 21 * row * 4), None, None, 0, 1, T, H, 128, 128, None)

    assert call(dq=base) == -13                  # dq over q: KDA_ERR_ALIAS
    assert call(dA=None) == -1                   # KDA_ERR_NULL
    assert call(dv=base + 10 * row * 4 + 4) == -4   # KDA_ERR_ALIGN
    assert kda.kda_bwd_workspace_bytes(1, T, H) > 13 * 1024 * T * H


@pytest.mark.gpu
def test_bwd_many_short_sequences():
    """600 sequences of 0-24 tokens (empty ones, single partial blocks, one block and a
    bit) in one varlen call, two heads, with an initial state and dL/d(final state)."""
    rng = np.random.default_rng(84)
    lens = [int(x) for x in rng.integers(0, 25, size=600)]
    d = synth.make_inputs(1, sum(lens), 2, seed=84, lengths=lens, init_dtype="bf16")
    dfinal = np.random.default_rng(85).standard_normal((len(lens), 2, 128, 128))
    gpu, ref = _run(d, _dout(d["v"].shape, 86), dfinal)
    _compare(gpu, ref)


@pytest.mark.gpu
def test_bwd_long_sequence():
    """One 65,536-token sequence, one head (8,192 checkpoint blocks): the reverse pass
    carries the state gradient over the whole sequence."""
    d = synth.make_inputs(1, 65536, 1, seed=87, init_dtype="f32")
    dfinal = np.random.default_rng(88).standard_normal((1, 1, 128, 128))
    gpu, ref = _run(d, _dout(d["v"].shape, 89), dfinal)
    _compare(gpu, ref)
