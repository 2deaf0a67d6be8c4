"""Build variants of the fused kernel: the bounded waits, exercised without faulting
anything, and the tf32 operand rounding.

A variant of the library is built with a pipeline-wait bound of 64 SM cycles
(-DKDA_SPIN_LIMIT=64), far below the time a TMA copy from HBM takes, so a wait
runs out on the first chunk of every CTA.  The call must then report
KDA_ERR_DEVICE_TIMEOUT through the device error word, having drained its own
copies and tensor-core operations, and the GPU must stay usable: a normal call
right after it matches the fp64 oracle.
"""
import ctypes

import pytest

import synth
from gpu_harness import run_gpu, run_oracle, to_f64, upload
from parity import out_error, state_error

KDA_ERR_DEVICE_TIMEOUT = -7


@pytest.mark.gpu
def test_wait_that_runs_out_reports_timeout_and_the_gpu_stays_usable():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_39_gb300 as kda
    from gated_delta_rule_39_gb300 import _build
    kda.load_library()
    path = _build.build(lib="libkda_spin64.so", extra_flags=["-DKDA_SPIN_LIMIT=64"])
    short = kda.declare(ctypes.CDLL(path))
    d = synth.make_inputs(1, 300, 2, seed=41, init_dtype="f32")
    x = upload(d)
    out = torch.full((1, 300, 2, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    fs = torch.full((1, 2, 128, 128), float("nan"), device="cuda")
    stream = torch.cuda.current_stream()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = short.kda_fwd(p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]),
                       ctypes.c_float(d["scale"]), p(out), p(x["A_log"]), p(x["dt_bias"]),
                       ctypes.c_float(d["lower_bound"]), p(x["initial_state"]), 1, p(fs), 1,
                       None, 0, 1, 300, 2, 128, 128, ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0
    assert short.kda_fwd_get_error(ctypes.c_void_p(stream.cuda_stream)) == KDA_ERR_DEVICE_TIMEOUT
    # the word is cleared by the read, and the device answers normally afterwards
    assert short.kda_fwd_get_error(ctypes.c_void_p(stream.cuda_stream)) == 0
    o, s = run_gpu(d)
    assert kda.kda_fwd_get_error() == 0
    ro, rs = run_oracle(d)
    assert out_error(to_f64(o), ro)["ok"]
    assert state_error(to_f64(s), rs)["ok"]


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["fixed_no_state", "short_persistent"])
def test_wait_that_runs_out_without_initial_state(case):
    """The same give-up path on the kernel without an initial state, with one CTA per
    unit and on persistent CTAs (400 short sequences: units taken from the counter,
    the next unit's hand-offs made before the output stores)."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import numpy as np
    import gated_delta_rule_39_gb300 as kda
    from gated_delta_rule_39_gb300 import _build
    kda.load_library()
    path = _build.build(lib="libkda_spin64.so", extra_flags=["-DKDA_SPIN_LIMIT=64"])
    short = kda.declare(ctypes.CDLL(path))
    if case == "fixed_no_state":
        d = synth.make_inputs(1, 300, 2, seed=43)
    else:
        lens = [int(x) for x in np.random.default_rng(44).integers(0, 21, size=400)]
        d = synth.make_inputs(1, sum(lens), 1, seed=44, lengths=lens)
    x = upload(d)
    B, T, H, _ = d["q"].shape
    out = torch.full((B, T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = short.kda_fwd(p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]),
                       ctypes.c_float(d["scale"]), p(out), p(x["A_log"]), p(x["dt_bias"]),
                       ctypes.c_float(d["lower_bound"]), None, 0, None, 1,
                       p(x["cu_seqlens"]), d["N"] if x["cu_seqlens"] is not None else 0,
                       B, T, H, 128, 128, ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0
    assert short.kda_fwd_get_error(ctypes.c_void_p(stream.cuda_stream)) == KDA_ERR_DEVICE_TIMEOUT
    assert short.kda_fwd_get_error(ctypes.c_void_p(stream.cuda_stream)) == 0
    o, _ = run_gpu(d)
    assert kda.kda_fwd_get_error() == 0
    ro, _ = run_oracle(d)
    assert out_error(to_f64(o), ro)["ok"]


@pytest.mark.gpu
def test_tf32_rounding_by_addition_equals_the_conversion():
    """The kernel rounds tf32 operands by adding half an ulp to the fp32 bits and lets
    the tensor core drop the low 13 bits.  A build that rounds with cvt.rna.tf32.f32
    instead (-DKDA_TF32_CVT) gives bit-identical outputs and states on a multi-chunk
    varlen call with both state dtypes."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_39_gb300 as kda
    from gated_delta_rule_39_gb300 import _build
    lib = kda.load_library()
    cvt = kda.declare(ctypes.CDLL(_build.build(lib="libkda_tf32cvt.so",
                                               extra_flags=["-DKDA_TF32_CVT"])))
    lens = [300, 17, 0, 529, 64]
    d = synth.make_inputs(1, sum(lens), 4, seed=42, lengths=lens, init_dtype="bf16")
    x = upload(d)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    res = []
    for lib_ in (lib, cvt):
        out = torch.full((1, sum(lens), 4, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        fs = torch.full((5, 4, 128, 128), float("nan"), device="cuda")
        rc = lib_.kda_fwd(p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]),
                          ctypes.c_float(d["scale"]), p(out), p(x["A_log"]), p(x["dt_bias"]),
                          ctypes.c_float(d["lower_bound"]), p(x["initial_state"]), 0, p(fs), 1,
                          p(x["cu_seqlens"]), 5, 1, sum(lens), 4, 128, 128, None)
        assert rc == 0
        torch.cuda.synchronize()
        assert lib_.kda_fwd_get_error(None) == 0
        res.append((out, fs))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
