"""kda_fwd_noalloc: the entry point for callers that cannot allocate device memory.

Some users of this library cannot call cudaMalloc: a serving runtime or
framework that reserves its whole memory budget at start-up and hands out
every byte through its own allocator, or a hot loop that must not pay for
an allocation.  kda_fwd_noalloc keeps its scratch in a fixed array inside
the library instead.  These tests call it through the C ABI and check that
it gives what kda_fwd gives, on two calls in a row (the second call reuses
the array the first one left behind).  This file is collected last.
"""
import ctypes

import numpy as np
import pytest

import synth
from gpu_harness import to_f64, upload
from parity import out_error, state_error


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call(lib_fn, d, x, out, fs, stream):
    B, T, H, K = d["q"].shape
    cu = x["cu_seqlens"]
    s0 = x["initial_state"]
    return lib_fn(_ptr(x["q"]), _ptr(x["k"]), _ptr(x["v"]), _ptr(x["g"]), _ptr(x["beta"]),
                  ctypes.c_float(d["scale"]), _ptr(out), _ptr(x["A_log"]), _ptr(x["dt_bias"]),
                  ctypes.c_float(d["lower_bound"]), _ptr(s0),
                  0 if s0 is None or s0.dtype.is_floating_point and s0.element_size() == 2 else 1,
                  _ptr(fs), 1, _ptr(cu), 0 if cu is None else cu.numel() - 1, B, T, H, K, 128,
                  ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.gpu
def test_noalloc_matches_kda_fwd_on_consecutive_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_39_gb300 as kda
    lib = kda.load_library()
    stream = torch.cuda.current_stream()
    problems = [
        synth.make_inputs(1, 300, 3, seed=31, lengths=[100, 7, 0, 176, 17], init_dtype="f32"),
        synth.make_inputs(1, 260, 3, seed=32, lengths=[33, 227], init_dtype="bf16"),
        synth.make_inputs(2, 45, 3, seed=33, init_dtype="f32"),
    ]
    for d in problems:
        x = upload(d)
        B, T, H, _ = d["q"].shape
        N = d["N"]
        ref_out = torch.full((B, T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        ref_fs = torch.full((N, H, 128, 128), float("nan"), device="cuda")
        out = torch.full_like(ref_out, float("nan"))
        fs = torch.full_like(ref_fs, float("nan"))
        assert _call(lib.kda_fwd, d, x, ref_out, ref_fs, stream) == 0
        assert _call(lib.kda_fwd_noalloc, d, x, out, fs, stream) == 0
        torch.cuda.synchronize()
        assert kda.kda_fwd_get_error() == 0
        e = out_error(to_f64(out), to_f64(ref_out))
        se = state_error(to_f64(fs), to_f64(ref_fs))
        assert e["ok"] and se["ok"], (e, se)
        assert torch.equal(out, ref_out) and torch.equal(fs, ref_fs)


def test_noalloc_rejects_too_many_sequences():
    """More sequences than the fixed scratch holds: a clear error, nothing launched."""
    import gated_delta_rule_39_gb300 as kda
    from gated_delta_rule_39_gb300 import _build
    _build.build()
    lib = kda.load_library()
    fake = ctypes.c_void_p(0x10000)
    n = 65536 + 1
    rc = lib.kda_fwd_noalloc(fake, fake, fake, fake, ctypes.c_void_p(0x90000), 0.1,
                             ctypes.c_void_p(0x80000000), fake, fake, -5.0, None, 0, None, 0,
                             ctypes.c_void_p(0x20000), n, 1, 16, 1, 128, 128, None)
    assert rc == -14
    assert "KDA_NOALLOC_MAX_SEQS" in kda.kda_status_string(rc)


@pytest.mark.gpu
def test_noalloc_at_the_scratch_limit():
    """Exactly KDA_NOALLOC_MAX_SEQS (65,536) sequences: the valid flag lands in the last
    element of the fixed array and the sequence map takes its input-order path.  One
    head, mostly empty sequences and a few non-empty ones; the result equals kda_fwd's
    and no device error is raised."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_39_gb300 as kda
    lib = kda.load_library()
    stream = torch.cuda.current_stream()
    n = 65536
    lens = np.zeros(n, dtype=np.int64)
    lens[[0, 1, 777, 40000, n - 1]] = [17, 3, 32, 5, 20]
    d = synth.make_inputs(1, int(lens.sum()), 1, seed=36, lengths=list(lens), init_dtype=None)
    x = upload(d)
    T = int(lens.sum())
    ref_out = torch.full((1, T, 1, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(ref_out, float("nan"))
    assert _call(lib.kda_fwd, d, x, ref_out, None, stream) == 0
    assert _call(lib.kda_fwd_noalloc, d, x, out, None, stream) == 0
    torch.cuda.synchronize()
    assert kda.kda_fwd_get_error() == 0
    assert torch.equal(out, ref_out)
    from gpu_harness import run_oracle
    ro, _ = run_oracle(d)
    e = out_error(to_f64(out), ro)
    assert e["ok"], e
