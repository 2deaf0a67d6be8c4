"""Sequence split of fixed-length calls (kda_fwd_segments; kda_fwd picks it for long
calls with few (sequence, head) recurrences).

The recurrence is affine in the state, S_end = P S_start + B over a segment, so a
sequence cut into s segments runs as window 0 (segment 0, and B and P of every
middle segment), a combine step and window 1 (segments 1 .. s-1).  These tests
compare the split against the fp64 oracle, including the cases that make P far
from zero (no decay) and the ones that make it vanish (every gate at the bound),
and check the argument errors on the host.
"""
import ctypes

import numpy as np
import pytest

import synth
from gpu_harness import run_oracle, to_f64, upload
from parity import out_error, state_error

KDA_ERR_SEGMENTS = -15


def _run(d, segments, final_dtype="f32", x=None, alias=False):
    import torch
    import gated_delta_rule_39_gb300 as kda
    x = upload(d) if x is None else x
    B, T, H, _ = d["q"].shape
    out = torch.full((B, T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    fs = None
    if alias:
        fs = x["initial_state"].clone()
        s0 = fs
    else:
        s0 = x["initial_state"]
        if final_dtype is not None:
            dt = torch.float32 if final_dtype == "f32" else torch.bfloat16
            fs = torch.full((B, H, 128, 128), float("nan"), dtype=dt, device="cuda")
    kda.kda_fwd_segments(x["q"], x["k"], x["v"], x["g"], x["beta"], d["scale"], out, x["A_log"],
                         x["dt_bias"], d["lower_bound"], initial_state=s0, final_state=fs,
                         num_segments=segments)
    torch.cuda.synchronize()
    assert kda.kda_fwd_get_error() == 0
    return out, fs


def _check(d, out, fs):
    ro, rs = run_oracle(d)
    e = out_error(to_f64(out), ro)
    assert e["ok"], e
    if fs is not None:
        se = state_error(to_f64(fs), rs)
        assert se["ok"], se
    return e


@pytest.mark.gpu
@pytest.mark.parametrize("segments", [2, 3, 5, 19])
@pytest.mark.parametrize("B", [1, 2])
def test_segments_match_oracle(segments, B):
    """300 tokens (19 chunks, the last one ragged) cut into 2, 3, 5 or 19 segments
    (19: one chunk each)."""
    d = synth.make_inputs(B, 300, 2, seed=60 + segments + 10 * B, init_dtype="f32")
    out, fs = _run(d, segments)
    _check(d, out, fs)


@pytest.mark.gpu
@pytest.mark.parametrize("init,final", [("bf16", "bf16"), ("bf16", "f32"), (None, "f32"),
                                        ("f32", None)])
def test_segments_state_dtypes(init, final):
    d = synth.make_inputs(1, 500, 3, seed=70, init_dtype=init)
    out, fs = _run(d, 4, final_dtype=final)
    _check(d, out, fs)


@pytest.mark.gpu
@pytest.mark.parametrize("lower_bound", [0.0, -1.0, -5.4])
def test_segments_across_decay_range(lower_bound):
    """lower_bound = 0: no decay, so each segment's transition P is a product of
    (I - b k k^T) factors far from zero and the combine step carries the whole
    earlier state; -5.4: every gate may reach the bound, P all but vanishes."""
    d = synth.make_inputs(1, 1000, 2, seed=71, init_dtype="f32", lower_bound=lower_bound)
    out, fs = _run(d, 6)
    _check(d, out, fs)


@pytest.mark.gpu
def test_segments_in_place_state():
    """initial_state and final_state the same buffer: window 0 reads it, window 1
    writes it."""
    d = synth.make_inputs(1, 400, 2, seed=72, init_dtype="f32")
    out, fs = _run(d, 3, alias=True)
    _check(d, out, fs)


@pytest.mark.gpu
def test_segments_deterministic_and_one_pass_close():
    import torch
    d = synth.make_inputs(1, 700, 2, seed=73, init_dtype="f32")
    x = upload(d)
    a = _run(d, 4, x=x)
    b = _run(d, 4, x=x)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    one = _run(d, 1, x=x)
    # one pass and split differ by rounding only
    o1, o2 = to_f64(one[0]), to_f64(a[0])
    rms = np.sqrt(np.mean(o1 ** 2))
    assert np.max(np.abs(o1 - o2)) < 2e-2 * rms


@pytest.mark.gpu
def test_automatic_split_on_few_heads():
    """kda_fwd on 4,096 tokens x 4 heads splits by itself (4 segments of 1,024 tokens:
    two fused launches and one combine) and matches the oracle."""
    import gated_delta_rule_39_gb300 as kda
    from gpu_harness import run_gpu
    d = synth.make_inputs(1, 4096, 4, seed=74, init_dtype="bf16")
    kda.kda_profile_enable(True)
    out, fs = run_gpu(d)
    prof = kda.kda_profile_read()
    kda.kda_profile_enable(False)
    assert prof["fused_kernel"][1] == 2 and prof["combine_kernel"][1] == 1
    assert prof["segprep_kernel"][1] == 1 and prof["segfinal_kernel"][1] == 1
    assert kda.kda_fwd_workspace_bytes(1, 4096, 4) == 65536 * 4 * (5 * 4 - 7) + 4096 * 4
    _check(d, out, fs)


@pytest.mark.gpu
def test_many_heads_run_one_pass():
    """96 heads leave no SMs for a split: kda_fwd runs one pass, bit-equal to
    num_segments = 1."""
    import torch
    import gated_delta_rule_39_gb300 as kda
    from gpu_harness import run_gpu
    d = synth.make_inputs(1, 4096, 96, seed=75, init_dtype="bf16")
    x = upload(d)
    kda.kda_profile_enable(True)
    out, fs = run_gpu(d, x=x)
    prof = kda.kda_profile_read()
    kda.kda_profile_enable(False)
    assert prof["fused_kernel"][1] == 1 and prof["combine_kernel"][1] == 0
    assert prof["segprep_kernel"][1] == 0
    one = _run(d, 1, x=x)
    assert torch.equal(out, one[0]) and torch.equal(fs, one[1])


def test_segment_argument_errors():
    """Rejected on the host before anything runs: a negative count, a split of a varlen
    call, more segments than 16-token chunks."""
    import gated_delta_rule_39_gb300 as kda
    from gated_delta_rule_39_gb300 import _build
    _build.build()
    lib = kda.load_library()
    fake = ctypes.c_void_p(0x10000)

    def call(segs, T=100, cu=None, n=0):
        return lib.kda_fwd_segments(fake, fake, fake, fake, ctypes.c_void_p(0x90000), 0.1,
                                    ctypes.c_void_p(0x80000000), fake, fake, -5.0, None, 0, None,
                                    0, cu, n, 1, T, 1, 128, 128, segs, None)

    assert call(-1) == KDA_ERR_SEGMENTS
    assert call(3, cu=ctypes.c_void_p(0x20000), n=2) == KDA_ERR_SEGMENTS
    assert call(8, T=100) == KDA_ERR_SEGMENTS     # 7 chunks of 16 tokens
    assert call(8, T=112) == KDA_ERR_SEGMENTS     # exactly 7 chunks
    assert "num_segments" in kda.kda_status_string(KDA_ERR_SEGMENTS)
