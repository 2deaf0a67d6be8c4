"""kda_decode: one decode step (a single token per sequence applied to the states).

GPU tests compare it with the fp64 oracle's token recurrence (the same definition
the prefill is checked against), element by element; CPU tests check the host-side
argument validation (nothing is launched)."""
import ctypes

import numpy as np
import pytest

import synth
from gpu_harness import bf16_tensor, to_f64, upload
from parity import out_error, state_error


def _device_inputs(d, device="cuda:0"):
    """kda_decode's layout: [N, H, 128] tensors from a [N, 1, H, 128] draw."""
    x = upload(d, device)
    N, T, H, K = d["q"].shape
    assert T == 1
    y = {n: x[n].reshape(N, H, K) for n in ("q", "k", "v", "g")}
    y["beta"] = x["beta"].reshape(N, H)
    y["A_log"], y["dt_bias"], y["initial_state"] = x["A_log"], x["dt_bias"], x["initial_state"]
    return y


def _decode(kda, d, y, state_in, state_out):
    import torch
    N, _, H, K = d["q"].shape
    out = torch.full((N, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    kda.kda_decode(y["q"], y["k"], y["v"], y["g"], y["beta"], d["scale"], out, y["A_log"],
                   y["dt_bias"], d["lower_bound"], state_in=state_in, state_out=state_out)
    return out


def _oracle(d):
    import oracle
    return oracle.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["A_log"],
                          d["dt_bias"], d["lower_bound"], initial_state=d.get("initial_state"))


@pytest.fixture(scope="module")
def kda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_39_gb300 as kda
    kda.load_library()
    return kda


@pytest.mark.gpu
@pytest.mark.parametrize("init,final", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32"),
                                        (None, "f32"), ("f32", None)])
def test_decode_step_matches_oracle(kda, init, final):
    import torch
    d = synth.make_inputs(7, 1, 3, seed=51, init_dtype=init)
    y = _device_inputs(d)
    so = None
    if final is not None:
        so = torch.full((7, 3, 128, 128), float("nan"),
                        dtype=torch.float32 if final == "f32" else torch.bfloat16, device="cuda")
    out = _decode(kda, d, y, y["initial_state"], so)
    torch.cuda.synchronize()
    ro, rs = _oracle(d)
    e = out_error(to_f64(out), ro.reshape(7, 3, 128))
    assert e["ok"], e
    if so is not None:
        se = state_error(to_f64(so), rs)
        assert se["ok"], se


@pytest.mark.gpu
def test_decode_steps_in_place_equal_a_prefill_of_the_same_tokens(kda):
    """40 decode steps updating fp32 states in place give the oracle's 40-token run."""
    import torch
    N, H, T = 5, 2, 40
    d = synth.make_inputs(N, T, H, seed=52, init_dtype="f32")
    x = upload(d)
    state = x["initial_state"].clone()
    outs = []
    for t in range(T):
        step = {n: x[n][:, t].contiguous() for n in ("q", "k", "v", "g", "beta")}
        out = torch.empty((N, H, 128), dtype=torch.bfloat16, device="cuda")
        kda.kda_decode(step["q"], step["k"], step["v"], step["g"], step["beta"], d["scale"], out,
                       x["A_log"], x["dt_bias"], d["lower_bound"], state_in=state, state_out=state)
        outs.append(out)
    torch.cuda.synchronize()
    got = torch.stack(outs, dim=1)
    ro, rs = _oracle(d)
    e = out_error(to_f64(got), ro)
    assert e["ok"], e
    se = state_error(to_f64(state), rs)
    assert se["ok"], se


@pytest.mark.gpu
def test_decode_continues_a_prefill(kda):
    """kda_fwd over 100 tokens, its fp32 final state fed to 20 decode steps: the oracle
    over all 120 tokens."""
    import torch
    N, H, T0, T1 = 3, 2, 100, 20
    d = synth.make_inputs(N, T0 + T1, H, seed=53, init_dtype="bf16")
    x = upload(d)
    pre = {n: x[n][:, :T0].contiguous() for n in ("q", "k", "v", "g", "beta")}
    out0 = torch.empty((N, T0, H, 128), dtype=torch.bfloat16, device="cuda")
    state = torch.empty((N, H, 128, 128), device="cuda")
    kda.kda_fwd(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], d["scale"], out0, x["A_log"],
                x["dt_bias"], d["lower_bound"], initial_state=x["initial_state"], final_state=state)
    outs = [out0]
    for t in range(T0, T0 + T1):
        step = {n: x[n][:, t].contiguous() for n in ("q", "k", "v", "g", "beta")}
        out = torch.empty((N, H, 128), dtype=torch.bfloat16, device="cuda")
        kda.kda_decode(step["q"], step["k"], step["v"], step["g"], step["beta"], d["scale"], out,
                       x["A_log"], x["dt_bias"], d["lower_bound"], state_in=state, state_out=state)
        outs.append(out.unsqueeze(1))
    torch.cuda.synchronize()
    got = torch.cat(outs, dim=1)
    ro, rs = _oracle(d)
    assert out_error(to_f64(got), ro)["ok"]
    assert state_error(to_f64(state), rs)["ok"]


@pytest.mark.gpu
def test_decode_full_batch(kda):
    """A serving-sized step (256 sequences x 96 heads, fp32 states in place), every
    element against the oracle."""
    import torch
    d = synth.make_inputs(256, 1, 96, seed=54, init_dtype="f32")
    y = _device_inputs(d)
    state = y["initial_state"].clone()
    out = _decode(kda, d, y, state, state)
    torch.cuda.synchronize()
    assert kda.kda_fwd_get_error() == 0
    ro, rs = _oracle(d)
    assert out_error(to_f64(out), ro.reshape(256, 96, 128))["ok"]
    assert state_error(to_f64(state), rs)["ok"]


def test_decode_rejects_bad_arguments():
    """Host-side checks: nothing is launched (fake, never dereferenced pointers)."""
    import gated_delta_rule_39_gb300 as kda
    from gated_delta_rule_39_gb300 import _build
    _build.build()
    lib = kda.load_library()
    fake = ctypes.c_void_p(0x10000)

    def call(**over):
        a = dict(q=fake, k=fake, v=fake, g=fake, beta=ctypes.c_void_p(0x90000), scale=0.1,
                 out=ctypes.c_void_p(0x80000000), A_log=fake, dt_bias=fake, lb=-5.0, s0=None,
                 d0=0, s1=None, d1=0, N=4, H=2, K=128, V=128)
        a.update(over)
        return lib.kda_decode(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["out"],
                              a["A_log"], a["dt_bias"], a["lb"], a["s0"], a["d0"], a["s1"],
                              a["d1"], a["N"], a["H"], a["K"], a["V"], None)
    assert call(K=64) == -3
    assert call(H=0) == -2
    assert call(q=None) == -1
    assert call(scale=float("inf")) == -12
    assert call(lb=-6.0) == -12
    assert call(q=ctypes.c_void_p(0x10008)) == -4
    assert call(s0=ctypes.c_void_p(0x100008)) == -4
    assert call(s1=ctypes.c_void_p(0x100000), d1=7) == -5
    # the output overlapping q
    assert call(out=fake) == -13
    # state_in and state_out overlapping without being the same buffer
    assert call(s0=ctypes.c_void_p(0x200000), d0=1, s1=ctypes.c_void_p(0x200100), d1=1) == -13
