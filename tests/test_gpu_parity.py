"""CUDA path (through the C ABI) against the fp64 oracle, element by element.

Every case compares every output element and every final-state element of
every (sequence, head) unit, the full-size workloads included (the oracle
runs all heads of a T = 8192 workload in a few seconds on the host cores).
"""
import numpy as np
import pytest

import synth
from gpu_harness import run_gpu, run_oracle, to_f64, upload
from parity import out_error, state_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_39_gb300 as kda
    kda.load_library()


def _check(d, heads=None, final_dtype="f32", tag=""):
    out, fs = run_gpu(d, final_dtype=final_dtype)
    ro, rs = run_oracle(d, heads=heads)
    o = to_f64(out)
    if heads is not None:
        o = o[:, :, heads]
        ro = ro[:, :, heads]
        rs = rs[:, heads]
    e = out_error(o, ro)
    assert e["ok"], f"{tag} out: {e}"
    if fs is not None:
        s = to_f64(fs)
        if heads is not None:
            s = s[:, heads]
        se = state_error(s, rs)
        assert se["ok"], f"{tag} state: {se}"
        return e, se
    return e, None


def test_tiny_workload():
    d = synth.make_workload("tiny_t64_h1")
    _check(d, tag="tiny")


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 31, 33, 100])
@pytest.mark.parametrize("B", [1, 2])
def test_ragged_lengths(T, B):
    d = synth.make_inputs(B, T, 2, seed=T + 100 * B, init_dtype="f32")
    _check(d, tag=f"B={B} T={T}")


@pytest.mark.parametrize("init", [None, "bf16", "f32"])
@pytest.mark.parametrize("final", ["f32", "bf16", None])
def test_state_dtypes(init, final):
    d = synth.make_inputs(1, 77, 3, seed=5, init_dtype=init)
    _check(d, final_dtype=final, tag=f"init={init} final={final}")


@pytest.mark.parametrize("lower_bound", [-5.4, 0.0])
@pytest.mark.parametrize("pattern", ["saturated", "mixed"])
def test_gate_range_edges(lower_bound, pattern):
    """Gates at the ends of the accepted range.  "saturated": every per-token
    log-decay equals lower_bound (at -5.4 a chunk spans 124.6 bits of decay, so the
    in-chunk factors 2^(+-G) reach the edge of the normal fp32 range); "mixed": even
    key channels decay at the bound and odd ones hardly at all.  lower_bound = 0 is
    the ungated delta rule."""
    d = synth.make_inputs(1, 100, 2, seed=21, init_dtype="f32", lower_bound=lower_bound)
    g = synth.bf16_bits_to_f32(d["g"]).copy()
    if pattern == "saturated":
        g[:] = 8.0
    else:
        g[..., 0::2] = 8.0
        g[..., 1::2] = -8.0
    d["g"] = synth.f32_to_bf16_bits(g)
    d["A_log"][:] = np.float32(np.log(16.0))   # sigmoid(16 (g + dt_bias)) is 0 or 1 in fp32
    _check(d, tag=f"lower_bound={lower_bound} {pattern}")


@pytest.mark.parametrize("similarity", [1.0, 0.99, 0.9])
@pytest.mark.parametrize("lower_bound", [0.0, -1.0])
def test_nearly_parallel_keys(similarity, lower_bound):
    """Keys of every token nearly equal (cosine `similarity` with token 0's key), write
    strength b ~ 1: A = diag(b) A_kk is then close to the all-ones strictly lower matrix,
    whose inverse (I + A)^-1 is I minus the subdiagonal although the powers of A grow to
    C(14, 7); with lower_bound = 0 nothing damps them."""
    d = synth.make_inputs(1, 64, 2, seed=41, init_dtype="f32", lower_bound=lower_bound)
    k = synth.bf16_bits_to_f32(d["k"]).astype(np.float64)
    mix = similarity * k[:, :1] + np.sqrt(max(0.0, 1.0 - similarity ** 2)) * k
    mix /= np.linalg.norm(mix, axis=-1, keepdims=True)
    d["k"] = synth.f32_to_bf16_bits(mix.astype(np.float32))
    d["beta"] = synth.f32_to_bf16_bits(np.full(d["beta"].shape, 12.0, np.float32))
    _check(d, tag=f"similarity={similarity} lower_bound={lower_bound}")


@pytest.mark.parametrize("pattern", ["alternate", "random_sign"])
def test_sign_flipping_keys(pattern):
    """One key with flipping signs (k, -k, k, ... or random signs), b ~ 1, no decay: the
    entries of A are +-1, the delta rule overwrites the same direction every token."""
    d = synth.make_inputs(1, 64, 2, seed=43, init_dtype="f32", lower_bound=0.0)
    k = synth.bf16_bits_to_f32(d["k"]).astype(np.float64)
    T = k.shape[1]
    if pattern == "alternate":
        sign = np.where(np.arange(T) % 2 == 0, 1.0, -1.0)
    else:
        sign = np.random.default_rng(5).choice([-1.0, 1.0], size=T)
    d["k"] = synth.f32_to_bf16_bits((k[:, :1] * sign[None, :, None, None]).astype(np.float32))
    d["beta"] = synth.f32_to_bf16_bits(np.full(d["beta"].shape, 12.0, np.float32))
    _check(d, tag=pattern)


def test_large_values():
    """v scaled by 1,000 (components up to a few thousand, inside the fp16 range that
    the u product needs) and a large initial state: the error stays relative."""
    d = synth.make_inputs(1, 100, 2, seed=45, init_dtype="f32")
    v = synth.bf16_bits_to_f32(d["v"]) * np.float32(1000.0)
    d["v"] = synth.f32_to_bf16_bits(v)
    d["initial_state"] = d["initial_state"] * np.float32(1000.0)
    _check(d, tag="large v")


def test_varlen_edge_lengths():
    lens = [1, 15, 16, 17, 0, 33, 64, 5, 2]
    d = synth.make_inputs(1, sum(lens), 4, seed=11, lengths=lens, init_dtype="f32")
    _check(d, tag="varlen edges")


@pytest.mark.parametrize("N", [3000, 9000, 20000])
def test_varlen_many_short_sequences(N):
    """Thousands of short sequences (lengths 0-20, empty ones included) in one call:
    many waves of small units, the longest-first order for N <= 16384 and the input
    order above it."""
    rng = np.random.default_rng(N)
    lens = rng.integers(0, 21, size=N)
    d = synth.make_inputs(1, int(lens.sum()), 2, seed=N, lengths=list(lens), init_dtype="f32")
    _check(d, tag=f"N={N}")


def test_varlen_single_sequence_equals_fixed():
    import torch
    d = synth.make_inputs(1, 200, 2, seed=12, init_dtype="f32")
    o1, s1 = run_gpu(d)
    d2 = dict(d)
    d2["cu_seqlens"] = np.array([0, 200], np.int32)
    o2, s2 = run_gpu(d2)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_prefill_h64_all_heads():
    d = synth.make_workload("prefill_t8192_h64")
    _check(d, tag="prefill h64")


def test_prefill_h96_all_heads():
    d = synth.make_workload("prefill_t8192_h96")
    _check(d, tag="prefill h96")


def test_varlen_mixed_all_heads():
    d = synth.make_workload("varlen_mixed_t8192_h96")
    _check(d, tag="varlen mixed")


def test_varlen_uniform_all_heads():
    d = synth.make_workload("varlen_uniform_8x1024_h96")
    _check(d, tag="varlen uniform")


def test_long_context_state_carry():
    """T=65536, H=32 in two 32768-token calls carrying the fp32 state: one pass
    (num_segments = 1) gives exactly the single call's result; kda_fwd (which splits
    these 32-head calls into 3 segments) matches the oracle on every head, in one call
    and in two."""
    import torch
    import gated_delta_rule_39_gb300 as kda
    d = synth.make_workload("carry_t65536_h32")
    x = upload(d)
    H, T = 32, 65536
    half = T // 2
    sl = lambda t, a, b: t[:, a:b].contiguous()

    def run(fn, segs=None):
        full = torch.empty((1, T, H, 128), dtype=torch.bfloat16, device="cuda:0")
        S_full = torch.empty((1, H, 128, 128), dtype=torch.float32, device="cuda:0")
        kw = {} if segs is None else {"num_segments": segs}
        fn(x["q"], x["k"], x["v"], x["g"], x["beta"], d["scale"], full, x["A_log"],
           x["dt_bias"], d["lower_bound"], final_state=S_full, **kw)
        S_mid = torch.empty_like(S_full)
        S_end = torch.empty_like(S_full)
        o1 = torch.empty((1, half, H, 128), dtype=torch.bfloat16, device="cuda:0")
        o2 = torch.empty_like(o1)
        fn(sl(x["q"], 0, half), sl(x["k"], 0, half), sl(x["v"], 0, half),
           sl(x["g"], 0, half), sl(x["beta"], 0, half), d["scale"], o1, x["A_log"],
           x["dt_bias"], d["lower_bound"], final_state=S_mid, **kw)
        fn(sl(x["q"], half, T), sl(x["k"], half, T), sl(x["v"], half, T),
           sl(x["g"], half, T), sl(x["beta"], half, T), d["scale"], o2, x["A_log"],
           x["dt_bias"], d["lower_bound"], initial_state=S_mid, final_state=S_end, **kw)
        torch.cuda.synchronize()
        return full, S_full, torch.cat([o1, o2], dim=1), S_end

    # one pass: chunk boundaries coincide at 32768, so the arithmetic is identical
    full, S_full, split, S_end = run(kda.kda_fwd_segments, 1)
    assert torch.equal(split, full)
    assert torch.equal(S_end, S_full)
    ro, rs = run_oracle(d)
    r = run(kda.kda_fwd)
    for o, s_ in [(full, S_full), (r[0], r[1]), (r[2], r[3])]:
        e = out_error(to_f64(o), ro)
        assert e["ok"], e
        se = state_error(to_f64(s_), rs)
        assert se["ok"], se


@pytest.mark.parametrize("segments", [1, 0])
def test_maximum_size_tail(segments):
    """The largest call the boundary accepts with one head: T = 2^24 - 7 tokens, so each
    token tensor holds 2^31 - 896 elements (the limit is 2^31) and the last chunk is
    ragged.  The oracle cannot replay 16.8 M tokens, but the recurrence forgets: over
    256 tokens every channel's decay exp(sum of gates) is below exp(-300) in this
    recipe, so the outputs of the last 256 tokens and the final state equal those of
    the oracle started from a zero state on the last 512 tokens (checked here against a
    768-token window).  This covers the far end of maximal tensors, where 32-bit index
    arithmetic would overflow first.  Run in one pass and as kda_fwd runs it (split
    into 77 segments on 152 SMs)."""
    import torch
    import gated_delta_rule_39_gb300 as kda
    T, H = (1 << 24) - 7, 1
    assert T * H * 128 < (1 << 31)
    d = synth.make_inputs_device(T, H, seed=31)
    out = torch.empty((1, T, H, 128), dtype=torch.bfloat16, device="cuda:0")
    fs = torch.empty((1, H, 128, 128), dtype=torch.float32, device="cuda:0")
    kda.kda_fwd_segments(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], out,
                         torch.from_numpy(d["A_log"]).cuda(), torch.from_numpy(d["dt_bias"]).cuda(),
                         d["lower_bound"], final_state=fs, num_segments=segments)
    torch.cuda.synchronize()
    assert kda.kda_fwd_get_error() == 0
    tail = 256

    def oracle_window(w):
        win = {n: synth.window_bits(d[n], T - w, T) for n in ("q", "k", "v", "g", "beta")}
        win.update(A_log=d["A_log"], dt_bias=d["dt_bias"], lower_bound=d["lower_bound"],
                   scale=d["scale"], initial_state=None, cu_seqlens=None)
        return run_oracle(win)

    ro, rs = oracle_window(512)
    ro2, rs2 = oracle_window(768)
    # the window is long enough: a longer one changes nothing
    assert np.max(np.abs(ro[:, -tail:] - ro2[:, -tail:])) < 1e-12
    assert np.max(np.abs(rs - rs2)) < 1e-12
    o = to_f64(out[:, T - tail:])
    e = out_error(o, ro[:, -tail:])
    assert e["ok"], e
    se = state_error(to_f64(fs), rs)
    assert se["ok"], se


def test_state_buffers_may_alias():
    import torch
    import gated_delta_rule_39_gb300 as kda
    d = synth.make_inputs(2, 50, 2, seed=21, init_dtype="f32")
    x = upload(d)
    ref_out, ref_S = run_gpu(d, x=x)
    S = x["initial_state"].clone()
    out = torch.empty_like(ref_out)
    kda.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], d["scale"], out, x["A_log"],
                x["dt_bias"], d["lower_bound"], initial_state=S, final_state=S)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(S, ref_S)


def test_zero_length_passes_state_through():
    import torch
    import gated_delta_rule_39_gb300 as kda
    d = synth.make_inputs(1, 0, 2, seed=3, init_dtype="f32")
    x = upload(d)
    fs = torch.full((1, 2, 128, 128), float("nan"), device="cuda:0")
    out = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device="cuda:0")
    kda.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], d["scale"], out, x["A_log"],
                x["dt_bias"], d["lower_bound"], initial_state=x["initial_state"], final_state=fs)
    torch.cuda.synchronize()
    assert torch.equal(fs, x["initial_state"])


def test_bad_cu_seqlens_reports_error_and_writes_nothing():
    import torch
    import gated_delta_rule_39_gb300 as kda
    d = synth.make_inputs(1, 64, 2, seed=4, lengths=[30, 34], init_dtype="f32")
    x = upload(d)
    x["cu_seqlens"] = torch.tensor([0, 40, 30], dtype=torch.int32, device="cuda:0")
    assert kda.kda_fwd_get_error() == 0
    out, fs = run_gpu(d, x=x)
    assert kda.kda_fwd_get_error() == -8          # KDA_ERR_BAD_SEQLENS
    assert torch.isnan(out.float()).all() and torch.isnan(fs).all()
    assert kda.kda_fwd_get_error() == 0           # the word is cleared by reading it
    # a later valid call works normally
    d2 = synth.make_inputs(1, 64, 2, seed=4, lengths=[30, 34], init_dtype="f32")
    _check(d2, tag="after bad call")


def test_deterministic():
    import torch
    d = synth.make_inputs(1, 300, 4, seed=8, lengths=[100, 3, 197], init_dtype="bf16")
    o1, s1 = run_gpu(d)
    o2, s2 = run_gpu(d)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_deterministic_across_waves():
    """Several waves of CTAs per SM (768 units on 152 SMs): repeated calls are bit-identical.
    Catches state left behind by one CTA that a later CTA on the same SM could see."""
    import torch
    d = synth.make_workload("varlen_uniform_8x1024_h96")
    x = upload(d)
    o1, s1 = run_gpu(d, x=x)
    for _ in range(4):
        o2, s2 = run_gpu(d, x=x)
        assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_host_entry_point_matches_device_entry_point():
    import torch
    import gated_delta_rule_39_gb300 as kda
    d = synth.make_inputs(1, 90, 2, seed=9, lengths=[40, 50], init_dtype="f32")
    o_dev, s_dev = run_gpu(d)
    x = upload(d, "cpu")
    out = torch.empty((1, 90, 2, 128), dtype=torch.bfloat16).pin_memory()
    fs = torch.empty((2, 2, 128, 128), dtype=torch.float32).pin_memory()
    kda.kda_fwd_host(x["q"].pin_memory(), x["k"].pin_memory(), x["v"].pin_memory(),
                     x["g"].pin_memory(), x["beta"].pin_memory(), d["scale"], out, x["A_log"],
                     x["dt_bias"], d["lower_bound"], initial_state=x["initial_state"],
                     final_state=fs, cu_seqlens=x["cu_seqlens"])
    assert torch.equal(out, o_dev.cpu()) and torch.equal(fs, s_dev.cpu())


@pytest.mark.parametrize("init,final", [("f32", "f32"), ("bf16", "bf16"), (None, None)])
def test_host_entry_point_blocks_match_device_entry_point(init, final):
    """T = 3000 on the host entry point runs as token blocks of 1024, 1024 and 952
    with the state carried between them; the result must be that of one call."""
    import torch
    import gated_delta_rule_39_gb300 as kda
    d = synth.make_inputs(1, 3000, 2, seed=17, init_dtype=init)
    o_dev, s_dev = run_gpu(d, final_dtype=final)
    x = upload(d, "cpu")
    out = torch.empty((1, 3000, 2, 128), dtype=torch.bfloat16).pin_memory()
    fs = None
    if final is not None:
        dt = torch.float32 if final == "f32" else torch.bfloat16
        fs = torch.empty((1, 2, 128, 128), dtype=dt).pin_memory()
    s0 = x["initial_state"]
    kda.kda_fwd_host(x["q"].pin_memory(), x["k"].pin_memory(), x["v"].pin_memory(),
                     x["g"].pin_memory(), x["beta"].pin_memory(), d["scale"], out, x["A_log"],
                     x["dt_bias"], d["lower_bound"],
                     initial_state=None if s0 is None else s0.pin_memory(), final_state=fs)
    assert torch.equal(out, o_dev.cpu())
    if fs is not None:
        assert torch.equal(fs, s_dev.cpu())


def test_profile_counts_launches():
    import gated_delta_rule_39_gb300 as kda
    d = synth.make_inputs(1, 64, 2, seed=2, lengths=[20, 44])
    kda.kda_profile_enable(True)
    run_gpu(d)
    run_gpu(d)
    prof = kda.kda_profile_read()
    kda.kda_profile_enable(False)
    assert prof["seqmap_kernel"][1] == 2 and prof["fused_kernel"][1] == 2
    assert all(ms > 0 for ms, n in prof.values() if n)


@pytest.mark.parametrize("N,H,lo,hi", [(2000, 2, 0, 40), (300, 3, 100, 400), (160, 1, 0, 0)])
def test_persistent_schedule_equals_one_cta_per_unit(N, H, lo, hi):
    """Varlen calls with more (sequence, head) units than SMs run persistent CTAs that
    take units from a device counter, longest first, with their pipelines carried from
    unit to unit; kda_fwd_noalloc always runs one CTA per unit.  The arithmetic of every
    unit is the same, so the results are bit-identical (here with empty sequences, one
    chunk, many chunks, ragged ends, and a call of empty sequences only)."""
    import torch
    import gated_delta_rule_39_gb300 as kda
    rng = np.random.default_rng(N + H)
    lens = [int(x) for x in rng.integers(lo, hi + 1, size=N)]
    T = sum(lens)
    d = synth.make_inputs(1, T, H, seed=N, lengths=lens, init_dtype="f32")
    x = upload(d)
    res = []
    for fn in (kda.kda_fwd, kda.kda_fwd_noalloc):
        out = torch.full((1, T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        fs = torch.full((N, H, 128, 128), float("nan"), device="cuda")
        fn(x["q"], x["k"], x["v"], x["g"], x["beta"], d["scale"], out, x["A_log"], x["dt_bias"],
           d["lower_bound"], initial_state=x["initial_state"], final_state=fs,
           cu_seqlens=x["cu_seqlens"])
        torch.cuda.synchronize()
        assert kda.kda_fwd_get_error() == 0
        res.append((out, fs))
    assert torch.equal(res[0][0], res[1][0]) or T == 0
    assert torch.equal(res[0][1], res[1][1])
    if T > 0 and N * H <= 900:
        ro, rs = run_oracle(d)
        e = out_error(to_f64(res[0][0]), ro)
        assert e["ok"], e
        assert state_error(to_f64(res[0][1]), rs)["ok"]


def test_varlen_short_20000_sampled_heads():
    """The many-short-prompts workload at full size (20,000 sequences of 0-16 tokens,
    16 heads, 320,000 units: the persistent schedule) against the oracle on three
    heads, every sequence of each."""
    d = synth.make_workload("varlen_short_20000_h16")
    _check(d, heads=[0, 7, 15], final_dtype=None, tag="short20000")


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["fixed", "varlen", "short_persistent"])
def test_no_initial_state_equals_zero_state(case):
    """Without an initial state every unit starts from zero, and the kernel leaves out
    the first chunk's products with the state (they would add exact zeros).  The
    results must be bit for bit those of an explicit all-zero fp32 initial state (and
    the outputs the same without a final state), on one CTA per unit (fixed length,
    varlen) and on persistent CTAs (many short sequences)."""
    import torch
    import gated_delta_rule_39_gb300 as kda
    if case == "fixed":
        d = synth.make_inputs(2, 300, 3, seed=91)
    elif case == "varlen":
        d = synth.make_inputs(1, 135, 3, seed=92, lengths=[17, 0, 48, 1, 69])
    else:
        rng = np.random.default_rng(93)
        lens = [int(x) for x in rng.integers(0, 21, size=2000)]
        d = synth.make_inputs(1, sum(lens), 1, seed=93, lengths=lens)
    x = upload(d)
    B, T, H, _ = d["q"].shape
    N = d["N"]
    zero = torch.zeros((N, H, 128, 128), dtype=torch.float32, device="cuda")
    res = []
    for s0 in (None, zero):
        out = torch.full((B, T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        fs = torch.full((N, H, 128, 128), float("nan"), device="cuda")
        kda.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], d["scale"], out, x["A_log"],
                    x["dt_bias"], d["lower_bound"], initial_state=s0, final_state=fs,
                    cu_seqlens=x["cu_seqlens"])
        torch.cuda.synchronize()
        assert kda.kda_fwd_get_error() == 0
        res.append((out, fs))
    assert torch.equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1])
    # and without a final state: the same outputs
    out = torch.full((B, T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    kda.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], d["scale"], out, x["A_log"],
                x["dt_bias"], d["lower_bound"], cu_seqlens=x["cu_seqlens"])
    torch.cuda.synchronize()
    assert kda.kda_fwd_get_error() == 0
    assert torch.equal(out, res[0][0])
    ro, rs = run_oracle(d)
    assert out_error(to_f64(res[0][0]), ro)["ok"]
    assert state_error(to_f64(res[0][1]), rs)["ok"]
