"""Seeded input generator and the frozen oracle fixture (CPU only)."""
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_t64_h1.txt")


def test_generator_is_deterministic():
    a = synth.make_inputs(1, 40, 2, seed=3, lengths=[7, 33], init_dtype="f32")
    b = synth.make_inputs(1, 40, 2, seed=3, lengths=[7, 33], init_dtype="f32")
    for key in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state", "cu_seqlens"):
        assert np.array_equal(a[key], b[key]), key


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38, 1e-40], np.float32)
    bits = synth.f32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(bits)
    assert back[0] == 1.0
    assert back[1] == 1.0                    # tie rounds to even (mantissa 0)
    assert back[2] == 1.0 + 4 * 2 ** -8      # tie rounds to even (up)
    assert back[3] == -2.5
    assert np.isfinite(back[4])


def test_workload_shapes_and_distributions():
    d = synth.make_inputs(1, 512, 4, init_dtype="bf16")
    q = synth.bf16_bits_to_f32(d["q"]).astype(np.float64)
    n = np.linalg.norm(q, axis=-1)
    assert np.all(np.abs(n - 1) < 1e-2)
    v = synth.bf16_bits_to_f32(d["v"])
    assert abs(v.std() - 1) < 0.05 and abs(v.mean()) < 0.05
    assert np.all((d["A_log"] >= 0) & (d["A_log"] <= np.log(16)))
    assert abs(d["dt_bias"].std() - 0.1) < 0.03
    s0 = synth.bf16_bits_to_f32(d["initial_state"])
    assert s0.shape == (1, 4, 128, 128) and abs(s0.std() - 0.02) < 0.002
    assert d["scale"] == pytest.approx(128 ** -0.5)


def test_mixed_lengths_recipe():
    d = synth.make_inputs(1, 8192, 1, lengths="mixed12", init_dtype="f32")
    cu = d["cu_seqlens"]
    lens = np.diff(cu)
    assert len(lens) == 12 and cu[0] == 0 and cu[-1] == 8192
    assert lens.min() >= 1 and np.count_nonzero(lens % 16) >= 3
    assert d["initial_state"].shape == (12, 1, 128, 128)


def test_uniform_lengths_recipe():
    d = synth.make_inputs(1, 8192, 1, lengths="uniform8x1024")
    assert np.array_equal(np.diff(d["cu_seqlens"]), np.full(8, 1024))


def test_golden_fixture_matches_oracle():
    """The oracle still gives the frozen numbers for the tiny workload."""
    from golden.make_golden import compute
    out, S = compute()
    rows = [ln.split() for ln in open(GOLDEN) if not ln.startswith("#")]
    for r in rows:
        if r[0] == "out_rms":
            assert float(r[1]) == pytest.approx(np.sqrt(np.mean(out ** 2)), rel=1e-12)
        elif r[0] == "state_fro":
            assert float(r[1]) == pytest.approx(np.linalg.norm(S), rel=1e-12)
        elif r[0] == "out":
            assert out[int(r[1]), int(r[2])] == pytest.approx(float(r[3]), rel=1e-12, abs=1e-15)
        elif r[0] == "state":
            assert S[int(r[1]), int(r[2])] == pytest.approx(float(r[3]), rel=1e-12, abs=1e-15)


def test_short_lengths_recipe():
    """20,000 lengths in [0, 16] summing to 160,000, the same for the same seed."""
    a = synth.short_lengths(np.random.default_rng(5))
    b = synth.short_lengths(np.random.default_rng(5))
    assert a.shape == (20000,) and a.sum() == 160000
    assert a.min() >= 0 and a.max() <= 16 and (a == 0).any() and (a == 16).any()
    assert np.array_equal(a, b)
    assert synth.WORKLOADS["varlen_short_20000_h16"].final_dtype is None
