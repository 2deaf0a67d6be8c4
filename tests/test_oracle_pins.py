"""The fp64 oracle against closed forms, invariants and independent algorithms (CPU only)."""
import numpy as np
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_neumann_equals_forward_substitution():
    """The 16x16 Neumann product equals forward substitution for a strictly lower A
    ("Moonshot AI Open-Sources FlashKDA", "What makes the kernel fast": chunk 16,
    16x16 inversion by Neumann series expansion)."""
    rng = np.random.default_rng(7)
    for n in (1, 5, 16):
        A = np.tril(rng.uniform(-1, 1, (n, n)), -1)
        T1 = P.inverse_forward_substitution(A)
        T2 = P.inverse_neumann(A)
        assert np.max(np.abs(T1 - T2)) <= 1e-9 * max(1.0, np.abs(T1).max())
        assert np.max(np.abs(T1 @ (np.eye(n) + A) - np.eye(n))) <= 1e-9 * max(1.0, np.abs(T1).max())


def test_chunk_interaction_bounded():
    """With unit-norm keys, beta in (0,1) and decay <= 1, every |A[r,s]| <= 1 (the pages'
    statement that the inverse's inputs lie within [-1, 1])."""
    rng = np.random.default_rng(8)
    q, k, v, la, beta = P.random_problem(rng, 1, 64, 1, 32, 8)
    stats = []
    P.chunked_unit(q[0, :, 0], k[0, :, 0], v[0, :, 0], la[0, :, 0], beta[0, :, 0], 1.0,
                   np.zeros((32, 8)), stats=stats)
    assert max(stats) <= 1.0


def test_chunked_form_with_neumann_inverse(orc):
    """The chunked form with the Neumann inverse also matches the token recurrence."""
    rng = np.random.default_rng(9)
    q, k, v, la, beta = P.random_problem(rng, 1, 35, 1, 16, 16)
    out, Sf = orc.kda_recurrence(q, k, v, la, beta, 0.5)
    o2, S2 = P.chunked_unit(q[0, :, 0], k[0, :, 0], v[0, :, 0], la[0, :, 0], beta[0, :, 0],
                            0.5, np.zeros((16, 16)), inverse=P.inverse_neumann)
    assert np.max(np.abs(out[0, :, 0] - o2)) <= 1e-10
    assert np.max(np.abs(Sf[0, 0] - S2)) <= 1e-10


def test_zero_length_and_empty(orc):
    """A zero-length sequence writes no output and passes its initial state through."""
    rng = np.random.default_rng(10)
    q, k, v, la, beta = P.random_problem(rng, 1, 3, 1, 4, 4)
    S0 = rng.standard_normal((2, 1, 4, 4))
    out, Sf = orc.kda_recurrence(q, k, v, la, beta, 1.0, initial_state=S0,
                                 cu_seqlens=np.array([0, 0, 3]))
    assert np.array_equal(Sf[0], S0[0])
    assert np.all(np.isfinite(out))


def test_full_config_gate_range(orc):
    """On the benchmark's input distribution the per-token log-decay stays inside
    [lower_bound, 0) (the sigmoid rounds to 1 in fp64 for large arguments), so a 16-token chunk spans at most 16*5/ln 2 < 116 bits of decay
    (the pages' reason for chunk 16: gate products stay representable without rescaling)."""
    import synth
    d = synth.make_inputs(1, 256, 4)
    la = orc.kda_gate(d["g"][0], d["A_log"], d["dt_bias"], d["lower_bound"])
    assert np.all(la < 0) and np.all(la >= d["lower_bound"])
    span_bits = -16 * la.min() / np.log(2)
    assert span_bits <= 16 * 5 / np.log(2) + 1e-9
