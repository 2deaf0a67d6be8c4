"""Pins of the fp64 oracle against what the mathematics fixes.

Each ``pin_*`` function takes an ``oracle.Oracle`` instance and raises
AssertionError if the oracle disagrees with an independent statement of the
same result: a different algorithm (chunked WY form, explicit transition
matrices), a closed form of a special case, or an invariant.  The same
functions run against mutated copies of the oracle in
``test_oracle_mutants.py`` to show that plausible mistakes are caught.

The KDA recurrence (per sequence and head, S is K x V):
  S_t = (I - b_t k_t k_t^T) Diag(alpha_t) S_{t-1} + b_t k_t v_t^T,  o_t = scale S_t^T q_t.
The pages ("Moonshot AI Open-Sources FlashKDA", section "Why KDA?") call KDA
Gated DeltaNet with channel-by-channel gating and describe its chunkwise
algorithm as a Diagonal-Plus-Low-Rank variant; section "What makes the
kernel fast" fixes chunk size 16 and a 16 x 16 inverse by Neumann series.
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit

RNG_SEED = 1234


# --------------------------------------------------------------------------
# independent evaluations used as pins
# --------------------------------------------------------------------------

def inverse_forward_substitution(A: np.ndarray) -> np.ndarray:
    """(I + A)^-1 for strictly lower-triangular A by forward substitution."""
    n = A.shape[0]
    Tm = np.eye(n)
    for i in range(n):
        for j in range(i):
            Tm[i, j] = -sum(A[i, m] * Tm[m, j] for m in range(j, i))
    return Tm


def inverse_neumann(A: np.ndarray) -> np.ndarray:
    """(I + A)^-1 = (I - A)(I + A^2)(I + A^4)(I + A^8) for nilpotent A of order <= 16."""
    n = A.shape[0]
    assert n <= 16
    I = np.eye(n)
    A2 = A @ A
    A4 = A2 @ A2
    A8 = A4 @ A4
    return (I - A) @ (I + A2) @ (I + A4) @ (I + A8)


def chunked_unit(q, k, v, log_alpha, beta, scale, S0, C=16, inverse=inverse_forward_substitution,
                 stats=None):
    """Chunkwise (WY / DPLR-variant) evaluation of one (sequence, head) in fp64.

    q, k, log_alpha: [L, K]; v: [L, V]; beta: [L] (post-activation); S0: [K, V].
    Per chunk with state S at its start (Gamma = in-chunk cumulative log-decay):
      A[r,s]   = b_r sum_c k_r[c] k_s[c] exp(Gamma_r[c] - Gamma_s[c])   (s < r)
      Aqk[r,s] =     sum_c q_r[c] k_s[c] exp(Gamma_r[c] - Gamma_s[c])   (s <= r)
      T = (I + A)^-1;  u = T diag(b) V;  w = T diag(b) (K * exp(Gamma))
      U = u - w S;     O = scale ((Q * exp(Gamma)) S + Aqk U)
      S <- Diag(exp(Gamma_last)) S + (K * exp(Gamma_last - Gamma))^T U
    """
    L, K = q.shape
    S = S0.copy()
    out = np.zeros((L, v.shape[1]))
    for c0 in range(0, L, C):
        Q, Kc, Vc = q[c0:c0 + C], k[c0:c0 + C], v[c0:c0 + C]
        b = beta[c0:c0 + C]
        G = np.cumsum(log_alpha[c0:c0 + C], axis=0)
        n = Q.shape[0]
        A = np.zeros((n, n))
        Aqk = np.zeros((n, n))
        for r in range(n):
            for s in range(r + 1):
                d = np.exp(G[r] - G[s])
                Aqk[r, s] = np.sum(Q[r] * Kc[s] * d)
                if s < r:
                    A[r, s] = b[r] * np.sum(Kc[r] * Kc[s] * d)
        if stats is not None:
            stats.append(np.abs(A).max(initial=0.0))
        Tm = inverse(A)
        u = Tm @ (b[:, None] * Vc)
        w = Tm @ (b[:, None] * (Kc * np.exp(G)))
        U = u - w @ S
        out[c0:c0 + n] = scale * ((Q * np.exp(G)) @ S + Aqk @ U)
        S = np.exp(G[-1])[:, None] * S + (Kc * np.exp(G[-1] - G)).T @ U
    return out, S


def matrix_unit(q, k, v, log_alpha, beta, scale, S0):
    """Token recurrence with the K x K transition matrix formed explicitly."""
    L, K = q.shape
    S = S0.copy()
    out = np.zeros((L, v.shape[1]))
    I = np.eye(K)
    for t in range(L):
        M = (I - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(log_alpha[t]))
        S = M @ S + beta[t] * np.outer(k[t], v[t])
        out[t] = scale * S.T @ q[t]
    return out, S


# --------------------------------------------------------------------------
# random problem helpers
# --------------------------------------------------------------------------

def unit_rows(rng, shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def random_problem(rng, B, T, H, K, V, lb=-5.0):
    q = unit_rows(rng, (B, T, H, K))
    k = unit_rows(rng, (B, T, H, K))
    v = rng.standard_normal((B, T, H, V))
    # log-decay in (lb, 0), mixing near-0 and near-lb channels like the sigmoid gate does
    la = lb * expit(3.0 * rng.standard_normal((B, T, H, K)))
    beta = expit(rng.standard_normal((B, T, H)))
    return q, k, v, la, beta


def _close(a, b, tol, what):
    err = np.max(np.abs(a - b)) if np.size(a) else 0.0
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    assert err <= tol, f"{what}: max |diff| = {err:.3e} > {tol:.1e}"


# --------------------------------------------------------------------------
# pins
# --------------------------------------------------------------------------

def pin_chunked_form(orc):
    """Token recurrence == chunked WY form (C=16, forward-substitution inverse)."""
    rng = np.random.default_rng(RNG_SEED)
    for (T, K, V, with_s0) in [(1, 4, 4, False), (15, 4, 4, True), (16, 4, 3, True),
                               (17, 4, 5, False), (40, 6, 4, True), (33, 128, 128, True)]:
        H = 2
        q, k, v, la, beta = random_problem(rng, 1, T, H, K, V)
        S0 = 0.3 * rng.standard_normal((1, H, K, V)) if with_s0 else None
        out, Sf = orc.kda_recurrence(q, k, v, la, beta, 0.7, initial_state=S0)
        for h in range(H):
            s0 = S0[0, h] if with_s0 else np.zeros((K, V))
            o_ref, S_ref = chunked_unit(q[0, :, h], k[0, :, h], v[0, :, h], la[0, :, h],
                                        beta[0, :, h], 0.7, s0)
            _close(out[0, :, h], o_ref, 1e-10, f"chunked out T={T} K={K}")
            _close(Sf[0, h], S_ref, 1e-10, f"chunked state T={T} K={K}")


def pin_matrix_form(orc):
    """Token recurrence == explicit transition-matrix form, tiny sizes."""
    rng = np.random.default_rng(RNG_SEED + 1)
    q, k, v, la, beta = random_problem(rng, 1, 9, 1, 5, 3)
    S0 = rng.standard_normal((1, 1, 5, 3))
    out, Sf = orc.kda_recurrence(q, k, v, la, beta, 1.3, initial_state=S0)
    o_ref, S_ref = matrix_unit(q[0, :, 0], k[0, :, 0], v[0, :, 0], la[0, :, 0], beta[0, :, 0],
                               1.3, S0[0, 0])
    _close(out[0, :, 0], o_ref, 1e-12, "matrix-form out")
    _close(Sf[0, 0], S_ref, 1e-12, "matrix-form state")


def pin_one_token_write(orc):
    """beta=1, alpha=1, S0=0, one token: S = k v^T and o = scale (q.k) v."""
    rng = np.random.default_rng(RNG_SEED + 2)
    K, V = 6, 4
    q = rng.standard_normal((1, 1, 1, K))
    k = rng.standard_normal((1, 1, 1, K))
    v = rng.standard_normal((1, 1, 1, V))
    out, Sf = orc.kda_recurrence(q, k, v, np.zeros((1, 1, 1, K)), np.ones((1, 1, 1)), 0.5)
    _close(Sf[0, 0], np.outer(k[0, 0, 0], v[0, 0, 0]), 1e-14, "one-token state")
    _close(out[0, 0, 0], 0.5 * np.dot(q[0, 0, 0], k[0, 0, 0]) * v[0, 0, 0], 1e-14,
           "one-token output")


def pin_delta_retrieval(orc):
    """beta=1, ||k_t||=1, any decay and state: S_t^T k_t = v_t after the step."""
    rng = np.random.default_rng(RNG_SEED + 3)
    K, V = 8, 5
    for T in (1, 3, 7):
        q, k, v, la, _ = random_problem(rng, 1, T, 1, K, V)
        S0 = rng.standard_normal((1, 1, K, V))
        _, Sf = orc.kda_recurrence(q, k, v, la, np.ones((1, T, 1)), 1.0, initial_state=S0)
        _close(Sf[0, 0].T @ k[0, -1, 0], v[0, -1, 0], 1e-12, "delta-rule retrieval")


def pin_pure_decay(orc):
    """beta=0: S_t = Diag(prod_{u<=t} alpha_u) S0 and o_t = scale S_t^T q_t (decay on K rows)."""
    rng = np.random.default_rng(RNG_SEED + 4)
    K, V, T = 6, 4, 5
    q, k, v, la, _ = random_problem(rng, 1, T, 1, K, V, lb=-1.0)
    S0 = rng.standard_normal((1, 1, K, V))
    out, Sf = orc.kda_recurrence(q, k, v, la, np.zeros((1, T, 1)), 0.9, initial_state=S0)
    cum = np.cumsum(la[0, :, 0], axis=0)             # [T, K]
    for t in range(T):
        St = np.exp(cum[t])[:, None] * S0[0, 0]
        _close(out[0, t, 0], 0.9 * St.T @ q[0, t, 0], 1e-13, "pure-decay output")
    _close(Sf[0, 0], np.exp(cum[-1])[:, None] * S0[0, 0], 1e-13, "pure-decay state")


def pin_causal_linear_attention(orc):
    """Orthonormal keys, beta=1, alpha=1, S0=0: O = scale (M o Q K^T) V, M inclusive-causal."""
    rng = np.random.default_rng(RNG_SEED + 5)
    K, V, T = 8, 3, 6
    basis = np.linalg.qr(rng.standard_normal((K, K)))[0]
    k = basis[:T][None, :, None, :]                   # T distinct orthonormal keys
    q = rng.standard_normal((1, T, 1, K))
    v = rng.standard_normal((1, T, 1, V))
    out, Sf = orc.kda_recurrence(q, k, v, np.zeros((1, T, 1, K)), np.ones((1, T, 1)), 0.25)
    Q, Kc, Vc = q[0, :, 0], k[0, :, 0], v[0, :, 0]
    ref = 0.25 * (np.tril(np.ones((T, T))) * (Q @ Kc.T)) @ Vc
    _close(out[0, :, 0], ref, 1e-13, "causal linear attention")
    _close(Sf[0, 0], Kc.T @ Vc, 1e-13, "linear-attention state")


def pin_no_write_keeps_state(orc):
    """beta=0 and alpha=1: the state never changes and o_t = scale S0^T q_t."""
    rng = np.random.default_rng(RNG_SEED + 6)
    K, V, T = 5, 4, 4
    q, k, v, _, _ = random_problem(rng, 1, T, 1, K, V)
    S0 = rng.standard_normal((1, 1, K, V))
    out, Sf = orc.kda_recurrence(q, k, v, np.zeros((1, T, 1, K)), np.zeros((1, T, 1)), 2.0,
                                 initial_state=S0)
    _close(out[0, :, 0], 2.0 * q[0, :, 0] @ S0[0, 0], 1e-13, "no-write output")
    _close(Sf[0, 0], S0[0, 0], 0.0, "no-write state")


def pin_gate(orc):
    """Gate values: midpoint lb/2 at g = -dt_bias, limits lb and 0, point symmetry, monotone."""
    H, K, lb = 3, 7, -5.0
    rng = np.random.default_rng(RNG_SEED + 7)
    A_log = rng.uniform(0, np.log(16), H)
    dtb = 0.1 * rng.standard_normal((H, K))
    mid = orc.kda_gate(-dtb[None], A_log, dtb, lb)
    _close(mid, np.full((1, H, K), lb / 2), 1e-15, "gate midpoint")
    big = orc.kda_gate(np.full((1, H, K), 1e6), A_log, dtb, lb)
    small = orc.kda_gate(np.full((1, H, K), -1e6), A_log, dtb, lb)
    _close(big, np.full((1, H, K), lb), 0.0, "gate upper limit")
    _close(small, np.zeros((1, H, K)), 0.0, "gate lower limit")
    x = rng.standard_normal((4, H, K))
    gp = orc.kda_gate(-dtb + x, A_log, dtb, lb)
    gm = orc.kda_gate(-dtb - x, A_log, dtb, lb)
    _close(gp + gm, np.full_like(gp, lb), 1e-14, "gate point symmetry")
    grid = np.linspace(-3, 3, 61)[:, None, None] + np.zeros((1, H, K))
    gg = orc.kda_gate(grid, A_log, dtb, lb)
    assert np.all(np.diff(gg, axis=0) < 0), "gate must decrease strictly in g (lb < 0)"
    assert np.all((gg > lb) & (gg < 0)), "gate must lie strictly inside (lb, 0)"
    # the slope at the midpoint is lb * exp(A_log) / 4 (derivative of sigmoid at 0 is 1/4)
    eps = 1e-6
    d = (orc.kda_gate(-dtb[None] + eps, A_log, dtb, lb)
         - orc.kda_gate(-dtb[None] - eps, A_log, dtb, lb)) / (2 * eps)
    _close(d, (lb * np.exp(A_log)[:, None] / 4)[None], 1e-6, "gate midpoint slope")


def pin_fwd_composition(orc):
    """kda_fwd == kda_recurrence(kda_gate(g), sigmoid(beta_logits))."""
    rng = np.random.default_rng(RNG_SEED + 8)
    B, T, H, K, V = 2, 19, 2, 8, 6
    q, k, v, _, _ = random_problem(rng, B, T, H, K, V)
    g = rng.standard_normal((B, T, H, K))
    bl = rng.standard_normal((B, T, H))
    A_log = rng.uniform(0, np.log(16), H)
    dtb = 0.1 * rng.standard_normal((H, K))
    S0 = rng.standard_normal((B, H, K, V))
    o1, S1 = orc.kda_fwd(q, k, v, g, bl, 0.3, A_log, dtb, -5.0, initial_state=S0)
    la = orc.kda_gate(g, A_log, dtb, -5.0)
    o2, S2 = orc.kda_recurrence(q, k, v, la, expit(bl), 0.3, initial_state=S0)
    _close(o1, o2, 1e-15, "fwd composition out")
    _close(S1, S2, 1e-15, "fwd composition state")


def pin_state_carry(orc):
    """Two calls with the final state fed back equal one call."""
    rng = np.random.default_rng(RNG_SEED + 9)
    T, H, K, V = 37, 2, 8, 8
    q, k, v, la, beta = random_problem(rng, 1, T, H, K, V)
    S0 = rng.standard_normal((1, H, K, V))
    o, S = orc.kda_recurrence(q, k, v, la, beta, 0.5, initial_state=S0)
    cut = 20
    o1, S1 = orc.kda_recurrence(q[:, :cut], k[:, :cut], v[:, :cut], la[:, :cut], beta[:, :cut],
                                0.5, initial_state=S0)
    o2, S2 = orc.kda_recurrence(q[:, cut:], k[:, cut:], v[:, cut:], la[:, cut:], beta[:, cut:],
                                0.5, initial_state=S1)
    _close(np.concatenate([o1, o2], axis=1), o, 1e-12, "state carry out")
    _close(S2, S, 1e-12, "state carry state")


def pin_varlen_independence(orc):
    """A packed varlen call equals independent per-sequence calls, bit for bit."""
    rng = np.random.default_rng(RNG_SEED + 10)
    lens = [5, 1, 17, 0, 9]
    T, H, K, V = sum(lens), 2, 6, 4
    q, k, v, la, beta = random_problem(rng, 1, T, H, K, V)
    N = len(lens)
    S0 = rng.standard_normal((N, H, K, V))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, S = orc.kda_recurrence(q, k, v, la, beta, 0.8, initial_state=S0, cu_seqlens=cu)
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        if b > a:
            on, Sn = orc.kda_recurrence(q[:, a:b], k[:, a:b], v[:, a:b], la[:, a:b],
                                        beta[:, a:b], 0.8, initial_state=S0[n:n + 1])
            assert np.array_equal(o[:, a:b], on), "varlen output differs from single run"
            assert np.array_equal(S[n], Sn[0]), "varlen state differs from single run"
        else:
            assert np.array_equal(S[n], S0[n]), "empty sequence must pass its state through"


def pin_linearity(orc):
    """With S0=0: out is linear in V, homogeneous in scale, equivariant to V permutations."""
    rng = np.random.default_rng(RNG_SEED + 11)
    T, H, K, V = 21, 1, 6, 5
    q, k, v, la, beta = random_problem(rng, 1, T, H, K, V)
    v2 = rng.standard_normal(v.shape)
    o1, _ = orc.kda_recurrence(q, k, v, la, beta, 1.0)
    o2, _ = orc.kda_recurrence(q, k, v2, la, beta, 1.0)
    o3, _ = orc.kda_recurrence(q, k, 2.0 * v - 3.0 * v2, la, beta, 1.0)
    _close(o3, 2.0 * o1 - 3.0 * o2, 1e-12, "linearity in v")
    o4, _ = orc.kda_recurrence(q, k, v, la, beta, 0.125)
    _close(o4, 0.125 * o1, 1e-15, "homogeneity in scale")
    perm = rng.permutation(V)
    o5, _ = orc.kda_recurrence(q, k, v[..., perm], la, beta, 1.0)
    _close(o5, o1[..., perm], 1e-15, "V-column equivariance")


def pin_heads_subset(orc):
    """Evaluating a subset of heads gives the same numbers as evaluating all heads."""
    rng = np.random.default_rng(RNG_SEED + 12)
    q, k, v, la, beta = random_problem(rng, 1, 11, 4, 6, 4)
    o, S = orc.kda_recurrence(q, k, v, la, beta, 1.0)
    os_, Ss = orc.kda_recurrence(q, k, v, la, beta, 1.0, heads=[3, 1])
    assert np.array_equal(os_[:, :, [3, 1]], o[:, :, [3, 1]])
    assert np.array_equal(Ss[:, [3, 1]], S[:, [3, 1]])
    assert np.all(np.isnan(os_[:, :, [0, 2]]))


ALL_PINS = [pin_chunked_form, pin_matrix_form, pin_one_token_write, pin_delta_retrieval,
            pin_pure_decay, pin_causal_linear_attention, pin_no_write_keeps_state, pin_gate,
            pin_fwd_composition, pin_state_carry, pin_varlen_independence, pin_linearity,
            pin_heads_subset]
