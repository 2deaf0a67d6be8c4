"""Pins of the backward oracle (``oracle.kda_bwd``, plain C in fp64) against things other
than itself:

* central finite differences of the forward oracle ``oracle.kda_fwd`` (a separate
  program) along random directions of every input, and element by element on a few
  entries;
* PyTorch autograd through a token recurrence written here, independently, in fp64.

The loss is L = sum(dout * out) + sum(dfinal * final_state).
"""
import numpy as np
import pytest

import oracle
import synth


def _inputs(K, V, lengths, H=2, seed=0, lower_bound=-5.0):
    T = sum(lengths)
    d = synth.make_inputs(1, T, H, K=K, V=V, seed=seed, lengths=lengths, init_dtype="f32",
                          lower_bound=lower_bound)
    f = {n: oracle.bf16_bits_to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")}
    f.update(A_log=d["A_log"].astype(np.float64), dt_bias=d["dt_bias"].astype(np.float64),
             initial_state=d["initial_state"].astype(np.float64), scale=d["scale"],
             lower_bound=d["lower_bound"], cu_seqlens=d["cu_seqlens"])
    rng = np.random.default_rng(seed + 1)
    f["dout"] = rng.standard_normal(f["v"].shape)
    f["dfinal"] = rng.standard_normal(f["initial_state"].shape)
    return f


def _loss(f):
    out, S = oracle.kda_fwd(f["q"], f["k"], f["v"], f["g"], f["beta"], f["scale"], f["A_log"],
                            f["dt_bias"], f["lower_bound"], initial_state=f["initial_state"],
                            cu_seqlens=f["cu_seqlens"])
    return float(np.sum(f["dout"] * out) + np.sum(f["dfinal"] * S))


def _grads(f):
    return oracle.kda_bwd(f["q"], f["k"], f["v"], f["g"], f["beta"], f["scale"], f["A_log"],
                          f["dt_bias"], f["lower_bound"], f["dout"],
                          initial_state=f["initial_state"], dfinal=f["dfinal"],
                          cu_seqlens=f["cu_seqlens"])


GRAD_OF = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "A_log": "dA_log",
           "dt_bias": "ddt_bias", "initial_state": "d_initial_state"}


@pytest.mark.parametrize("K,V,lengths", [(8, 8, [5, 0, 23]), (8, 4, [1, 17]), (128, 128, [9])])
def test_directional_derivatives_match_finite_differences(K, V, lengths):
    f = _inputs(K, V, lengths)
    g = _grads(f)
    rng = np.random.default_rng(7)
    eps = 1e-6
    for name, gname in GRAD_OF.items():
        D = rng.standard_normal(np.shape(f[name]))
        fp, fm = dict(f), dict(f)
        fp[name] = f[name] + eps * D
        fm[name] = f[name] - eps * D
        fd = (_loss(fp) - _loss(fm)) / (2 * eps)
        an = float(np.sum(g[gname] * D))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_single_entries_match_finite_differences():
    f = _inputs(6, 5, [4, 11], seed=3)
    g = _grads(f)
    rng = np.random.default_rng(11)
    eps = 1e-6
    for name, gname in GRAD_OF.items():
        for _ in range(3):
            idx = tuple(int(rng.integers(s)) for s in np.shape(f[name]))
            fp, fm = dict(f), dict(f)
            fp[name] = f[name].copy()
            fm[name] = f[name].copy()
            fp[name][idx] += eps
            fm[name][idx] -= eps
            fd = (_loss(fp) - _loss(fm)) / (2 * eps)
            assert abs(fd - g[gname][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, g[gname][idx])


def test_equals_autograd_of_an_independent_recurrence():
    torch = pytest.importorskip("torch")
    f = _inputs(6, 5, [7, 3], seed=5, lower_bound=-2.0)
    t = {n: torch.tensor(f[n], dtype=torch.float64, requires_grad=True)
         for n in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state")}
    cu = f["cu_seqlens"]
    H = t["q"].shape[2]
    total = torch.zeros((), dtype=torch.float64)
    dout = torch.tensor(f["dout"])
    dfinal = torch.tensor(f["dfinal"])
    for n in range(len(cu) - 1):
        for h in range(H):
            S = t["initial_state"][n, h]
            for s in range(int(cu[n]), int(cu[n + 1])):
                x = torch.exp(t["A_log"][h]) * (t["g"][0, s, h] + t["dt_bias"][h])
                alpha = torch.exp(f["lower_bound"] * torch.sigmoid(x))
                b = torch.sigmoid(t["beta"][0, s, h])
                k = t["k"][0, s, h]
                # (I - b k k^T) Diag(alpha) S + b k v^T, written as one matrix product
                M = (torch.eye(k.shape[0], dtype=torch.float64) - b * torch.outer(k, k)) @ torch.diag(alpha)
                S = M @ S + b * torch.outer(k, t["v"][0, s, h])
                o = f["scale"] * (S.T @ t["q"][0, s, h])
                total = total + torch.sum(dout[0, s, h] * o)
            total = total + torch.sum(dfinal[n, h] * S)
    total.backward()
    g = _grads(f)
    for name, gname in GRAD_OF.items():
        ref = t[name].grad.numpy()
        assert np.allclose(g[gname], ref, rtol=1e-10, atol=1e-12), name


def test_no_final_gradient_and_empty_sequences():
    """Without dfinal the final-state term is absent; an empty sequence passes its state
    gradient straight through (here: zero) and leaves its tokens out."""
    f = _inputs(8, 8, [0, 6, 0], seed=9)
    f["dfinal"] = np.zeros_like(f["dfinal"])
    g1 = _grads(f)
    g2 = oracle.kda_bwd(f["q"], f["k"], f["v"], f["g"], f["beta"], f["scale"], f["A_log"],
                        f["dt_bias"], f["lower_bound"], f["dout"], initial_state=f["initial_state"],
                        cu_seqlens=f["cu_seqlens"])
    for name in g1:
        assert np.array_equal(g1[name], g2[name]), name
    assert np.all(g1["d_initial_state"][0] == 0) and np.all(g1["d_initial_state"][2] == 0)
