"""Plant plausible mistakes in copies of the oracle and check that the pins catch each.

Every mutant is a textual edit of ``oracle/kda_oracle.c`` compiled to a
temporary library on the CPU; the real oracle is never modified.
"""
import os

import pytest

import oracle
import oracle_pins as P

MUTANTS = {
    "delta_sign": ("p[j] = b * (vt[j] - p[j]);", "p[j] = b * (vt[j] + p[j]);"),
    "decay_on_value_axis": ("S[(long)c * V + j] *= a[c];", "S[(long)c * V + j] *= a[j % K];"),
    "gate_missing_exp": ("oracle_sigmoid(exp(A_log) * (g + dt_bias))",
                         "oracle_sigmoid(A_log * (g + dt_bias))"),
    "gate_wrong_sign": ("oracle_sigmoid(exp(A_log) * (g + dt_bias))",
                        "oracle_sigmoid(exp(A_log) * (g - dt_bias))"),
    "beta_no_sigmoid": ("b = oracle_sigmoid(J->beta[t * H + h]);", "b = J->beta[t * H + h];"),
    "scale_dropped": ("ot[j] *= J->scale;", "ot[j] *= 1.0;"),
    "retrieval_uses_q": ("p[j] += S[(long)c * V + j] * kt[c];",
                         "p[j] += S[(long)c * V + j] * qt[c];"),
    "output_transposed_state": ("ot[j] += S[(long)c * V + j] * qt[c];",
                                "ot[j] += S[(long)j * V + c] * qt[c];"),
    "write_uses_q": ("S[(long)c * V + j] += kt[c] * p[j];", "S[(long)c * V + j] += qt[c] * p[j];"),
    "decay_after_retrieval": (
        "        /* p = S'^T k */",
        "        for (int c = 0; c < K; ++c)\n"
        "            for (int j = 0; j < V; ++j) S[(long)c * V + j] /= a[c];\n"
        "        /* p = S'^T k */"),
    "initial_state_ignored": ("if (J->S0)\n        memcpy", "if (0)\n        memcpy"),
    "output_before_update": ("/* o_t = scale * S^T q */\n        double* ot = J->out + rv;",
                             "/* o_t = scale * S^T q */\n        double* ot = J->out + rv;\n"
                             "        for (int c = 0; c < K; ++c)\n"
                             "            for (int j = 0; j < V; ++j) S[(long)c * V + j] -= kt[c] * p[j];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation target for {name} not found in the oracle source"
    mutated = src.replace(old, new, 1)
    cpath = os.path.join(tmp_path, f"mut_{name}.c")
    with open(cpath, "w") as f:
        f.write(mutated)
    lib = oracle.build(force=True, src=cpath, out=os.path.join(tmp_path, f"mut_{name}.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
