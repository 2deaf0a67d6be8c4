"""Write the oracle's numbers for the tiny workload to ``tiny_t64_h1.txt``.

Calls only the oracle (and the seeded input generator).  The fixture freezes
the oracle's result so that any later change to the oracle's arithmetic, or
to the input generator, shows up as a diff that its commit must justify.
Run:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_t64_h1.txt")
# fixed sample positions: (t, v) for out, (c, v) for the final state
OUT_POS = [(t, v) for t in (0, 1, 15, 16, 17, 31, 47, 63) for v in (0, 5, 77, 127)]
STATE_POS = [(c, v) for c in (0, 3, 64, 127) for v in (0, 9, 100, 127)]


def compute():
    d = synth.make_workload("tiny_t64_h1")
    out, S = oracle.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["A_log"],
                            d["dt_bias"], d["lower_bound"], n_threads=1)
    return out[0, :, 0, :], S[0, 0]


def main():
    out, S = compute()
    lines = ["# oracle (fp64) on workload tiny_t64_h1, seed 0; written by make_golden.py",
             f"out_rms {np.sqrt(np.mean(out ** 2)):.17e}",
             f"state_fro {np.linalg.norm(S):.17e}"]
    lines += [f"out {t} {v} {out[t, v]:.17e}" for t, v in OUT_POS]
    lines += [f"state {c} {v} {S[c, v]:.17e}" for c, v in STATE_POS]
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
