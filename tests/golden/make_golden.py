"""Writes tests/golden/tiny_regression.json from the fp64 oracle (and nothing else).

The fixture is a regression guard: it freezes the oracle's output on one tiny, fixed
problem so that any later change to the oracle's arithmetic shows up as a failing test
(and must then be justified by the passage of the pages it follows).

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))


def tiny_case():
    """B=1, T=6, H=2, dk=4, dv=3 with fixed, hand-picked-by-seed inputs."""
    rng = np.random.default_rng(20240601)
    B, T, H, dk, dv = 1, 6, 2, 4, 3
    return dict(q=rng.normal(size=(B, T, H, dk)), k=rng.normal(size=(B, T, H, dk)),
                v=rng.normal(size=(B, T, H, dv)), g=rng.normal(size=(B, T, H, dk)),
                beta_logits=rng.normal(size=(B, T, H)), a_log=rng.uniform(-1, 1, H),
                dt_bias=rng.normal(0, 0.1, (dk, H)), scale=0.5, lower_bound=-2.0,
                initial_state=rng.normal(0, 0.3, (B, H, dk, dv)))


def main():
    from oracle import kda_forward
    out, S = kda_forward(**tiny_case())
    with open(os.path.join(HERE, "tiny_regression.json"), "w") as f:
        json.dump({"written_by": "tests/golden/make_golden.py (oracle only)",
                   "out": out.tolist(), "final_state": S.tolist()}, f, indent=1)


if __name__ == "__main__":
    main()
