"""Writes tests/golden/oracle_small.json. Calls only the oracle and the seeded
input generator; never the CUDA path.

The FLARE++ pages print no worked example with numbers, so this fixture is a
regression pin: it freezes (1) a few values of each seeded input tensor, so the
generator gives the same workload on every host, and (2) the fp64 oracle's
outputs on one small case (B=1, H=2, N=24, M=4, D=8, i.i.d. inputs, seed 77),
so a later change to the oracle's arithmetic shows up as a diff that its commit
has to justify.

Run from the repository root: python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from rank_latent_routing_gb300 import workloads  # noqa: E402

CASE = dict(B=1, H=2, N=24, M=4, D=8, dtype="fp32", structure="iid", seed=77)


def build():
    s = workloads.Shape(CASE["B"], CASE["H"], CASE["N"], CASE["M"], CASE["D"])
    wl = workloads.make(s, CASE["dtype"], CASE["structure"], CASE["seed"])
    res = oracle.forward(wl.K, wl.V, wl.Ks_raw, wl.Qseed, wl.Qf, wl.gate)
    return {
        "what": "oracle regression fixture; no printed example exists in the FLARE++ pages",
        "case": CASE,
        "inputs_head": {k: getattr(wl, k).reshape(-1)[:6].astype(float).tolist()
                        for k in ("K", "V", "Ks_raw", "Qseed", "Qf", "gate")},
        "outputs": {k: res[k].reshape(-1).tolist() for k in ("Qd", "Q", "Z", "L", "Y")},
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(build(), f, indent=1)
        f.write("\n")
