"""Writes tests/golden/oracle_tiny.json: a tiny regression fixture of the FP64 oracle.

The pages print no worked example, so this fixture is not a pin from the pages:
it freezes the oracle's own output on one tiny seeded case (calls only
``oracle`` and the seeded input generator) so that an accidental change to the
oracle's arithmetic shows up as a diff. Regenerate only with a commit message
that names the passage or reading that justifies the change.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from bwd_tri_attn_gb300.workloads import make_inputs  # noqa: E402

CASE = dict(B=1, S=2, N=4, H=1, d=2, seed=123, mask=("tail", 1))


def compute():
    x = make_inputs(CASE["B"], CASE["S"], CASE["N"], CASE["H"], CASE["d"], CASE["seed"], mask=CASE["mask"])
    O, LSE = oracle.fwd(x["Q"], x["K"], x["V"], x["bias"], x["mask"])
    g = oracle.bwd(x["Q"], x["K"], x["V"], x["bias"], x["mask"], x["dO"])
    return {"O": O.tolist(), "LSE": LSE.tolist(), **{k: g[k].tolist() for k in ("dQ", "dK", "dV", "dBias", "D")}}


if __name__ == "__main__":
    out = {"case": {**CASE, "mask": list(CASE["mask"])},
           "source": "FP64 oracle (regression fixture; the pages print no worked example)",
           "values": compute()}
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as f:
        json.dump(out, f, indent=1)
