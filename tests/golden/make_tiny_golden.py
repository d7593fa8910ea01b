"""Write tests/golden/tiny_decode.json: the oracle's outputs on the tiny decode
workload (B=2, Hk=2, Hv=4, dk=dv=32, 8 steps, fp32 state and inputs, seed 0).

The file is a regression fixture for the oracle itself: it is written only by
this script, which calls only oracle/ and the seeded workload generator, and
it lets a test notice any later change to the oracle's arithmetic.
Run from the repository root:  python tests/golden/make_tiny_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from hybrid_ssm_gated_gb300 import workload as wl  # noqa: E402


def compute():
    w = wl.WORKLOADS["tiny"]
    pool = wl.initial_pool(w)
    A_log, dt_bias = wl.head_params(w)
    slots = wl.slots(w)
    outs = []
    for t in range(w.steps):
        x = wl.step_inputs(w, t)
        o, bad = oracle.decode_step(pool, w.state_dtype, slots, x["q"], x["k"], x["v"], x["a"], x["b"],
                                    w.in_dtype, A_log, dt_bias)
        assert bad == 0
        outs.append(o)
    return np.array(outs), pool


def main():
    outs, pool = compute()
    doc = {
        "what": "oracle outputs of the tiny GDN decode workload; regression fixture for the oracle",
        "workload": "tiny: B=2, Hk=2, Hv=4, dk=dv=32, 8 steps, fp32 state/inputs, seed 0",
        "writer": "tests/golden/make_tiny_golden.py (calls only oracle/ and the workload generator)",
        "out_step0_b0_h0": outs[0, 0, 0].tolist(),
        "out_step7_b1_h3": outs[7, 1, 3].tolist(),
        "final_state_slot1_h2_col5": pool[1, 2, 5].astype(np.float64).tolist(),
        "sum_abs_out": float(np.abs(outs).sum()),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_decode.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
