"""Write the oracle regression fixtures in this folder.

The pages describing the method print no worked example for the tree ops
(Lucebox hub README, section "02 DFlash DDtree", names the three tree-aware
state-rollback kernels but gives no numbers for them), so these fixtures are
not values from the pages: they are the oracle's own outputs on the seeded
tiny workload, kept to catch unintended changes to the oracle.  This script
calls only ``oracle`` and the seeded input generator.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from tree_verify_linear_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402


def main():
    w = WORKLOADS["tiny"]
    inp = make_inputs(w)
    o, state, cache = oracle.verify_step_full(w, inp)
    s = int(inp["slot"][0])
    out = {
        "what": "fp64 oracle on the seeded tiny workload (1 layer, Hk=2, Hv=4, d=32, K=4, "
                "8-node uniform tree); regression fixture written by make_golden.py",
        "workload": "tiny",
        "seed": w.seed,
        "parent": inp["parent"][0].tolist(),
        "accepted": int(inp["accepted"][0]),
        "o_head0": [[float(v) for v in row] for row in o[0, 0, :, 0, :]],
        "o_abs_max": float(np.abs(o).max()),
        "state_row0_per_head": [[float(v) for v in state[0, s, h, 0, :]] for h in range(w.Hv)],
        "state_fro_per_head": [float(np.linalg.norm(state[0, s, h])) for h in range(w.Hv)],
        "conv_cache_new_bits_row_sums": [int(cache[0, s, r].view(np.uint32).astype(np.uint64).sum())
                                         for r in range(w.K - 1)],
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
