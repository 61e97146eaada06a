"""The oracle still reproduces its committed regression fixture (tiny workload).

The fixture is written by tests/golden/make_golden.py, which calls only the
oracle; it guards against unintended changes to the oracle's arithmetic.
"""
import json
import os

import numpy as np

import oracle
from tree_verify_linear_gb300.inputs import WORKLOADS, make_inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_committed_tiny_fixture():
    with open(os.path.join(HERE, "golden", "tiny_oracle.json")) as f:
        g = json.load(f)
    w = WORKLOADS["tiny"]
    inp = make_inputs(w)
    assert inp["parent"][0].tolist() == g["parent"]
    assert int(inp["accepted"][0]) == g["accepted"]
    o, state, cache = oracle.verify_step_full(w, inp)
    s = int(inp["slot"][0])
    np.testing.assert_allclose(o[0, 0, :, 0, :], np.array(g["o_head0"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.abs(o).max(), g["o_abs_max"], rtol=1e-12)
    for h in range(w.Hv):
        np.testing.assert_allclose(state[0, s, h, 0, :], g["state_row0_per_head"][h], rtol=0,
                                   atol=1e-12)
        np.testing.assert_allclose(np.linalg.norm(state[0, s, h]), g["state_fro_per_head"][h],
                                   rtol=1e-12)
    sums = [int(cache[0, s, r].view(np.uint32).astype(np.uint64).sum()) for r in range(w.K - 1)]
    assert sums == g["conv_cache_new_bits_row_sums"]
