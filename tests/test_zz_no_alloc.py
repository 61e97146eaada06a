"""lbx_verify_step_noalloc, the verify step for callers that cannot allocate
device memory (an engine that has reserved all of it for its caches and allows
no later cudaMalloc, or a plugin inside a framework that owns the allocator):
it must give the same results as lbx_verify_step with a caller workspace, on
two calls in a row (the fixed counter array is reused between calls).

Kept in its own file, collected last, so that a run stopping at its first
failure has already run every other test.  Passes alone in a fresh process
and after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

from tree_verify_linear_gb300 import lbx
import oracle
from tree_verify_linear_gb300.inputs import WORKLOADS, Workload, make_inputs

from gpu_util import O_TOL, STATE_TOL, dev_inputs, o_error, state_rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from tree_verify_linear_gb300 import build
    build.build()
    lbx.load()
    oracle.lib()


def _two_calls(w, inp, noalloc: bool):
    d = dev_inputs(inp)
    cfg = lbx.cfg_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = None if noalloc else lbx.new_workspace(cfg)
    outs = []
    for _ in range(2):
        o = torch.full((w.L, w.Bq, w.N, w.Hv, w.d), float("nan"), device="cuda")
        args = (cfg, d["x"], d["conv_w"], d["a"], d["b"], d["parent"], d["slot"], d["accepted"],
                d["state"], d["conv_cache"], o)
        if noalloc:
            lbx.lbx_verify_step_noalloc(*args, d_status=status)
        else:
            lbx.lbx_verify_step(*args, ws, d_status=status)
        torch.cuda.synchronize()
        outs.append((o.cpu().numpy(), d["state"].cpu().numpy(), d["conv_cache"].cpu().numpy()))
    assert int(status.item()) == 0
    return outs


NOALLOC_CASES = {
    "tiny": WORKLOADS["tiny"],
    "serve27b_b22_l4": WORKLOADS["serve27b_b22"].replace(L=4),
    # small enough that the tensor-core step's records fit the fixed array:
    # the tensor-core kernels run with the array as their workspace
    "tc_small": Workload("tc_small", L=1, Bq=1, N=8, Hk=1, Hv=2, d=128, seed=3100),
}


@pytest.mark.parametrize("name", sorted(NOALLOC_CASES))
def test_noalloc_matches_workspace_entry_point_on_two_calls(name):
    w = NOALLOC_CASES[name]
    inp = make_inputs(w)
    ref = _two_calls(w, inp, noalloc=False)
    got = _two_calls(w, inp, noalloc=True)
    for (o_r, s_r, c_r), (o_g, s_g, c_g) in zip(ref, got):
        assert o_error(o_g, o_r.astype(np.float64)) <= O_TOL
        for l in range(w.L):
            for b in range(w.Bq):
                s = inp["slot"][b]
                for h in range(w.Hv):
                    assert state_rel(s_g[l, s, h], s_r[l, s, h].astype(np.float64)) <= STATE_TOL
        assert c_g.tobytes() == c_r.tobytes()
        assert s_g[:, w.Bq:].tobytes() == s_r[:, w.Bq:].tobytes()  # canary slots untouched


def test_noalloc_tensor_core_path_matches_oracle_on_two_calls():
    """The tensor-core case against the fp64 oracle: the first call from the
    seeded caches, the second from the caches the first one persisted."""
    w = NOALLOC_CASES["tc_small"]
    lib = lbx.load()
    cfg = lbx.cfg_of(w)
    # the configuration's tensor-core workspace fits the fixed array
    assert 0 < lib.lbx_workspace_size(ctypes.byref(cfg)) <= 4 * lbx.LBX_NOALLOC_MAX_GROUPS
    inp = make_inputs(w)
    got = _two_calls(w, inp, noalloc=True)
    o_ref, s_ref, c_ref = oracle.verify_step_full(w, inp)
    o1, s1, c1 = got[0]
    assert o_error(o1, o_ref) <= O_TOL
    for h in range(w.Hv):
        assert state_rel(s1[0, inp["slot"][0], h], s_ref[0, inp["slot"][0], h]) <= STATE_TOL
    assert c1.tobytes() == c_ref.tobytes()
    inp2 = dict(inp)
    inp2["state"] = s_ref.astype(np.float32)
    inp2["conv_cache"] = c_ref
    o_ref2, s_ref2, c_ref2 = oracle.verify_step_full(w, inp2)
    o2, s2, c2 = got[1]
    assert o_error(o2, o_ref2) <= O_TOL
    for h in range(w.Hv):
        assert state_rel(s2[0, inp["slot"][0], h], s_ref2[0, inp["slot"][0], h]) <= STATE_TOL
    assert c2.tobytes() == c_ref2.tobytes()


@pytest.mark.parametrize("name", ["tiny", "tc_small"])
def test_noalloc_calls_leave_free_device_memory_unchanged(name):
    """After a first call (which may load the library's kernels onto the
    device), further calls take no device memory."""
    w = NOALLOC_CASES[name]
    inp = make_inputs(w)
    d = dev_inputs(inp)
    cfg = lbx.cfg_of(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.empty((w.L, w.Bq, w.N, w.Hv, w.d), device="cuda")
    args = (cfg, d["x"], d["conv_w"], d["a"], d["b"], d["parent"], d["slot"], d["accepted"],
            d["state"], d["conv_cache"], o)
    lbx.lbx_verify_step_noalloc(*args, d_status=status)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        lbx.lbx_verify_step_noalloc(*args, d_status=status)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert int(status.item()) == 0
    assert free1 == free0, (free0, free1)


def test_noalloc_rejects_configs_over_its_capacity():
    lib = lbx.load()
    groups = lbx.LBX_NOALLOC_MAX_GROUPS
    cfg = lbx.make_cfg(L=groups // 16 + 1, Bq=1, N=22, Hk=16, Hv=48, d=128, K=4, n_slots=1)
    fake = ctypes.c_void_p(1 << 20)  # rejected before any pointer is used
    rc = lib.lbx_verify_step_noalloc(ctypes.byref(cfg), *([fake] * 10), None, None)
    assert rc == lbx.LBX_EINVAL
