"""GPU parity of the fused verify step (lbx_verify_step) against the fp64
oracle, on the seeded workloads at full size and on edge cases.  Calls go
through the C ABI (ctypes binding)."""
import numpy as np
import pytest
import torch

import oracle
from tree_verify_linear_gb300 import lbx
from tree_verify_linear_gb300.inputs import WORKLOADS, Workload, bf16_bits, make_inputs

from gpu_util import (O_TOL, STATE_TOL, check_verify, counters_cleared, dev_inputs,
                      run_verify)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from tree_verify_linear_gb300 import build
    build.build()
    lbx.load()
    oracle.lib()


def test_tiny_all_heads():
    w = WORKLOADS["tiny"]
    inp = make_inputs(w)
    o, st, cc, status, ws = run_verify(w, inp)
    assert status == 0
    check_verify(w, inp, o, st, cc)
    assert not ws.any(), "workspace counters must be left at zero"


def test_layer27b_all_heads():
    w = WORKLOADS["layer27b"]
    inp = make_inputs(w)
    o, st, cc, status, _ = run_verify(w, inp)
    assert status == 0
    check_verify(w, inp, o, st, cc)


def test_step27b_all_heads_full_size():
    """The 48-layer budget-22 step, every head checked (the bench workload)."""
    w = WORKLOADS["step27b"]
    inp = make_inputs(w)
    o, st, cc, status, ws = run_verify(w, inp)
    assert status == 0
    assert np.isfinite(o).all()
    check_verify(w, inp, o, st, cc)
    assert counters_cleared(w, ws)


def test_serve27b_b22_all_heads_permuted_slots():
    w = WORKLOADS["serve27b_b22"]
    inp = make_inputs(w, slots=np.array([4, 0, 6, 2, 1], dtype=np.int32))
    o, st, cc, status, _ = run_verify(w, inp)
    assert status == 0
    check_verify(w, inp, o, st, cc)


def test_serve27b_b64_all_layers():
    """Budget 64, 5 requests, 48 layers: every (layer, request, head)."""
    w = WORKLOADS["serve27b_b64"]
    inp = make_inputs(w)
    o, st, cc, status, _ = run_verify(w, inp)
    assert status == 0
    assert np.isfinite(o).all()
    check_verify(w, inp, o, st, cc)


def test_chain08b_all_heads_chunked():
    """4096-token chain, 18 layers, chunked mode, against the sequential
    recurrence of the oracle on every (layer, head): all o and every
    persisted state."""
    w = WORKLOADS["chain08b"]
    inp = make_inputs(w)
    o, st, cc, status, _ = run_verify(w, inp, mode=lbx.LBX_MODE_CHUNKED)
    assert status == 0
    assert np.isfinite(o).all()
    check_verify(w, inp, o, st, cc, form=oracle.FORM_SEQUENTIAL)


def small(**kw):
    base = dict(name="edge", L=2, Bq=2, N=13, Hk=2, Hv=4, d=32, tree="uniform",
                accepted="node", seed=500)
    base.update(kw)
    return Workload(**base)


EDGE = {
    "root_only": small(N=1),
    "two_nodes": small(N=2),
    "ragged_13": small(N=13),
    "deep_uniform_64": small(N=64, seed=501),
    "ddtree_37_d128": small(N=37, Hk=2, Hv=6, d=128, tree="ddtree", seed=502),
    "d64": small(d=64, N=22, tree="ddtree", seed=503),
    "conv_k3": small(K=3, seed=504),
    "conv_k2": small(K=2, seed=505),
    "conv_k1": small(K=1, seed=506),
    "q_scale": small(q_scale=float(1 / np.sqrt(32)), seed=507),
    "gqa_1to1": small(Hk=4, Hv=4, seed=508),
    "three_requests": small(Bq=3, N=9, tree="ddtree", seed=509),
    "leaf_accepted": small(accepted="leaf", seed=510),
    "chain_tree_mode": small(N=64, tree="chain", accepted="last", seed=511),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(name):
    w = EDGE[name]
    slots = None
    if w.Bq == 3:
        slots = np.array([2, 0, 4], dtype=np.int32)
    inp = make_inputs(w, slots=slots)
    o, st, cc, status, ws = run_verify(w, inp, mode=lbx.LBX_MODE_TREE)
    assert status == 0
    check_verify(w, inp, o, st, cc)
    assert counters_cleared(w, ws, lbx.LBX_MODE_TREE)


@pytest.mark.parametrize("N,acc", [(64, 63), (100, 99), (100, 70), (130, 5), (7, 3)])
def test_chunked_chain_lengths(N, acc):
    """Chains processed in 64-token chunks, ragged last chunk, accepted node
    anywhere along the chain (its state is captured mid-chain)."""
    w = small(N=N, tree="chain", accepted="last", d=128, Hk=2, Hv=2, seed=600 + N)
    inp = make_inputs(w)
    inp["accepted"][:] = acc
    o, st, cc, status, _ = run_verify(w, inp, mode=lbx.LBX_MODE_CHUNKED)
    assert status == 0
    check_verify(w, inp, o, st, cc, form=oracle.FORM_SEQUENTIAL)


def _at_16_past_32(t: torch.Tensor) -> torch.Tensor:
    """A copy of t whose data starts 16 bytes past a 32-byte boundary: the
    weakest alignment the header allows for every array."""
    es = t.element_size()
    buf = torch.empty(t.numel() + 64 // es, dtype=t.dtype, device=t.device)
    k = next(k for k in range(64 // es) if (buf.data_ptr() + k * es) % 32 == 16)
    v = buf[k:k + t.numel()].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 32 == 16
    return v


@pytest.mark.parametrize("mode,kw", [
    (lbx.LBX_MODE_CHUNKED, dict(N=100, tree="chain", accepted="last", Hk=2, Hv=2)),
    (lbx.LBX_MODE_TREE, dict(N=22, Hk=2, Hv=4)),
    (lbx.LBX_MODE_TREE_CUDA_CORES, dict(N=22, Hk=2, Hv=4)),
])
def test_arrays_16_bytes_past_a_32_byte_boundary(mode, kw):
    """Every array 16-byte aligned but not 32-byte aligned (the header asks
    for 16): the chunked tensor-core path, the tree tensor-core path and the
    CUDA-core tree kernel give the same outputs, bit for bit, as with
    aligned arrays."""
    w = small(d=128, seed=3100 + mode, **kw)
    inp = make_inputs(w)
    ref = run_verify(w, inp, mode=mode)
    d = {k: _at_16_past_32(v) for k, v in dev_inputs(inp).items()}
    cfg = lbx.cfg_of(w, mode)
    o = _at_16_past_32(torch.full((w.L, w.Bq, w.N, w.Hv, w.d), float("nan"), device="cuda"))
    ws = lbx.new_workspace(cfg)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lbx.lbx_verify_step(cfg, d["x"], d["conv_w"], d["a"], d["b"], d["parent"], d["slot"],
                        d["accepted"], d["state"], d["conv_cache"], o, ws, status)
    torch.cuda.synchronize()
    assert ref[3] == 0 and int(status.item()) == 0
    assert o.cpu().numpy().tobytes() == ref[0].tobytes()
    assert d["state"].cpu().numpy().tobytes() == ref[1].tobytes()
    assert d["conv_cache"].cpu().numpy().tobytes() == ref[2].tobytes()


def test_tree_and_chunked_modes_agree_on_a_chain():
    w = small(N=64, tree="chain", accepted="last", d=128, Hk=2, Hv=4, seed=700)
    inp = make_inputs(w)
    o1, s1, c1, st1, _ = run_verify(w, inp, mode=lbx.LBX_MODE_TREE)
    o2, s2, c2, st2, _ = run_verify(w, inp, mode=lbx.LBX_MODE_CHUNKED)
    assert st1 == st2 == 0
    # chunked mode at d = 128 runs on tensor cores (bf16 hi/lo products),
    # tree mode at N = 64 on CUDA cores (fp32): the same bound as for the
    # two tree kernels
    assert np.abs(o1 - o2).max() <= 1e-4 * np.abs(o1).max()
    assert c1.tobytes() == c2.tobytes()
    used = inp["slot"]  # the other slots hold the canary pattern
    rel = np.linalg.norm((s1 - s2)[:, used].reshape(-1)) / np.linalg.norm(s1[:, used].reshape(-1))
    assert rel <= 1e-5


def test_identity_gates_keep_state_and_read_out_S0_q():
    """a = 1, b = 0: the persisted state equals the cached state and
    o_n = S0 q_n."""
    w = small(seed=800)
    inp = make_inputs(w)
    inp["a"][...] = bf16_bits(np.ones(inp["a"].shape, np.float32))
    inp["b"][...] = 0
    o, st, cc, status, _ = run_verify(w, inp)
    assert status == 0
    check_verify(w, inp, o, st, cc)
    for l in range(w.L):
        for b in range(w.Bq):
            s = inp["slot"][b]
            d = st[l, s].astype(np.float64) - inp["state"][l, s]
            assert np.abs(d).max() <= 1e-6 * np.abs(inp["state"][l, s]).max()


def test_two_consecutive_steps_match_oracle_twice():
    """The caches updated in place by one step feed the next; the same
    workspace serves both calls."""
    w = WORKLOADS["serve27b_b22"].replace(L=4)
    inp = make_inputs(w)
    o, st, cc, status, ws = run_verify(w, inp, steps=2)
    assert status == 0 and counters_cleared(w, ws)
    # oracle: two steps in sequence on the same inputs
    _, s1, c1 = oracle.verify_step_full(w, inp)
    inp2 = dict(inp)
    inp2["state"] = inp["state"].copy()
    for b in range(w.Bq):
        inp2["state"][:, inp["slot"][b]] = s1[:, inp["slot"][b]].astype(np.float32)
    inp2["conv_cache"] = c1
    check_verify(w, inp2, o, st, cc)


# -------------------------------------------------------------------------
# Errors the device detects: status is set and nothing is written.
# -------------------------------------------------------------------------
def _assert_untouched(inp, o, st, cc):
    assert st.tobytes() == inp["state"].tobytes()
    assert cc.tobytes() == inp["conv_cache"].tobytes()
    assert np.isnan(o).all()


@pytest.mark.parametrize("bad", ["root_parent", "forward_parent", "out_of_range"])
def test_invalid_tree_sets_status_and_writes_nothing(bad):
    w = small(seed=900)
    inp = make_inputs(w)
    if bad == "root_parent":
        inp["parent"][1, 0] = 0
    elif bad == "forward_parent":
        inp["parent"][0, 5] = 7
    else:
        inp["parent"][1, 3] = 99
    o, st, cc, status, ws = run_verify(w, inp)
    assert status == lbx.LBX_ETREE
    _assert_untouched(inp, o, st, cc)
    assert not ws.any()


def test_duplicate_slots_and_bad_accepted_rejected_on_device():
    w = small(seed=901)
    inp = make_inputs(w, slots=np.array([1, 1], dtype=np.int32))
    o, st, cc, status, _ = run_verify(w, inp)
    assert status == lbx.LBX_EINVAL
    _assert_untouched(inp, o, st, cc)
    inp = make_inputs(w)
    inp["accepted"][1] = w.N
    o, st, cc, status, _ = run_verify(w, inp)
    assert status == lbx.LBX_EINVAL
    _assert_untouched(inp, o, st, cc)
    inp = make_inputs(w)
    inp["slot"][0] = w.n_slots
    o, st, cc, status, _ = run_verify(w, inp)
    assert status == lbx.LBX_EINVAL


def test_chunked_mode_rejects_a_non_chain():
    w = small(N=80, tree="chain", accepted="last", seed=902)
    inp = make_inputs(w)
    inp["parent"][0, 40] = 10
    o, st, cc, status, _ = run_verify(w, inp, mode=lbx.LBX_MODE_CHUNKED)
    assert status == lbx.LBX_ETREE
    _assert_untouched(inp, o, st, cc)


# -------------------------------------------------------------------------
# Tensor-core kernel (d = 128, tree mode, N <= 64; node capacities 8, 16 and
# 24 at two CTAs per SM, 32 and 64 at one): shapes at its limits, and
# agreement with the CUDA-core kernel on the same inputs.
# -------------------------------------------------------------------------
def tc(**kw):
    base = dict(name="tc", L=2, Bq=2, N=22, Hk=2, Hv=6, d=128, tree="ddtree", accepted="node",
                seed=1100)
    base.update(kw)
    return Workload(**base)


TC_EDGE = {
    "n1": tc(N=1, seed=1101),
    "n2": tc(N=2, seed=1102),
    "n8": tc(N=8, seed=1103),
    "n9": tc(N=9, seed=1104),
    "n16": tc(N=16, tree="uniform", seed=1105),
    "n24_chain": tc(N=24, tree="chain", accepted="last", seed=1106),
    "n24_uniform": tc(N=24, tree="uniform", seed=1107),
    "g1": tc(Hk=3, Hv=3, seed=1108),
    "g4": tc(Hk=1, Hv=4, seed=1109),
    "three_requests": tc(Bq=3, N=13, seed=1110),
    "k2": tc(K=2, seed=1111),
    "k1": tc(K=1, seed=1112),
    "q_scale": tc(q_scale=float(1 / np.sqrt(128)), seed=1113),
    "leaf": tc(accepted="leaf", seed=1114),
    "many_tiles": tc(L=7, Bq=3, Hk=4, Hv=12, N=22, seed=1115),
    "n25": tc(N=25, seed=1116),
    "n32_uniform": tc(N=32, tree="uniform", seed=1117),
    "n33": tc(N=33, seed=1118),
    "n40_leaf": tc(N=40, accepted="leaf", seed=1119),
    "n64_chain": tc(N=64, tree="chain", accepted="last", seed=1120),
    "n64_uniform": tc(N=64, tree="uniform", seed=1121),
    "n64_ddtree_b4": tc(N=64, max_children=4, seed=1122),
    "n64_three_requests": tc(Bq=3, N=64, max_children=4, seed=1123),
    "n48_k2_g4": tc(N=48, K=2, Hk=1, Hv=4, tree="uniform", seed=1124),
    # node capacities 32 and 64 (16-warp step, prep with the new conv window
    # kept aside during the conv) at the other conv widths and with the
    # accepted node at the root (the new window is old cached rows + root)
    "n64_k3": tc(N=64, K=3, max_children=4, seed=1125),
    "n30_k1_g1": tc(N=30, K=1, Hk=3, Hv=3, seed=1126),
    "n64_root": tc(N=64, accepted="root", seed=1127),
    "n22_root": tc(N=22, accepted="root", seed=1128),
    "n40_k2_root": tc(N=40, K=2, accepted="root", seed=1129),
}


@pytest.mark.parametrize("name", sorted(TC_EDGE))
def test_tensor_core_edge_cases(name):
    w = TC_EDGE[name]
    slots = np.array([3, 0, 4], dtype=np.int32) if w.Bq == 3 else None
    inp = make_inputs(w, slots=slots)
    o, st, cc, status, ws = run_verify(w, inp, mode=lbx.LBX_MODE_TREE)
    assert status == 0
    check_verify(w, inp, o, st, cc)
    assert counters_cleared(w, ws, lbx.LBX_MODE_TREE)


def test_tensor_core_and_cuda_core_kernels_agree_budget64():
    """Node capacity 64 (one CTA per SM) against the CUDA-core kernel on the
    budget-64 serving shapes (4 layers of them)."""
    w = WORKLOADS["serve27b_b64"].replace(L=4)
    inp = make_inputs(w)
    o1, s1, c1, st1, _ = run_verify(w, inp, mode=lbx.LBX_MODE_TREE)
    o2, s2, c2, st2, _ = run_verify(w, inp, mode=lbx.LBX_MODE_TREE_CUDA_CORES)
    assert st1 == st2 == 0
    assert np.abs(o1 - o2).max() <= 1e-4 * np.abs(o2).max()
    assert c1.tobytes() == c2.tobytes()
    # the request slots (the spare slots hold a NaN canary, checked elsewhere)
    used = inp["slot"]
    rel = np.linalg.norm((s1 - s2)[:, used].reshape(-1)) / np.linalg.norm(s2[:, used].reshape(-1))
    assert rel <= 1e-5


def test_tensor_core_and_cuda_core_kernels_agree_full_step():
    w = WORKLOADS["step27b"]
    inp = make_inputs(w)
    o1, s1, c1, st1, _ = run_verify(w, inp, mode=lbx.LBX_MODE_TREE)
    o2, s2, c2, st2, _ = run_verify(w, inp, mode=lbx.LBX_MODE_TREE_CUDA_CORES)
    assert st1 == st2 == 0
    assert np.abs(o1 - o2).max() <= 1e-4 * np.abs(o2).max()
    assert c1.tobytes() == c2.tobytes()
    rel = np.linalg.norm((s1 - s2)[:, :1].reshape(-1)) / np.linalg.norm(s2[:, :1].reshape(-1))
    assert rel <= 1e-5
