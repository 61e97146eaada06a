"""GPU parity of the three unfused entry points against the fp64 oracle.

The pages name three tree-aware state-rollback kernels (Lucebox hub README,
section "02 DFlash DDtree", list "Implemented here"): the tree conv, the tree
gated delta-rule recurrence and the persist ("state rollback").  Here they run
as three C-ABI calls chained on the device -- lbx_tree_conv -> lbx_tree_deltanet
(with per-node state snapshots) -> lbx_tree_persist -- and every output is
compared with the oracle on the same seeded inputs:

* qkv_out (conv + SiLU + L2) within QKV_TOL * max |ref|.  The GPU computes it
  in fp32 from bf16-exact inputs: a K-term dot product, SiLU through the
  hardware exponential and a fast divide (CUDA documents __expf at
  2 + floor(1.173 |y|) ulp, so ~1e-6 relative for the pre-activations' range
  |y| < 10, and __fdividef at 2 ulp), and rsqrtf for the norm (absolute error
  ~1e-6 on outputs up to ~5), so 1e-5 of the largest output leaves a ~5-10x
  margin and still catches a dropped tap or a wrong window row;
* o within O_TOL * max |ref| (the stated bar), from the chained GPU qkv;
* every node's snapshot S_n within STATE_TOL relative Frobenius error of the
  oracle's per-node state, per (layer, request, node, head);
* the persisted state a byte copy of the accepted node's snapshot (and so
  within STATE_TOL of the oracle's accepted state), the conv window
  bit-exact, and slots no request names unchanged byte for byte.

The oracle sees only the seeded inputs: its qkv is its own fp64 conv.
"""
import numpy as np
import pytest
import torch

import oracle
from tree_verify_linear_gb300 import lbx
from tree_verify_linear_gb300.inputs import WORKLOADS, Workload, make_inputs

from gpu_util import O_TOL, STATE_TOL, dev_inputs, o_error, state_rel

pytestmark = pytest.mark.gpu

QKV_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from tree_verify_linear_gb300 import build
    build.build()
    lbx.load()
    oracle.lib()


def run_unfused(w, inp, snapshots=True, persist=True):
    """conv -> deltanet (-> persist) through the C ABI, on one stream.
    Returns numpy copies and the device status."""
    d = dev_inputs(inp)
    cfg = lbx.cfg_of(w)
    nan = float("nan")
    qkv = torch.full((w.L, w.Bq, w.N, w.C), nan, device="cuda")
    o = torch.full((w.L, w.Bq, w.N, w.Hv, w.d), nan, device="cuda")
    ns = (torch.full((w.L, w.Bq, w.N, w.Hv, w.d, w.d), nan, device="cuda")
          if snapshots else None)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lbx.lbx_tree_conv(cfg, d["x"], d["conv_w"], d["conv_cache"], d["parent"], d["slot"], qkv,
                      status)
    lbx.lbx_tree_deltanet(cfg, qkv, d["a"], d["b"], d["state"], d["parent"], d["slot"], o, ns,
                          status)
    if persist:
        lbx.lbx_tree_persist(cfg, d["x"], ns, d["parent"], d["slot"], d["accepted"], d["state"],
                             d["conv_cache"], status)
    torch.cuda.synchronize()
    return dict(qkv=qkv.cpu().numpy(), o=o.cpu().numpy(),
                ns=None if ns is None else ns.cpu().numpy(), state=d["state"].cpu().numpy(),
                cache=d["conv_cache"].cpu().numpy(), status=int(status.item()))


def check_unfused(w, inp, r):
    """Every output of the chained calls against the oracle."""
    assert r["status"] == 0
    # a1: conv + SiLU + L2 of the whole batch
    qkv_ref = oracle.tree_conv(w, inp)
    err = np.abs(r["qkv"].astype(np.float64) - qkv_ref).max() / np.abs(qkv_ref).max()
    assert err <= QKV_TOL, f"qkv error {err:.3e} > {QKV_TOL}"
    # a2: o and every node's state, per head (the oracle's own conv output)
    o_ref = np.zeros((w.L, w.Bq, w.N, w.Hv, w.d))
    worst_ns, worst_acc = 0.0, 0.0
    for l in range(w.L):
        for b in range(w.Bq):
            s = int(inp["slot"][b])
            acc = int(inp["accepted"][b])
            for h in range(w.Hv):
                o_h, ns_h, sacc = oracle.deltanet_head(
                    w.N, w.Hk, w.Hv, w.d, h, w.q_scale, oracle.FORM_PATH, qkv_ref[l, b],
                    inp["a"][l, b], inp["b"][l, b], inp["state"][l, s, h], inp["parent"][b],
                    accepted=acc, want_states=True)
                o_ref[l, b, :, h] = o_h
                for n in range(w.N):
                    worst_ns = max(worst_ns, state_rel(r["ns"][l, b, n, h], ns_h[n]))
                # a3: the persisted state is the accepted node's snapshot, copied
                assert r["state"][l, s, h].tobytes() == r["ns"][l, b, acc, h].tobytes(), \
                    f"persisted state is not the snapshot at layer {l} request {b} head {h}"
                worst_acc = max(worst_acc, state_rel(r["state"][l, s, h], sacc))
    err_o = o_error(r["o"], o_ref)
    assert err_o <= O_TOL, f"o error {err_o:.3e} > {O_TOL}"
    assert worst_ns <= STATE_TOL, f"node state rel error {worst_ns:.3e} > {STATE_TOL}"
    assert worst_acc <= STATE_TOL, f"accepted state rel error {worst_acc:.3e} > {STATE_TOL}"
    # a3: conv window bit-exact; untouched slots byte for byte
    for l in range(w.L):
        for b in range(w.Bq):
            s = int(inp["slot"][b])
            exp = oracle.persist_conv_lb(w.N, w.C, w.K, inp["x"][l, b], inp["conv_cache"][l, s],
                                         inp["parent"][b], inp["accepted"][b])
            assert exp.view(np.uint32).tobytes() == r["cache"][l, s].view(np.uint32).tobytes(), \
                f"conv window mismatch at layer {l} request {b}"
    used = set(int(s) for s in inp["slot"])
    for s in range(w.n_slots):
        if s not in used:
            assert r["state"][:, s].tobytes() == inp["state"][:, s].tobytes(), f"slot {s} touched"
            assert r["cache"][:, s].tobytes() == inp["conv_cache"][:, s].tobytes(), \
                f"conv slot {s} touched"
    return err, err_o, worst_ns


def small(**kw):
    base = dict(name="unfused", L=2, Bq=2, N=13, Hk=2, Hv=4, d=32, tree="ddtree",
                accepted="node", seed=2000)
    base.update(kw)
    return Workload(**base)


CASES = {
    "tiny": WORKLOADS["tiny"],
    "layer27b": WORKLOADS["layer27b"],
    "serve27b_b22_l2": WORKLOADS["serve27b_b22"].replace(L=2),
    "d32_k4": small(seed=2001),
    "d64_k3": small(d=64, K=3, N=22, seed=2002),
    "d128_k2": small(d=128, K=2, Hv=6, N=22, seed=2003),
    "d128_k1": small(d=128, K=1, N=9, seed=2004),
    "d32_k1": small(K=1, seed=2005),
    "uniform_64_d128": small(d=128, N=64, tree="uniform", Hv=6, seed=2006),
    "uniform_64_d32_leaf": small(N=64, tree="uniform", accepted="leaf", seed=2007),
    "root_only": small(N=1, seed=2008),
    "accepted_root": small(N=22, accepted="root", d=128, seed=2009),
    "chain_22": small(N=22, tree="chain", accepted="last", d=64, seed=2010),
    "q_scale_gqa1": small(Hk=4, Hv=4, q_scale=float(1 / np.sqrt(32)), seed=2011),
    "three_requests": small(Bq=3, N=17, seed=2012),
    # 160 (layer, request) pairs over 5 head blocks: the conv grid puts two
    # blocks in each CTA, and the last CTA of each pair holds only one
    "partial_head_group": small(d=128, L=4, Bq=40, Hk=1, Hv=3, seed=2013),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_conv_deltanet_persist_chain_matches_oracle(name):
    w = CASES[name]
    slots = None
    if w.Bq == 3:
        slots = np.array([3, 0, 4], dtype=np.int32)
    elif w.Bq == 5:
        slots = np.array([4, 0, 6, 2, 1], dtype=np.int32)
    inp = make_inputs(w, slots=slots)
    r = run_unfused(w, inp)
    check_unfused(w, inp, r)


def test_deltanet_without_snapshots_gives_the_same_o():
    """node_states = NULL: o unchanged (the snapshot-free instance)."""
    w = small(d=128, Hv=6, N=22, seed=2020)
    inp = make_inputs(w)
    r1 = run_unfused(w, inp, snapshots=True, persist=False)
    r2 = run_unfused(w, inp, snapshots=False, persist=False)
    assert r1["status"] == r2["status"] == 0
    assert np.abs(r1["o"] - r2["o"]).max() <= 1e-6 * np.abs(r1["o"]).max()
    # nothing persisted without lbx_tree_persist
    assert r2["state"].tobytes() == inp["state"].tobytes()
    assert r2["cache"].tobytes() == inp["conv_cache"].tobytes()


def test_unfused_chain_agrees_with_fused_step():
    """The chained unfused calls and lbx_verify_step give the same outputs and
    caches (tensor-core fused step against the CUDA-core unfused kernels)."""
    from gpu_util import run_verify
    w = WORKLOADS["serve27b_b22"].replace(L=2)
    inp = make_inputs(w)
    r = run_unfused(w, inp)
    o, st, cc, status, _ = run_verify(w, inp)
    assert r["status"] == 0 and status == 0
    assert np.abs(r["o"] - o).max() <= 1e-4 * np.abs(o).max()
    assert r["cache"].tobytes() == cc.tobytes()
    used = inp["slot"]
    rel = (np.linalg.norm((r["state"] - st)[:, used].reshape(-1))
           / np.linalg.norm(st[:, used].reshape(-1)))
    assert rel <= 1e-5


# -------------------------------------------------------------------------
# Errors the device detects: status set, nothing written by that call.
# -------------------------------------------------------------------------
@pytest.mark.parametrize("bad", ["root_parent", "forward_parent", "out_of_range"])
def test_invalid_tree_rejected_by_each_call(bad):
    w = small(seed=2030)
    inp = make_inputs(w)
    if bad == "root_parent":
        inp["parent"][1, 0] = 0
    elif bad == "forward_parent":
        inp["parent"][0, 5] = 7
    else:
        inp["parent"][1, 3] = 99
    d = dev_inputs(inp)
    cfg = lbx.cfg_of(w)
    nan = float("nan")
    qkv = torch.full((w.L, w.Bq, w.N, w.C), nan, device="cuda")
    o = torch.full((w.L, w.Bq, w.N, w.Hv, w.d), nan, device="cuda")
    ns = torch.full((w.L, w.Bq, w.N, w.Hv, w.d, w.d), nan, device="cuda")
    for call in ("conv", "deltanet", "persist"):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        if call == "conv":
            lbx.lbx_tree_conv(cfg, d["x"], d["conv_w"], d["conv_cache"], d["parent"], d["slot"],
                              qkv, status)
        elif call == "deltanet":
            lbx.lbx_tree_deltanet(cfg, qkv, d["a"], d["b"], d["state"], d["parent"], d["slot"],
                                  o, ns, status)
        else:
            lbx.lbx_tree_persist(cfg, d["x"], ns, d["parent"], d["slot"], d["accepted"],
                                 d["state"], d["conv_cache"], status)
        torch.cuda.synchronize()
        assert int(status.item()) == lbx.LBX_ETREE, call
    assert torch.isnan(qkv).all() and torch.isnan(o).all() and torch.isnan(ns).all()
    assert d["state"].cpu().numpy().tobytes() == inp["state"].tobytes()
    assert d["conv_cache"].cpu().numpy().tobytes() == inp["conv_cache"].tobytes()


@pytest.mark.parametrize("bad", ["accepted", "slot", "duplicate_slots"])
def test_persist_rejects_bad_indices(bad):
    w = small(seed=2031)
    slots = np.array([1, 1], dtype=np.int32) if bad == "duplicate_slots" else None
    inp = make_inputs(w, slots=slots)
    if bad == "accepted":
        inp["accepted"][1] = w.N
    elif bad == "slot":
        inp["slot"][0] = w.n_slots
    d = dev_inputs(inp)
    cfg = lbx.cfg_of(w)
    ns = torch.randn((w.L, w.Bq, w.N, w.Hv, w.d, w.d), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lbx.lbx_tree_persist(cfg, d["x"], ns, d["parent"], d["slot"], d["accepted"], d["state"],
                         d["conv_cache"], status)
    torch.cuda.synchronize()
    assert int(status.item()) == lbx.LBX_EINVAL
    assert d["state"].cpu().numpy().tobytes() == inp["state"].tobytes()
    assert d["conv_cache"].cpu().numpy().tobytes() == inp["conv_cache"].tobytes()
