"""GPU parity of the tree-masked attention (lbx_tree_attention, tensor cores)
against the fp64 oracle, through the C ABI.

Tolerance: max |o_gpu - o_ref| <= 1e-4 * max |o_ref| per case.  The kernel's
operands are the exact bf16 inputs, its products accumulate in fp32, and P
enters the P.V product as bf16 hi + lo (about 2^-17 relative), so its error is
a few 1e-6 of max |o|; 1e-4 leaves a wide margin while still catching any
missing or extra key (one key of ~4000 moves o by ~1e-3 of its scale).
"""
import numpy as np
import pytest

import oracle
from tree_verify_linear_gb300 import lbx
from tree_verify_linear_gb300.inputs import ATTN_WORKLOADS, AttnWorkload, make_attn_inputs

from gpu_util import to_dev

pytestmark = pytest.mark.gpu

ATTN_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from tree_verify_linear_gb300 import build
    build.build()
    lbx.load()
    oracle.lib()


def run_attn(w, inp, calls=1, o_fill=float("nan")):
    import torch
    d = {k: to_dev(v) for k, v in inp.items()}
    o = torch.full((w.L, w.Bq, w.N, w.Hq, w.dh), o_fill, device="cuda")
    ws = lbx.new_attn_workspace(w.L, w.Bq, w.N, w.Hq, w.Hkv, w.dh, w.T)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(calls):
        lbx.lbx_tree_attention(w.scale, d["ctx_len"], d["parent"], d["q"], d["k_cache"],
                               d["v_cache"], d["k_tree"], d["v_tree"], o, ws, status)
    torch.cuda.synchronize()
    return o.cpu().numpy(), int(status.item()), ws.cpu().numpy()


def ref_layers(w, inp, layers):
    sl = {k: (np.ascontiguousarray(v[layers]) if k not in ("ctx_len", "parent") else v)
          for k, v in inp.items()}
    return oracle.tree_attention(sl["q"], sl["k_cache"], sl["v_cache"], sl["k_tree"],
                                 sl["v_tree"], sl["ctx_len"], sl["parent"], w.scale)


def err(o_gpu, o_ref):
    return float(np.abs(o_gpu.astype(np.float64) - o_ref).max() / np.abs(o_ref).max())


def counters_zero(w, ws):
    """The per-row-tile arrival counters (the workspace's 256-byte rounded
    tail, one uint32 per (layer, request, KV head, row tile)) are re-armed."""
    G = w.Hq // w.Hkv
    tiles = 1
    while -(-G // tiles) * w.N > 128:
        tiles += 1
    tiles = -(-G // -(-G // tiles))
    cb = (w.L * w.Bq * w.Hkv * tiles * 4 + 255) // 256 * 256
    return not ws[-cb:].any()


def test_tiny_all_outputs():
    w = ATTN_WORKLOADS["attn_tiny"]
    inp = make_attn_inputs(w)
    o, status, ws = run_attn(w, inp)
    assert status == 0
    e = err(o, ref_layers(w, inp, slice(0, w.L)))
    assert e <= ATTN_TOL, e


def test_attn27b_full_size_all_layers():
    """The 16-layer budget-22 workload (the bench's), every layer checked."""
    w = ATTN_WORKLOADS["attn27b"]
    inp = make_attn_inputs(w)
    o, status, _ = run_attn(w, inp)
    assert status == 0
    assert np.isfinite(o).all()
    e = err(o, ref_layers(w, inp, slice(0, w.L)))
    assert e <= ATTN_TOL, e


def test_attn27b_serve_ragged_contexts():
    """Five requests with contexts of 4096..8192 keys and one empty context;
    the first, a middle and the last layer checked (about 9 s of oracle time
    per layer)."""
    w = ATTN_WORKLOADS["attn27b_serve"]
    inp = make_attn_inputs(w)
    assert inp["ctx_len"][1] == 0
    o, status, _ = run_attn(w, inp)
    assert status == 0
    assert np.isfinite(o).all()
    for l in (0, 7, w.L - 1):
        e = err(o[l:l + 1], ref_layers(w, inp, slice(l, l + 1)))
        assert e <= ATTN_TOL, (l, e)


def small(**kw):
    base = dict(name="edge", L=2, Bq=2, N=22, Hq=12, Hkv=2, dh=256, T=200, ctx="ragged",
                tree="ddtree", seed=4000)
    base.update(kw)
    return AttnWorkload(**base)


EDGE = {
    "n1": small(N=1, seed=4001),
    "n64_chain": small(N=64, tree="chain", seed=4002),
    "n64_g2_one_tile": small(N=64, Hq=4, Hkv=2, max_children=4, seed=4003),
    "n40_g8_three_tiles": small(N=40, Hq=16, Hkv=2, tree="uniform", seed=4004),
    "g1": small(Hq=3, Hkv=3, seed=4005),
    "no_context": small(T=0, ctx="full", seed=4006),
    "t33_ragged_blocks": small(T=33, ctx="full", seed=4007),
    "t77_three_requests": small(Bq=3, T=77, seed=4008),
    "long_context": small(L=1, Bq=1, T=3000, ctx="full", seed=4009),
    "n23_g6": small(N=23, Hq=6, Hkv=1, T=64, ctx="full", seed=4010),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(name):
    w = EDGE[name]
    inp = make_attn_inputs(w)
    o, status, ws = run_attn(w, inp)
    assert status == 0
    e = err(o, ref_layers(w, inp, slice(0, w.L)))
    assert e <= ATTN_TOL, e
    assert counters_zero(w, ws)


def test_garbage_past_the_context_does_not_leak():
    """Cache rows at or past ctx_len hold NaN: the result is unchanged."""
    w = small(Bq=3, T=100, seed=4020)
    inp = make_attn_inputs(w)
    o1, st1, _ = run_attn(w, inp)
    bad = dict(inp)
    for k in ("k_cache", "v_cache"):
        a = inp[k].copy()
        for b in range(w.Bq):
            a[:, b, inp["ctx_len"][b]:] = np.uint16(0x7FC0)  # bf16 NaN
        bad[k] = a
    o2, st2, _ = run_attn(w, bad)
    assert st1 == st2 == 0
    assert np.isfinite(o2).all()
    assert np.array_equal(o1, o2)


def test_two_calls_in_a_row_agree():
    w = small(seed=4021)
    inp = make_attn_inputs(w)
    o1, _, _ = run_attn(w, inp, calls=1)
    o2, st, ws = run_attn(w, inp, calls=2)
    assert st == 0
    assert np.array_equal(o1, o2)
    assert counters_zero(w, ws)


@pytest.mark.parametrize("bad", ["parent_forward", "root_parent", "ctx_over"])
def test_invalid_inputs_set_status_and_write_nothing(bad):
    w = small(seed=4022)
    inp = make_attn_inputs(w)
    inp = {k: v.copy() for k, v in inp.items()}
    if bad == "parent_forward":
        inp["parent"][1, 5] = 7
    elif bad == "root_parent":
        inp["parent"][0, 0] = 0
    else:
        inp["ctx_len"][0] = w.T + 1
    o, status, _ = run_attn(w, inp)
    assert status == lbx.LBX_ETREE
    assert np.isnan(o).all()
