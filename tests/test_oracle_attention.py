"""Pins of the oracle's tree-masked attention (CPU only).

The oracle (oracle/lbx_oracle.c, lbxo_tree_attention) walks each node's root
path and takes a softmax over the cached context plus that path.  It is
checked here against what the reading of the pages and the mathematics fix:
scipy's softmax over explicitly built key sets (a root-only tree, and every
node of a random tree as the last query of the chain ctx + its root path),
causal attention over [context; tree] for a chain-shaped tree, closed forms
(an empty context, identical keys, a hand-worked two-key case), the GQA
mapping, the mask (a node's subtree-external changes leave it alone) and
relabelling invariance.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from tree_verify_linear_gb300.inputs import (ATTN_WORKLOADS, AttnWorkload, bf16_bits,
                                             bf16_to_f32, make_attn_inputs)


def f64(b):
    return bf16_to_f32(b).astype(np.float64)


def run(w, inp, scale=None):
    return oracle.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["k_tree"],
                                 inp["v_tree"], inp["ctx_len"], inp["parent"],
                                 w.scale if scale is None else scale)


def small(**kw):
    base = dict(name="pin", L=2, Bq=3, N=9, Hq=6, Hkv=2, dh=16, T=11, ctx="ragged",
                tree="uniform", seed=3000)
    base.update(kw)
    return AttnWorkload(**base)


def path_of(parent, n):
    p = []
    while n >= 0:
        p.append(n)
        n = parent[n]
    return p[::-1]  # root first


def reference_node(w, inp, l, b, n, hq):
    """scipy softmax over the explicit key set of (l, b, n, hq)."""
    G = w.Hq // w.Hkv
    g = hq // G
    C = int(inp["ctx_len"][b])
    path = path_of(inp["parent"][b], n)
    K = np.concatenate([f64(inp["k_cache"][l, b, :C, g]), f64(inp["k_tree"][l, b, path, g])])
    V = np.concatenate([f64(inp["v_cache"][l, b, :C, g]), f64(inp["v_tree"][l, b, path, g])])
    q = f64(inp["q"][l, b, n, hq])
    return softmax(w.scale * (K @ q)) @ V


def test_root_only_tree_is_plain_attention():
    w = small(N=1, ctx="full", seed=3001)
    inp = make_attn_inputs(w)
    o = run(w, inp)
    for l in range(w.L):
        for b in range(w.Bq):
            for hq in range(w.Hq):
                np.testing.assert_allclose(o[l, b, 0, hq], reference_node(w, inp, l, b, 0, hq),
                                           rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("tree", ["uniform", "ddtree", "chain"])
def test_every_node_is_attention_over_context_and_its_path(tree):
    w = small(tree=tree, seed=3002 + len(tree))
    inp = make_attn_inputs(w)
    o = run(w, inp)
    for l in range(w.L):
        for b in range(w.Bq):
            for n in range(w.N):
                for hq in range(w.Hq):
                    np.testing.assert_allclose(o[l, b, n, hq],
                                               reference_node(w, inp, l, b, n, hq),
                                               rtol=1e-11, atol=1e-12)


def test_chain_tree_is_causal_attention_over_context_then_tree():
    w = small(tree="chain", ctx="full", N=7, T=5, L=1, Bq=1, seed=3010)
    inp = make_attn_inputs(w)
    o = run(w, inp)
    G = w.Hq // w.Hkv
    for hq in range(w.Hq):
        g = hq // G
        K = np.concatenate([f64(inp["k_cache"][0, 0, :, g]), f64(inp["k_tree"][0, 0, :, g])])
        V = np.concatenate([f64(inp["v_cache"][0, 0, :, g]), f64(inp["v_tree"][0, 0, :, g])])
        Q = f64(inp["q"][0, 0, :, hq])
        S = w.scale * Q @ K.T                              # [N][T + N]
        T = w.T
        mask = np.tril(np.ones((w.N, w.N), dtype=bool))    # node n sees tree nodes 0..n
        full = np.concatenate([np.ones((w.N, T), dtype=bool), mask], axis=1)
        S = np.where(full, S, -np.inf)
        np.testing.assert_allclose(o[0, 0, :, hq], softmax(S, axis=1) @ V, rtol=1e-12,
                                   atol=1e-12)


def test_empty_context_root_returns_its_own_value():
    w = small(ctx="full", T=0, seed=3011)
    inp = make_attn_inputs(w)
    o = run(w, inp)
    G = w.Hq // w.Hkv
    for hq in range(w.Hq):
        assert np.array_equal(o[:, :, 0, hq], f64(inp["v_tree"][:, :, 0, hq // G]))


def test_identical_keys_average_the_visible_values():
    w = small(seed=3012)
    inp = make_attn_inputs(w)
    key = inp["k_cache"][0, 0, 0, 0].copy()
    inp["k_cache"][:] = key
    inp["k_tree"][:] = key
    o = run(w, inp)
    G = w.Hq // w.Hkv
    for l in range(w.L):
        for b in range(w.Bq):
            C = int(inp["ctx_len"][b])
            for n in range(w.N):
                path = path_of(inp["parent"][b], n)
                for hq in range(w.Hq):
                    g = hq // G
                    vals = np.concatenate([f64(inp["v_cache"][l, b, :C, g]),
                                           f64(inp["v_tree"][l, b, path, g])])
                    np.testing.assert_allclose(o[l, b, n, hq], vals.mean(axis=0), rtol=1e-12,
                                               atol=1e-13)


def test_hand_worked_two_key_case():
    """dh = 2, scale 1, one cached key (0, 0) with value (1, 0), a root whose
    key (1, 0) and value (0, 1) meet the query (1, 0): scores 0 and 1, so
    o = (1, e) / (1 + e)."""
    w = AttnWorkload("hand", L=1, Bq=1, N=1, Hq=1, Hkv=1, dh=2, T=1)
    one = bf16_bits(np.array([1.0], np.float32))[0]
    zero = np.uint16(0)
    inp = dict(q=np.array([one, zero], np.uint16).reshape(1, 1, 1, 1, 2),
               k_cache=np.array([zero, zero], np.uint16).reshape(1, 1, 1, 1, 2),
               v_cache=np.array([one, zero], np.uint16).reshape(1, 1, 1, 1, 2),
               k_tree=np.array([one, zero], np.uint16).reshape(1, 1, 1, 1, 2),
               v_tree=np.array([zero, one], np.uint16).reshape(1, 1, 1, 1, 2),
               ctx_len=np.array([1], np.int32), parent=np.array([[-1]], np.int32))
    o = run(w, inp, scale=1.0)
    e = np.e
    np.testing.assert_allclose(o.reshape(2), [1 / (1 + e), e / (1 + e)], rtol=1e-15)


def test_gqa_groups_are_contiguous():
    w = small(Hq=6, Hkv=3, seed=3013)
    inp = make_attn_inputs(w)
    o0 = run(w, inp)
    inp2 = {k: v.copy() for k, v in inp.items()}
    inp2["k_cache"][:, :, :, 1] = bf16_bits(np.random.default_rng(1).standard_normal(
        inp2["k_cache"][:, :, :, 1].shape, dtype=np.float32))
    o1 = run(w, inp2)
    changed = [hq for hq in range(w.Hq) if not np.array_equal(o0[:, :, :, hq], o1[:, :, :, hq])]
    assert changed == [2, 3]  # G = 2: query heads 2 and 3 read KV head 1


def test_a_node_sees_only_its_root_path():
    """Changing node m's key and value changes exactly m and its descendants."""
    w = small(L=1, Bq=1, N=12, seed=3014)
    inp = make_attn_inputs(w)
    par = inp["parent"][0]
    o0 = run(w, inp)
    for m in range(w.N):
        inp2 = {k: v.copy() for k, v in inp.items()}
        inp2["k_tree"][0, 0, m] ^= np.uint16(0x0040)
        inp2["v_tree"][0, 0, m] ^= np.uint16(0x0040)
        o1 = run(w, inp2)
        desc = {n for n in range(w.N) if m in path_of(par, n)}
        moved = {n for n in range(w.N) if not np.array_equal(o0[0, 0, n], o1[0, 0, n])}
        assert moved == desc, (m, moved, desc)


def test_topological_relabelling_permutes_outputs():
    w = small(L=1, Bq=1, N=10, tree="ddtree", seed=3015)
    inp = make_attn_inputs(w)
    par = inp["parent"][0]
    # a different topological order: breadth first by depth, ties by index
    depth = np.array([len(path_of(par, n)) for n in range(w.N)])
    order = np.lexsort((np.arange(w.N), depth))      # new label i -> old node order[i]
    new_of = np.empty(w.N, np.int64)
    new_of[order] = np.arange(w.N)
    par2 = np.array([-1 if par[o] < 0 else new_of[par[o]] for o in order], np.int32)
    inp2 = dict(inp)
    for k in ("q", "k_tree", "v_tree"):
        inp2[k] = np.ascontiguousarray(inp[k][:, :, order])
    inp2["parent"] = par2.reshape(1, -1)
    o0, o1 = run(w, inp), run(w, inp2)
    np.testing.assert_allclose(o1, o0[:, :, order], rtol=1e-13, atol=1e-14)


def test_invalid_inputs_rejected():
    w = ATTN_WORKLOADS["attn_tiny"]
    inp = make_attn_inputs(w)
    bad = dict(inp)
    bad["parent"] = inp["parent"].copy()
    bad["parent"][0, 3] = 5
    with pytest.raises(oracle.OracleError):
        run(w, bad)
    bad = dict(inp)
    bad["ctx_len"] = np.array([w.T + 1, 0, 1], np.int32)
    with pytest.raises(oracle.OracleError):
        run(w, bad)
