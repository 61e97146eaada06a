"""Pins for the fp64 oracle: checks against the mathematics of the gated delta
rule, closed forms, textbook/library routines and brute force -- never against
the oracle itself.  No GPU needed.

Method: the three tree-aware state-rollback ops of the DDTree verify step
(Lucebox hub README, section "02 DFlash DDtree", "Implemented here"), with the
gated delta rule S_n = a_n S_p (I - b_n k_n k_n^T) + b_n v_n k_n^T, o_n = S_n q_n.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
from tree_verify_linear_gb300.inputs import (WORKLOADS, Workload, bf16_bits, bf16_to_f32,
                                             make_inputs, make_tree)

RNG = np.random.default_rng(12345)


def bf(x):
    """Round to bf16 and return (bits, exact float64 value)."""
    bits = bf16_bits(np.asarray(x, dtype=np.float32))
    return bits, bf16_to_f32(bits).astype(np.float64)


def qkv_row(q, k, v):
    """One [C] row for Hk = Hv = 1 (channel order q | k | v)."""
    return np.concatenate([q, k, v]).astype(np.float64)


def unit(v):
    return v / np.linalg.norm(v)


def small_workload(**kw):
    base = dict(name="small", L=2, Bq=2, N=9, Hk=2, Hv=4, d=8, tree="uniform",
                accepted="node", seed=77)
    base.update(kw)
    return Workload(**base)


# --------------------------------------------------------------------------
# One step of the delta rule, pinned by what it must do to k and to k's
# orthogonal complement (together these fix S_n completely).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("a,b", [(0.5, 0.25), (1.0, 1.0), (0.8125, 0.0), (1.0, 0.0), (0.375, 0.9375)])
def test_single_step_fixes_state_on_k_and_its_complement(a, b):
    d = 8
    k = unit(RNG.standard_normal(d))
    q = RNG.standard_normal(d)
    v = RNG.standard_normal(d)
    S0 = (RNG.standard_normal((d, d)) * 0.1).astype(np.float32)
    ab, av = bf(a)
    bb, bv = bf(b)
    qkv = qkv_row(q, k, v)[None, :]
    o, ns, _ = oracle.deltanet_head(1, 1, 1, d, 0, 1.0, oracle.FORM_PATH, qkv, ab.reshape(1, 1),
                                    bb.reshape(1, 1), S0, np.array([-1]), want_states=True)
    S1 = ns[0]
    S0d = S0.astype(np.float64)
    # along k: the delta rule moves S k toward v by a fraction b
    np.testing.assert_allclose(S1 @ k, av[()] * (1 - bv[()]) * (S0d @ k) + bv[()] * v, atol=1e-12)
    # orthogonal to k: only the decay acts
    for _ in range(3):
        x = RNG.standard_normal(d)
        x -= (x @ k) * k
        np.testing.assert_allclose(S1 @ x, av[()] * (S0d @ x), atol=1e-12)
    # the read-out is the state applied to q
    np.testing.assert_allclose(o[0], S1 @ q, atol=1e-12)


def test_write_with_basis_key_replaces_one_column():
    """a = b = 1, k = e_j: the update overwrites column j of S with v."""
    d, j = 6, 4
    k = np.zeros(d)
    k[j] = 1.0
    v = RNG.standard_normal(d)
    S0 = RNG.standard_normal((d, d)).astype(np.float32)
    one, _ = bf(1.0)
    qkv = qkv_row(np.ones(d), k, v)[None, :]
    _, ns, _ = oracle.deltanet_head(1, 1, 1, d, 0, 1.0, oracle.FORM_PATH, qkv, one.reshape(1, 1),
                                    one.reshape(1, 1), S0, np.array([-1]), want_states=True)
    expect = S0.astype(np.float64).copy()
    expect[:, j] = v
    np.testing.assert_array_equal(ns[0], expect)


# --------------------------------------------------------------------------
# Tree structure: chain == sequential recurrence, every node == its path,
# rank-1 form == explicit transition matrices.
# --------------------------------------------------------------------------
def _random_head_inputs(N, d, Hk=1, Hv=1, unit_k=True):
    C = 2 * Hk * d + Hv * d
    qkv = RNG.standard_normal((N, C))
    if unit_k:
        for n in range(N):
            for g in range(2 * Hk):
                qkv[n, g * d:(g + 1) * d] = unit(qkv[n, g * d:(g + 1) * d])
    a = bf16_bits(np.exp(-np.logaddexp(0, RNG.standard_normal((N, Hv)))).astype(np.float32))
    b = bf16_bits(expit(RNG.standard_normal((N, Hv))).astype(np.float32))
    S0 = (RNG.standard_normal((d, d)) * 0.1).astype(np.float32)
    return qkv, a, b, S0


def test_chain_tree_equals_sequential_recurrence():
    N, d = 24, 16
    qkv, a, b, S0 = _random_head_inputs(N, d)
    chain = np.arange(-1, N - 1, dtype=np.int32)
    o1, s1, acc1 = oracle.deltanet_head(N, 1, 1, d, 0, 1.0, oracle.FORM_PATH, qkv, a, b, S0,
                                        chain, accepted=N - 1, want_states=True)
    o2, s2, acc2 = oracle.deltanet_head(N, 1, 1, d, 0, 1.0, oracle.FORM_SEQUENTIAL, qkv, a, b,
                                        S0, chain, accepted=N - 1, want_states=True)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s1, s2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(acc1, s2[-1], rtol=0, atol=1e-12)


def test_sequential_form_rejects_non_chain():
    N, d = 5, 4
    qkv, a, b, S0 = _random_head_inputs(N, d)
    with pytest.raises(oracle.OracleError):
        oracle.deltanet_head(N, 1, 1, d, 0, 1.0, oracle.FORM_SEQUENTIAL, qkv, a, b, S0,
                             np.array([-1, 0, 0, 1, 2], dtype=np.int32))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_every_node_equals_sequential_over_its_path(seed):
    """North-star check: each node of a random tree equals the recurrence
    brute-forced over its root-to-node path (run as a chain)."""
    rng = np.random.default_rng(seed)
    N, d = 14, 8
    parent = make_tree(rng, N, "uniform")
    qkv, a, b, S0 = _random_head_inputs(N, d)
    o, ns, _ = oracle.deltanet_head(N, 1, 1, d, 0, 1.0, oracle.FORM_PATH, qkv, a, b, S0, parent,
                                    want_states=True)
    for n in range(N):
        path = []
        m = n
        while m >= 0:
            path.append(m)
            m = parent[m]
        path = path[::-1]
        T = len(path)
        chain = np.arange(-1, T - 1, dtype=np.int32)
        oc, sc, _ = oracle.deltanet_head(T, 1, 1, d, 0, 1.0, oracle.FORM_SEQUENTIAL,
                                         qkv[path], a[path], b[path], S0, chain,
                                         want_states=True)
        np.testing.assert_allclose(o[n], oc[-1], rtol=0, atol=1e-12)
        np.testing.assert_allclose(ns[n], sc[-1], rtol=0, atol=1e-12)


def test_rank1_form_equals_explicit_matrix_form():
    rng = np.random.default_rng(5)
    N, d = 10, 8
    parent = make_tree(rng, N, "uniform")
    qkv, a, b, S0 = _random_head_inputs(N, d, Hk=2, Hv=4)
    for h in range(4):
        o1, s1, _ = oracle.deltanet_head(N, 2, 4, d, h, 1.0, oracle.FORM_PATH, qkv, a, b, S0,
                                         parent, want_states=True)
        o2, s2, _ = oracle.deltanet_head(N, 2, 4, d, h, 1.0, oracle.FORM_MATRIX, qkv, a, b, S0,
                                         parent, want_states=True)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(s1, s2, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Special gate values.
# --------------------------------------------------------------------------
def _tiny_with_gates(a_val, b_val, seed=3):
    w = small_workload(seed=seed)
    inp = make_inputs(w)
    inp["a"][...] = bf16_bits(np.full(inp["a"].shape, a_val, np.float32))
    inp["b"][...] = bf16_bits(np.full(inp["b"].shape, b_val, np.float32))
    return w, inp


def test_a1_b0_leaves_state_unchanged_and_reads_out_S0_q():
    w, inp = _tiny_with_gates(1.0, 0.0)
    qkv = oracle.tree_conv(w, inp)
    o, ns = oracle.tree_deltanet(w, qkv, inp, want_states=True)
    G = w.Hv // w.Hk
    for l in range(w.L):
        for b in range(w.Bq):
            s = inp["slot"][b]
            for h in range(w.Hv):
                S0 = inp["state"][l, s, h].astype(np.float64)
                kh = h // G
                for n in range(w.N):
                    np.testing.assert_array_equal(ns[l, b, n, h], S0)
                    q = qkv[l, b, n, kh * w.d:(kh + 1) * w.d]
                    np.testing.assert_allclose(o[l, b, n, h], S0 @ q, rtol=1e-13, atol=1e-14)


def test_b0_state_is_path_decay_times_S0():
    w = small_workload(seed=9)
    inp = make_inputs(w)
    inp["b"][...] = 0
    qkv = oracle.tree_conv(w, inp)
    _, ns = oracle.tree_deltanet(w, qkv, inp, want_states=True)
    av = bf16_to_f32(inp["a"]).astype(np.float64)
    for b in range(w.Bq):
        par = inp["parent"][b]
        for n in range(w.N):
            for l in range(w.L):
                for h in range(w.Hv):
                    g = 1.0
                    m = n
                    while m >= 0:
                        g *= av[l, b, m, h]
                        m = par[m]
                    S0 = inp["state"][l, inp["slot"][b], h].astype(np.float64)
                    np.testing.assert_allclose(ns[l, b, n, h], g * S0, rtol=1e-13, atol=0)


def test_a1_b1_state_maps_k_to_v():
    """With a = b = 1 and unit-norm k the new state sends k_n to v_n."""
    w, inp = _tiny_with_gates(1.0, 1.0, seed=11)
    w0 = w.replace(l2_eps=0.0)
    qkv = oracle.tree_conv(w0, inp)
    _, ns = oracle.tree_deltanet(w0, qkv, inp, want_states=True)
    d, Hk, G = w.d, w.Hk, w.Hv // w.Hk
    for l in range(w.L):
        for b in range(w.Bq):
            for n in range(w.N):
                for h in range(w.Hv):
                    kh = h // G
                    k = qkv[l, b, n, Hk * d + kh * d:Hk * d + (kh + 1) * d]
                    v = qkv[l, b, n, 2 * Hk * d + h * d:2 * Hk * d + (h + 1) * d]
                    np.testing.assert_allclose(ns[l, b, n, h] @ k, v, rtol=0, atol=1e-12)


def test_q_scale_scales_output():
    w = small_workload(seed=13)
    inp = make_inputs(w)
    items = [(l, b, h) for l in range(w.L) for b in range(w.Bq) for h in range(w.Hv)]
    o1, s1, _ = oracle.verify_heads(w, inp, items)
    o2, s2, _ = oracle.verify_heads(w.replace(q_scale=1 / np.sqrt(w.d)), inp, items)
    np.testing.assert_allclose(o2, o1 / np.sqrt(w.d), rtol=1e-14, atol=0)
    np.testing.assert_array_equal(s1, s2)


# --------------------------------------------------------------------------
# Conv along the ancestor path.
# --------------------------------------------------------------------------
def _silu(y):
    return y * expit(y)


def test_conv_on_chain_is_causal_conv1d():
    """On a chain the tree conv is the textbook causal depthwise conv1d over
    [cache rows, inputs] (numpy's convolve), then SiLU; v channels are not
    normalised, q and k channels are rescaled to unit length."""
    w = small_workload(tree="chain", N=12, seed=21)
    inp = make_inputs(w)
    qkv = oracle.tree_conv(w, inp)
    K, C, d, Hk = w.K, w.C, w.d, w.Hk
    for l in range(w.L):
        for b in range(w.Bq):
            s = inp["slot"][b]
            seq = np.concatenate([inp["conv_cache"][l, s].astype(np.float64),
                                  bf16_to_f32(inp["x"][l, b]).astype(np.float64)])
            wts = bf16_to_f32(inp["conv_w"][l]).astype(np.float64)
            pre = np.empty((w.N, C))
            for c in range(C):
                # np.convolve flips its kernel: y[t] = sum_j w[K-1-j] x[t-j]
                full = np.convolve(seq[:, c], wts[c][::-1], mode="full")
                pre[:, c] = full[K - 1:K - 1 + w.N]
            act = _silu(pre)
            np.testing.assert_allclose(qkv[l, b, :, 2 * Hk * d:], act[:, 2 * Hk * d:],
                                       rtol=1e-13, atol=1e-14)
            for g in range(2 * Hk):
                blk = act[:, g * d:(g + 1) * d]
                ref = blk / np.sqrt((blk ** 2).sum(axis=1, keepdims=True) + w.l2_eps)
                np.testing.assert_allclose(qkv[l, b, :, g * d:(g + 1) * d], ref, rtol=1e-12,
                                           atol=1e-14)


def test_conv_tap_direction_and_cache_continuation():
    """Single-tap weights select one window position: tap K-1 is the node
    itself, tap 0 the (K-1)-th element back, continuing into the cache with
    the most recent cached row first."""
    N, Hk, Hv, d, K = 5, 1, 1, 4, 4
    C = 2 * Hk * d + Hv * d
    parent = np.array([-1, 0, 1, 0, 3], dtype=np.int32)   # depths 0,1,2,1,2
    x = bf16_bits(RNG.standard_normal((N, C)).astype(np.float32))
    xf = bf16_to_f32(x).astype(np.float64)
    cache = RNG.standard_normal((K - 1, C)).astype(np.float32)
    cf = cache.astype(np.float64)
    windows = {  # window element j = 0..3 for each node, written out by hand
        0: [xf[0], cf[2], cf[1], cf[0]],
        1: [xf[1], xf[0], cf[2], cf[1]],
        2: [xf[2], xf[1], xf[0], cf[2]],
        3: [xf[3], xf[0], cf[2], cf[1]],
        4: [xf[4], xf[3], xf[0], cf[2]],
    }
    for j in range(K):
        wt = np.zeros((C, K), dtype=np.float32)
        wt[:, K - 1 - j] = 1.0
        out = oracle.conv_lb(N, Hk, Hv, d, K, 1e-6, x, bf16_bits(wt), cache, parent)
        for n in range(N):
            np.testing.assert_allclose(out[n, 2 * d:], _silu(windows[n][j][2 * d:]), rtol=1e-14,
                                       atol=0)


def test_tree_conv_equals_conv_over_each_path():
    w = small_workload(seed=31, N=12)
    inp = make_inputs(w)
    qkv = oracle.tree_conv(w, inp)
    K = w.K
    for l in range(w.L):
        for b in range(w.Bq):
            s = inp["slot"][b]
            par = inp["parent"][b]
            for n in range(w.N):
                path = []
                m = n
                while m >= 0:
                    path.append(m)
                    m = par[m]
                path = path[::-1]
                T = len(path)
                chain_out = oracle.conv_lb(T, w.Hk, w.Hv, w.d, K, w.l2_eps,
                                           inp["x"][l, b][path], inp["conv_w"][l],
                                           inp["conv_cache"][l, s],
                                           np.arange(-1, T - 1, dtype=np.int32))
                np.testing.assert_array_equal(qkv[l, b, n], chain_out[-1])


def test_q_and_k_have_unit_norm_after_l2():
    w = WORKLOADS["tiny"]
    inp = make_inputs(w)
    qkv = oracle.tree_conv(w, inp)
    d = w.d
    for g in range(2 * w.Hk):
        nrm = np.linalg.norm(qkv[..., g * d:(g + 1) * d], axis=-1)
        np.testing.assert_allclose(nrm, 1.0, atol=1e-5)


# --------------------------------------------------------------------------
# Head mapping (GQA): value head h reads key head h // (Hv / Hk).
# --------------------------------------------------------------------------
def test_value_head_reads_its_key_head_only():
    w = small_workload(L=1, Bq=1, seed=41)
    inp = make_inputs(w)
    items = [(0, 0, h) for h in range(w.Hv)]
    o_ref, _, _ = oracle.verify_heads(w, inp, items)
    G, d = w.Hv // w.Hk, w.d
    for kh in range(w.Hk):
        pert = {k: v.copy() for k, v in inp.items()}
        cols = np.r_[kh * d:(kh + 1) * d, w.Hk * d + kh * d:w.Hk * d + (kh + 1) * d]
        pert["x"][..., cols] = bf16_bits(RNG.standard_normal(pert["x"][..., cols].shape)
                                         .astype(np.float32))
        o_p, _, _ = oracle.verify_heads(w, pert, items)
        for h in range(w.Hv):
            changed = not np.array_equal(o_p[h], o_ref[h])
            assert changed == (h // G == kh), (kh, h)


# --------------------------------------------------------------------------
# Relabelling and persist.
# --------------------------------------------------------------------------
def test_topological_relabelling_permutes_outputs():
    w = small_workload(L=1, Bq=1, N=10, seed=51)
    inp = make_inputs(w)
    par = inp["parent"][0]
    N = w.N
    # random topological order: repeatedly pick any node whose parent is placed
    rng = np.random.default_rng(3)
    order, placed = [0], {0}
    while len(order) < N:
        ready = [i for i in range(N) if i not in placed and par[i] in placed]
        i = int(rng.choice(ready))
        order.append(i)
        placed.add(i)
    new_of = {old: new for new, old in enumerate(order)}
    pinp = {k: v.copy() for k, v in inp.items()}
    pinp["parent"][0] = [-1 if par[o] < 0 else new_of[int(par[o])] for o in order]
    pinp["x"][0, 0] = inp["x"][0, 0][order]
    pinp["a"][0, 0] = inp["a"][0, 0][order]
    pinp["b"][0, 0] = inp["b"][0, 0][order]
    pinp["accepted"][0] = new_of[int(inp["accepted"][0])]
    items = [(0, 0, h) for h in range(w.Hv)]
    o1, s1, _ = oracle.verify_heads(w, inp, items)
    o2, s2, _ = oracle.verify_heads(w, pinp, items)
    np.testing.assert_allclose(o2, o1[:, order], rtol=0, atol=1e-14)
    np.testing.assert_allclose(s2, s1, rtol=0, atol=1e-14)


def test_persist_state_is_accepted_node_state_for_every_choice():
    w = WORKLOADS["tiny"]
    inp = make_inputs(w)
    qkv = oracle.tree_conv(w, inp)
    _, ns = oracle.tree_deltanet(w, qkv, inp, want_states=True)
    items = [(0, 0, h) for h in range(w.Hv)]
    for acc in range(w.N):
        inp2 = dict(inp)
        inp2["accepted"] = np.array([acc], dtype=np.int32)
        _, sacc, _ = oracle.verify_heads(w, inp2, items, want_o=False)
        for h in range(w.Hv):
            np.testing.assert_array_equal(sacc[h], ns[0, 0, acc, h])


def test_persist_conv_window_is_last_inputs_of_accepted_path():
    w = WORKLOADS["tiny"]
    inp = make_inputs(w)
    par = inp["parent"][0]
    s = inp["slot"][0]
    K = w.K
    for acc in range(w.N):
        path = []
        m = acc
        while m >= 0:
            path.append(m)
            m = par[m]
        rows = list(inp["conv_cache"][0, s]) + [bf16_to_f32(inp["x"][0, 0, p]) for p in path[::-1]]
        expect = np.stack(rows[-(K - 1):]).astype(np.float32)
        got = oracle.persist_conv_lb(w.N, w.C, K, inp["x"][0, 0], inp["conv_cache"][0, s], par, acc)
        np.testing.assert_array_equal(got.view(np.uint32), expect.view(np.uint32))


def test_unfused_persist_copies_snapshot_and_leaves_other_slots():
    w = small_workload(seed=61)
    inp = make_inputs(w, slots=np.array([3, 1], dtype=np.int32))
    ns = RNG.standard_normal((w.L, w.Bq, w.N, w.Hv, w.d, w.d)).astype(np.float32)
    state, cache = oracle.tree_persist(w, inp, ns)
    for l in range(w.L):
        for b in range(w.Bq):
            s = inp["slot"][b]
            np.testing.assert_array_equal(state[l, s], ns[l, b, inp["accepted"][b]])
        for s in set(range(w.n_slots)) - set(inp["slot"].tolist()):
            assert state[l, s].tobytes() == inp["state"][l, s].tobytes()
            assert cache[l, s].tobytes() == inp["conv_cache"][l, s].tobytes()


# --------------------------------------------------------------------------
# Error reporting.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("parent,ok", [
    ([-1, 0, 1, 1], True),
    ([0, 0, 1, 1], False),       # root must have parent -1
    ([-1, 0, 2, 1], False),      # parent must precede the node
    ([-1, 0, -1, 1], False),     # only node 0 is a root
    ([-1, 0, 1, 7], False),      # out of range
])
def test_tree_validation(parent, ok):
    rc = oracle.check_tree(np.array(parent, dtype=np.int32))
    assert (rc == oracle.OK) == ok


def test_bad_slot_and_accepted_are_rejected():
    w = small_workload(L=1, Bq=1, seed=71)
    inp = make_inputs(w)
    bad = dict(inp)
    bad["slot"] = np.array([w.n_slots], dtype=np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.verify_heads(w, bad, [(0, 0, 0)])
    bad = dict(inp)
    bad["accepted"] = np.array([w.N], dtype=np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.verify_heads(w, bad, [(0, 0, 0)])
