"""Pins of the oracle's DDTree construction (best first by summed draft
log-probability, budget B).

The pages (Lucebox hub README: DDTree in "Algorithms used", budget 22 in
"Implemented here", the draft's per-position top-K in "GPU draft top-K &
verify-argmax (DFlash)") print no construction rule or example.  The oracle is
pinned to a hand-worked example, to brute force over every node of small
tries (the tree must be the B-1 highest-scoring nodes), to closed forms (K =
1 gives a chain; a budget above the trie size takes the whole trie) and to
invariants (topological numbering, depth and score of every node from its
parent, non-increasing scores in selection order).
"""
import itertools

import numpy as np
import pytest

import oracle


def rand_scores(rng, Bq, D, K, V=1000):
    p = rng.dirichlet(np.ones(K + 2), size=(Bq, D))[..., :K]
    p = -np.sort(-p, axis=-1)  # top-K, descending
    logp = np.log(p).astype(np.float32)
    tok = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(D)])
                    for _ in range(Bq)]).astype(np.int32)
    return logp, tok


def test_hand_worked_example():
    """p = [0.6, 0.3, 0.1] at position 1, [0.5, 0.4, 0.1] at position 2.
    Root; then 0.6 (token 10).  Next the candidates 0.3 (token 11 under the
    root) and 0.6 * 0.5 = 0.3 (token 20 under node 1) tie in fp32: the lower
    parent wins, token 11.  Then 0.3 (token 20 under node 1), 0.24 (token
    21 under node 1) and 0.15 (token 20 under node 2)."""
    lp = np.log(np.array([[[0.6, 0.3, 0.1], [0.5, 0.4, 0.1]]], dtype=np.float32))
    tk = np.array([[[10, 11, 12], [20, 21, 22]]], dtype=np.int32)
    par, tn, dp, sc, nn = oracle.ddtree_build(lp, tk, np.array([7], np.int32), 6)
    assert nn.tolist() == [6]
    assert par.tolist() == [[-1, 0, 0, 1, 1, 2]]
    assert tn.tolist() == [[7, 10, 11, 20, 21, 20]]
    assert dp.tolist() == [[0, 1, 1, 2, 2, 2]]
    assert np.allclose(np.exp(sc[0]), [1.0, 0.6, 0.3, 0.3, 0.24, 0.15], rtol=1e-6)


@pytest.mark.parametrize("D,K,B", [(3, 3, 12), (4, 2, 9), (2, 4, 14), (5, 2, 22)])
def test_brute_force_top_scores(D, K, B):
    """Every node of the trie scored (fp32, root down); the tree's non-root
    nodes are exactly the B-1 best (continuous random scores: no ties)."""
    rng = np.random.default_rng(10 + D * 7 + K)
    logp, tok = rand_scores(rng, 1, D, K)
    nodes = {}
    for d in range(1, D + 1):
        for ks in itertools.product(range(K), repeat=d):
            s = np.float32(0.0)
            for j, k in enumerate(ks):
                s = np.float32(s + logp[0, j, k])
            nodes[ks] = s
    best = sorted(nodes, key=lambda ks: -nodes[ks])[:B - 1]
    par, tn, dp, sc, nn = oracle.ddtree_build(logp, tok, np.array([0], np.int32), B)
    got = set()
    for i in range(1, nn[0]):
        ks, v = [], i
        while v != 0:
            d = dp[0, v] - 1
            ks.append(int(np.flatnonzero(tok[0, d] == tn[0, v])[0]))
            v = par[0, v]
        got.add(tuple(reversed(ks)))
    assert got == set(best)
    assert nn[0] == min(B, 1 + len(nodes))


def test_chain_and_whole_trie():
    rng = np.random.default_rng(11)
    logp, tok = rand_scores(rng, 2, 6, 1)
    par, tn, dp, _, nn = oracle.ddtree_build(logp, tok, np.array([5, 6], np.int32), 22)
    assert nn.tolist() == [7, 7]  # K = 1: a chain of D + 1 nodes
    assert par[0, :7].tolist() == [-1, 0, 1, 2, 3, 4, 5]
    assert (par[:, 7:] == -1).all() and (tn[:, 7:] == -1).all()
    logp, tok = rand_scores(rng, 1, 3, 3)
    *_, nn = oracle.ddtree_build(logp, tok, np.array([0], np.int32), 64)
    assert nn[0] == 1 + 3 + 9 + 27  # the whole trie


def test_invariants_budget22():
    rng = np.random.default_rng(12)
    Bq, D, K, B = 6, 16, 8, 22
    logp, tok = rand_scores(rng, Bq, D, K, V=150000)
    rt = rng.integers(0, 150000, Bq).astype(np.int32)
    par, tn, dp, sc, nn = oracle.ddtree_build(logp, tok, rt, B)
    assert (nn == B).all()
    for b in range(Bq):
        assert tn[b, 0] == rt[b] and par[b, 0] == -1 and dp[b, 0] == 0 and sc[b, 0] == 0
        for i in range(1, B):
            p = par[b, i]
            assert 0 <= p < i
            assert dp[b, i] == dp[b, p] + 1
            k = int(np.flatnonzero(tok[b, dp[b, p]] == tn[b, i])[0])
            assert sc[b, i] == np.float32(sc[b, p] + logp[b, dp[b, p], k])
            assert sc[b, i] <= sc[b, i - 1]
        # no two nodes share (parent, token)
        pairs = set(zip(par[b, 1:].tolist(), tn[b, 1:].tolist()))
        assert len(pairs) == B - 1
