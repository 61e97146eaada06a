"""Pins of the oracle's verify argmax and greedy acceptance walk.

The pages (Lucebox hub README, "GPU draft top-K & verify-argmax (DFlash)")
say the target's per-node argmax decides acceptance and that greedy decoding
is the high-acceptance mode; they print no worked example.  The oracle's
argmax is pinned to numpy's library routines (argmax, nanargmax) on the cases
where the definitions coincide, and the walk to a hand-worked example, to a
closed form on chains, to brute force over every root path of small trees
whose siblings carry distinct tokens, and to the invariants that determine
the walk's result uniquely.
"""
import numpy as np
import pytest

import oracle


def rand_tree(rng, N, max_children=None):
    parent = np.full(N, -1, dtype=np.int32)
    kids = np.zeros(N, dtype=np.int64)
    for i in range(1, N):
        while True:
            p = int(rng.integers(0, i))
            if max_children is None or kids[p] < max_children:
                break
        parent[i] = p
        kids[p] += 1
    return parent


def test_hand_worked_example():
    """Rows: [0,3,3,1] -> the tie at 3 goes to index 1; [5,1,1,1] -> 0;
    [0,0,0,9] -> 3; [1,2,3,4] -> 3.  Tree 0 -> 1 -> {2, 3}.  From the root
    the target chooses 1 and node 1 carries token 1: accept 1.  At node 1 it
    chooses 0; children 2 (token 0) and 3 (token 3): accept 2.  Node 2 has no
    children: stop at 2, next token = choice at 2 = 3."""
    lg = np.array([[[0, 3, 3, 1], [5, 1, 1, 1], [0, 0, 0, 9], [1, 2, 3, 4]]], dtype=np.float32)
    dr = np.array([[7, 1, 0, 3]], dtype=np.int32)
    pa = np.array([[-1, 0, 1, 1]], dtype=np.int32)
    am, acc, nxt = oracle.accept_walk(lg, dr, pa)
    assert am.tolist() == [[1, 0, 3, 3]]
    assert acc.tolist() == [2] and nxt.tolist() == [3]


def test_argmax_is_numpy_argmax_with_ties():
    """Finite rows with many ties (small integer values): numpy's argmax
    returns the first maximal index, the oracle's rule on finite rows."""
    rng = np.random.default_rng(3)
    lg = rng.integers(-3, 4, size=(3, 9, 257)).astype(np.float32)
    lg[0, 0] = 2.0  # a whole row of equal values
    lg[1, 2, :] = -np.inf
    am, _, _ = oracle.accept_walk(lg, np.zeros((3, 9), np.int32),
                                  np.tile(rand_tree(rng, 9), (3, 1)))
    assert np.array_equal(am, np.argmax(lg, axis=-1))


def test_argmax_nan_is_numpy_nanargmax():
    """NaN ranks below every number: on rows with a number the choice is
    numpy's nanargmax (first maximal non-NaN index); an all-NaN row gives 0."""
    rng = np.random.default_rng(4)
    lg = rng.normal(size=(2, 6, 100)).astype(np.float32)
    mask = rng.random(lg.shape) < 0.3
    lg[mask] = np.nan
    lg[0, 1, :50] = np.nan
    lg[0, 1, 50:] = -np.inf
    lg[1, 3, :] = np.nan
    am, _, _ = oracle.accept_walk(lg, np.zeros((2, 6), np.int32),
                                  np.tile(rand_tree(rng, 6), (2, 1)))
    for b in range(2):
        for n in range(6):
            row = lg[b, n]
            if (b, n) == (0, 1):
                # NaN ranks below -inf too: the first -inf (index 50) wins;
                # numpy's nanargmax, which maps NaN to -inf, would give 0
                want = 50
            else:
                want = 0 if np.isnan(row).all() else int(np.nanargmax(row))
            assert am[b, n] == want, (b, n)


def test_chain_closed_form():
    """On a chain the walk accepts the longest prefix whose every token
    matches the target's choice one position earlier."""
    rng = np.random.default_rng(5)
    Bq, N, V = 8, 12, 5
    lg = rng.normal(size=(Bq, N, V)).astype(np.float32)
    am = np.argmax(lg, axis=-1)
    dr = rng.integers(0, V, size=(Bq, N)).astype(np.int32)
    # plant matching prefixes of varied length
    for b in range(Bq):
        m = int(rng.integers(0, N))
        dr[b, 1:m + 1] = am[b, :m]
    pa = np.tile(np.arange(-1, N - 1, dtype=np.int32), (Bq, 1))
    _, acc, nxt = oracle.accept_walk(lg, dr, pa)
    match = (dr[:, 1:] == am[:, :-1]).astype(np.int64)
    want = np.cumprod(match, axis=1).sum(axis=1)
    assert np.array_equal(acc, want)
    assert np.array_equal(nxt, am[np.arange(Bq), want])


def test_brute_force_distinct_siblings():
    """Siblings with distinct tokens (as in a draft tree of top-K children):
    at most one child of a node can match, so the accepted node is the
    deepest node whose whole root path matches, found by trying every node."""
    rng = np.random.default_rng(6)
    for trial in range(40):
        N, V = int(rng.integers(1, 14)), 6
        pa = rand_tree(rng, N, max_children=V)
        lg = rng.normal(size=(1, N, V)).astype(np.float32)
        am = np.argmax(lg[0], axis=-1)
        dr = np.zeros(N, dtype=np.int32)
        for u in range(N):
            kids = [c for c in range(N) if pa[c] == u]
            toks = rng.permutation(V)[:len(kids)]
            # bias toward a match so that paths grow
            if kids and rng.random() < 0.7:
                toks[int(rng.integers(0, len(kids)))] = -1
                toks = np.where(toks == -1, am[u], toks)
                if len(set(toks.tolist())) < len(kids):
                    toks = rng.permutation(V)[:len(kids)]
            for c, t in zip(kids, toks):
                dr[c] = t
        best, best_depth = 0, 0
        for n in range(N):
            ok, depth, v = True, 0, n
            while v != 0:
                if dr[v] != am[pa[v]]:
                    ok = False
                    break
                v, depth = pa[v], depth + 1
            if ok and depth > best_depth:
                best, best_depth = n, depth
        _, acc, nxt = oracle.accept_walk(lg, dr[None], pa[None])
        assert acc[0] == best, trial
        assert nxt[0] == am[best]


def test_walk_invariants_random_trees():
    """The result is the unique node reached by: every edge on its root path
    matches (token of the child = choice at the parent), each edge takes the
    lowest-index matching child, and no child of it matches."""
    rng = np.random.default_rng(7)
    Bq, N, V = 16, 22, 4  # few tokens: many sibling collisions
    lg = rng.normal(size=(Bq, N, V)).astype(np.float32)
    pa = np.stack([rand_tree(rng, N) for _ in range(Bq)])
    dr = rng.integers(0, V, size=(Bq, N)).astype(np.int32)
    am, acc, nxt = oracle.accept_walk(lg, dr, pa)
    assert np.array_equal(am, np.argmax(lg, axis=-1))
    for b in range(Bq):
        path = [int(acc[b])]
        while path[-1] != 0:
            path.append(int(pa[b, path[-1]]))
        path.reverse()
        for u, c in zip(path[:-1], path[1:]):
            assert dr[b, c] == am[b, u]
            assert not any(pa[b, c2] == u and dr[b, c2] == am[b, u] for c2 in range(c))
        a = int(acc[b])
        assert not any(pa[b, c] == a and dr[b, c] == am[b, a] for c in range(N))
        assert nxt[b] == am[b, a]


def test_invalid_tree_rejected():
    lg = np.zeros((1, 3, 4), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.accept_walk(lg, np.zeros((1, 3), np.int32), np.array([[-1, 2, 0]], np.int32))
