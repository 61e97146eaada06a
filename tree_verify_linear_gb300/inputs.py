"""Seeded synthetic inputs for the tree-verify gated-DeltaNet step.

This module is shared by the CUDA path's tests/bench and by the fp64 oracle's
tests. It only draws random numbers and lays them out; it holds none of the
method's arithmetic (no conv, no normalisation, no recurrence).

Shapes and distributions follow the workloads described for the DDTree verify
step of a 27B-class hybrid target (Lucebox hub README, section "02 DFlash
DDtree": budget 22 as the RTX 3090 sweet spot, tree-structured verify) and the
tiny / serving / long-chain variants of the same layer shapes:

* ``x`` (pre-conv q|k|v inputs) ~ N(0, 1), rounded to bf16.
* ``conv_cache`` (K-1 prior raw inputs per channel) ~ N(0, 1), fp32.
* ``conv_w`` ~ N(0, 1/K), rounded to bf16 (separate per layer).
* gates: ``a = exp(-softplus(z))``, ``b = sigmoid(z)``, z ~ N(0, 1), each
  drawn independently and rounded to bf16 (the gates are given already
  activated).
* initial recurrent state ~ N(0, 0.1^2), fp32.
* draft tree: parent-index array with ``parent[0] = -1`` and
  ``parent[i] < i``.  "uniform": parent[i] uniform on [0, i).  "ddtree":
  parent[i] drawn over nodes j < i with weight 2^-depth(j), restricted to
  depth(j) <= 8 (root-to-node paths of at most 10 nodes), optionally with at
  most ``max_children`` children per node.  "chain": parent[i] = i - 1.
* accepted node: "leaf" (random leaf), "node" (uniform random node), "last",
  "root".
* slots: request b uses cache slot ``slot[b]``; the pool has ``spare_slots``
  extra slots that no request names, filled with a canary byte pattern.

bf16 values are carried as ``uint16`` bit patterns.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# Canary bit pattern written to every cache slot no request names.  It is a
# quiet NaN, so a kernel that reads it by mistake also poisons its outputs.
CANARY_U32 = 0x7FC0DEAD


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one verify step (one batch of draft trees)."""

    name: str
    L: int            # gated-DeltaNet layers
    Bq: int           # requests in the batch
    N: int            # draft-tree nodes (budget) / chain length
    Hk: int           # key heads
    Hv: int           # value heads
    d: int            # d_k = d_v
    K: int = 4        # conv width
    tree: str = "ddtree"          # uniform | ddtree | chain
    accepted: str = "node"        # leaf | node | last | root
    max_children: Optional[int] = None
    max_parent_depth: int = 8
    spare_slots: int = 2
    seed: int = 1000
    l2_eps: float = 1e-6
    q_scale: float = 1.0

    @property
    def C(self) -> int:
        """Conv channels, ordered q | k | v."""
        return 2 * self.Hk * self.d + self.Hv * self.d

    @property
    def n_slots(self) -> int:
        return self.Bq + self.spare_slots

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the verify step (plus the budget-64 serving variant).
WORKLOADS = {
    "tiny": Workload("tiny", L=1, Bq=1, N=8, Hk=2, Hv=4, d=32,
                     tree="uniform", accepted="leaf", seed=1001),
    "layer27b": Workload("layer27b", L=1, Bq=1, N=22, Hk=16, Hv=48, d=128,
                         seed=1002),
    "step27b": Workload("step27b", L=48, Bq=1, N=22, Hk=16, Hv=48, d=128,
                        seed=1003),
    "serve27b_b22": Workload("serve27b_b22", L=48, Bq=5, N=22, Hk=16, Hv=48,
                             d=128, seed=1004),
    "serve27b_b64": Workload("serve27b_b64", L=48, Bq=5, N=64, Hk=16, Hv=48,
                             d=128, max_children=4, seed=1004),
    "chain08b": Workload("chain08b", L=18, Bq=1, N=4096, Hk=16, Hv=16, d=128,
                         tree="chain", accepted="last", seed=1005),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even).

    Returns the bf16 bit patterns as uint16.  Inputs here are finite.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, *key]))


def make_tree(rng: np.random.Generator, N: int, kind: str,
              max_parent_depth: int = 8,
              max_children: Optional[int] = None) -> np.ndarray:
    """Draw a topologically numbered parent-index array (parent[0] = -1)."""
    parent = np.full(N, -1, dtype=np.int32)
    if kind == "chain":
        parent[1:] = np.arange(N - 1, dtype=np.int32)
        return parent
    depth = np.zeros(N, dtype=np.int64)
    nchild = np.zeros(N, dtype=np.int64)
    for i in range(1, N):
        if kind == "uniform":
            j = int(rng.integers(0, i))
        elif kind == "ddtree":
            cand = np.arange(i)
            ok = depth[:i] <= max_parent_depth
            if max_children is not None:
                ok &= nchild[:i] < max_children
            cand = cand[ok]
            w = np.exp2(-depth[cand].astype(np.float64))
            j = int(rng.choice(cand, p=w / w.sum()))
        else:
            raise ValueError(f"unknown tree kind {kind!r}")
        parent[i] = j
        depth[i] = depth[j] + 1
        nchild[j] += 1
    return parent


def pick_accepted(rng: np.random.Generator, parent: np.ndarray, kind: str) -> int:
    N = parent.shape[0]
    if kind == "last":
        return N - 1
    if kind == "root":
        return 0
    if kind == "node":
        return int(rng.integers(0, N))
    if kind == "leaf":
        has_child = np.zeros(N, dtype=bool)
        has_child[parent[1:]] = True
        leaves = np.flatnonzero(~has_child)
        return int(leaves[rng.integers(0, leaves.shape[0])])
    raise ValueError(f"unknown accepted kind {kind!r}")


def make_inputs(w: Workload, seed: Optional[int] = None,
                slots: Optional[np.ndarray] = None) -> dict:
    """Generate every input of one verify step for workload ``w``.

    Returns a dict of numpy arrays:
      x          uint16 (bf16) [L][Bq][N][C]
      conv_w     uint16 (bf16) [L][C][K]
      conv_cache float32       [L][n_slots][K-1][C]
      a, b       uint16 (bf16) [L][Bq][N][Hv]
      state      float32       [L][n_slots][Hv][d][d]   (row = value dim)
      parent     int32         [Bq][N]
      slot       int32         [Bq]
      accepted   int32         [Bq]
    Slots no request names hold the canary pattern.
    """
    seed = w.seed if seed is None else seed
    L, Bq, N, Hv, d, K, C = w.L, w.Bq, w.N, w.Hv, w.d, w.K, w.C
    S = w.n_slots

    parent = np.empty((Bq, N), dtype=np.int32)
    accepted = np.empty(Bq, dtype=np.int32)
    for b in range(Bq):
        r = _rng(seed, 1, b, N)
        parent[b] = make_tree(r, N, w.tree, w.max_parent_depth, w.max_children)
        accepted[b] = pick_accepted(r, parent[b], w.accepted)

    if slots is None:
        slots = np.arange(Bq, dtype=np.int32)
    slots = np.asarray(slots, dtype=np.int32)

    x = np.empty((L, Bq, N, C), dtype=np.uint16)
    a = np.empty((L, Bq, N, Hv), dtype=np.uint16)
    bg = np.empty((L, Bq, N, Hv), dtype=np.uint16)
    conv_w = np.empty((L, C, K), dtype=np.uint16)
    canary = np.uint32(CANARY_U32)
    conv_cache = np.full((L, S, K - 1, C), canary, dtype=np.uint32).view(np.float32)
    state = np.full((L, S, Hv, d, d), canary, dtype=np.uint32).view(np.float32)

    for l in range(L):
        r = _rng(seed, 2, l)
        conv_w[l] = bf16_bits(r.standard_normal((C, K), dtype=np.float32)
                              * np.float32(1.0 / np.sqrt(K)))
        for b in range(Bq):
            r = _rng(seed, 3, l, b, N)
            x[l, b] = bf16_bits(r.standard_normal((N, C), dtype=np.float32))
            za = r.standard_normal((N, Hv))
            zb = r.standard_normal((N, Hv))
            a[l, b] = bf16_bits(np.exp(-np.logaddexp(0.0, za)).astype(np.float32))
            bg[l, b] = bf16_bits((1.0 / (1.0 + np.exp(-zb))).astype(np.float32))
            s = int(slots[b])
            conv_cache[l, s] = r.standard_normal((K - 1, C), dtype=np.float32)
            state[l, s] = r.standard_normal((Hv, d, d), dtype=np.float32) * np.float32(0.1)

    return dict(x=x, conv_w=conv_w, conv_cache=conv_cache, a=a, b=bg,
                state=state, parent=parent, slot=slots, accepted=accepted)


# ---- acceptance walk inputs -------------------------------------------------

# Vocabulary of the synthetic target: a 152K-entry vocabulary, the size class
# of the 27B target's tokenizer (the pages give no figure).
ACCEPT_VOCAB = 152064


def make_accept_inputs(Bq: int, N: int, V: int, seed: int, tree: str = "ddtree",
                       p_plant: float = 0.7, ties: bool = False) -> dict:
    """Seeded inputs of the verify argmax / acceptance walk.

    logits ~ N(0, 1) fp32 [Bq][N][V]; draft tokens uniform on [0, V) with
    distinct siblings (while V allows); trees as for the verify step.  To make acceptance
    paths longer than chance, for a fraction p_plant of the nodes one child's
    draft token is planted as the node's top score (logit 8 + U(0,1), above
    any N(0, 1) draw at these sizes); with ``ties`` a second child gets the
    same planted value at another token (the lower token index then wins)."""
    rng = _rng(seed, 77)
    logits = rng.standard_normal((Bq, N, V), dtype=np.float32)
    draft = np.zeros((Bq, N), dtype=np.int32)
    parent = np.zeros((Bq, N), dtype=np.int32)
    for b in range(Bq):
        par = make_tree(rng, N, tree)
        parent[b] = par
        for u in range(N):
            kids = np.flatnonzero(par == u)
            if len(kids) == 0:
                continue
            # distinct siblings while the vocabulary allows it
            toks = rng.choice(V, size=len(kids), replace=len(kids) > V).astype(np.int32)
            draft[b, kids] = toks
            if rng.random() < p_plant:
                pick = int(rng.integers(0, len(kids)))
                val = np.float32(8.0 + rng.random())
                logits[b, u, toks[pick]] = val
                if ties and len(kids) > 1:
                    other = int((pick + 1) % len(kids))
                    logits[b, u, toks[other]] = val
    return {"logits": logits, "draft": draft, "parent": parent}


def make_draft_topk(Bq: int, D: int, K: int, V: int, seed: int) -> dict:
    """Seeded draft top-K scores for the DDTree construction: per request and
    position, K distinct tokens uniform on [0, V) and the log of K
    probabilities drawn as the top K of a Dirichlet(1) over K + 8 outcomes,
    sorted descending; root tokens uniform on [0, V)."""
    rng = _rng(seed, 88)
    p = rng.dirichlet(np.ones(K + 8), size=(Bq, D))
    p = -np.sort(-p, axis=-1)[..., :K]
    logp = np.log(p).astype(np.float32)
    tok = np.empty((Bq, D, K), dtype=np.int32)
    for b in range(Bq):
        for d in range(D):
            tok[b, d] = rng.choice(V, size=K, replace=False)
    root = rng.integers(0, V, size=Bq).astype(np.int32)
    return {"logp": logp, "tok": tok, "root_tok": root}


# ---- tree-masked attention inputs -------------------------------------------

@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """Shape of the tree-masked attention of the full-attention layers in one
    verify step.  The pages give no attention shapes; the 27B-class layer is
    taken as 24 query heads over 4 KV heads of dimension 256 (GQA groups of 6)."""

    name: str
    L: int            # full-attention layers (a batch dimension)
    Bq: int           # requests
    N: int            # draft-tree nodes
    Hq: int           # query heads
    Hkv: int          # KV heads
    dh: int           # head dimension
    T: int            # KV-cache capacity (positions)
    ctx: str = "full"  # full: ctx_len = T; ragged: uniform on [T/2, T], plus one 0 when Bq > 2
    tree: str = "ddtree"
    max_children: Optional[int] = None
    seed: int = 2000

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.dh))

    def replace(self, **kw) -> "AttnWorkload":
        return dataclasses.replace(self, **kw)


ATTN_WORKLOADS = {
    "attn_tiny": AttnWorkload("attn_tiny", L=1, Bq=3, N=8, Hq=4, Hkv=2, dh=256, T=40,
                              ctx="ragged", tree="uniform", seed=2001),
    "attn27b": AttnWorkload("attn27b", L=16, Bq=1, N=22, Hq=24, Hkv=4, dh=256, T=4096,
                            seed=2002),
    "attn27b_serve": AttnWorkload("attn27b_serve", L=16, Bq=5, N=22, Hq=24, Hkv=4, dh=256,
                                  T=8192, ctx="ragged", seed=2003),
}


def make_attn_inputs(w: AttnWorkload, seed: Optional[int] = None) -> dict:
    """Seeded inputs of the tree-masked attention: q, k, v ~ N(0, 1) rounded
    to bf16 (the configs' input distribution), as bit patterns; DDTree-shaped
    (or uniform / chain) trees as for the verify step; context lengths.

      q        uint16 [L][Bq][N][Hq][dh]
      k_cache  uint16 [L][Bq][T][Hkv][dh]    (v_cache alike)
      k_tree   uint16 [L][Bq][N][Hkv][dh]    (v_tree alike)
      ctx_len  int32  [Bq]
      parent   int32  [Bq][N]
    """
    s = w.seed if seed is None else seed
    rng = _rng(s, 99)
    L, Bq, N = w.L, w.Bq, w.N

    def normal(*shape):
        return bf16_bits(rng.standard_normal(shape, dtype=np.float32))

    q = normal(L, Bq, N, w.Hq, w.dh)
    k_cache = normal(L, Bq, w.T, w.Hkv, w.dh)
    v_cache = normal(L, Bq, w.T, w.Hkv, w.dh)
    k_tree = normal(L, Bq, N, w.Hkv, w.dh)
    v_tree = normal(L, Bq, N, w.Hkv, w.dh)
    if w.ctx == "full":
        ctx_len = np.full(Bq, w.T, dtype=np.int32)
    elif w.ctx == "ragged":
        ctx_len = rng.integers(w.T // 2, w.T + 1, size=Bq).astype(np.int32)
        if Bq > 2:
            ctx_len[1] = 0
    else:
        raise ValueError(f"unknown context kind {w.ctx!r}")
    parent = np.stack([make_tree(rng, N, w.tree, max_children=w.max_children)
                       for _ in range(Bq)]).astype(np.int32)
    return dict(q=q, k_cache=k_cache, v_cache=v_cache, k_tree=k_tree, v_tree=v_tree,
                ctx_len=ctx_len, parent=parent)
