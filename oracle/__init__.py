"""fp64 CPU oracle for the tree-verify gated-DeltaNet step -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
may import this package.  The product (the CUDA library and its binding)
never imports, links or runs it, and it shares no code with the product.

The arithmetic lives in ``lbx_oracle.c`` (plain C, double precision); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lbx_oracle.c")
_LIB = os.path.join(_HERE, "liblbx_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ETREE, ENOMEM = 0, -1, -3, -4
FORM_PATH, FORM_MATRIX, FORM_SEQUENTIAL = 0, 1, 2


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no arch-specific flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
                        "-o", tmp, _SRC, "-lm", "-lpthread"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int), ("Bq", ctypes.c_int), ("N", ctypes.c_int),
                ("Hk", ctypes.c_int), ("Hv", ctypes.c_int), ("d", ctypes.c_int),
                ("K", ctypes.c_int), ("n_slots", ctypes.c_int),
                ("l2_eps", ctypes.c_double), ("q_scale", ctypes.c_double)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            for name in ("lbxo_check_tree", "lbxo_conv_lb", "lbxo_tree_conv",
                         "lbxo_deltanet_head", "lbxo_persist_conv_lb", "lbxo_verify_heads",
                         "lbxo_tree_deltanet", "lbxo_tree_persist", "lbxo_accept_walk",
                         "lbxo_ddtree_build", "lbxo_tree_attention"):
                getattr(_lib, name).restype = ctypes.c_int
        return _lib


def _p(arr: Optional[np.ndarray]):
    if arr is None:
        return None
    assert arr.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(arr.ctypes.data)


def _check(rc: int, what: str):
    if rc != OK:
        raise OracleError(f"{what} returned {rc}")


def cfg_of(w, L=None, Bq=None, N=None, n_slots=None) -> _Cfg:
    """ctypes config from a Workload (optionally overriding sizes)."""
    return _Cfg(L=w.L if L is None else L, Bq=w.Bq if Bq is None else Bq,
                N=w.N if N is None else N, Hk=w.Hk, Hv=w.Hv, d=w.d, K=w.K,
                n_slots=w.n_slots if n_slots is None else n_slots,
                l2_eps=w.l2_eps, q_scale=w.q_scale)


def check_tree(parent: np.ndarray) -> int:
    p = np.ascontiguousarray(parent, dtype=np.int32)
    return lib().lbxo_check_tree(_p(p), ctypes.c_int(p.shape[0]))


def tree_conv(w, inp: dict, lb_mask: Optional[np.ndarray] = None) -> np.ndarray:
    """conv+SiLU+L2 for the whole batch -> float64 [L][Bq][N][C]."""
    cfg = cfg_of(w)
    out = np.zeros((w.L, w.Bq, w.N, w.C), dtype=np.float64)
    m = None if lb_mask is None else np.ascontiguousarray(lb_mask, dtype=np.uint8)
    _check(lib().lbxo_tree_conv(ctypes.byref(cfg), _p(inp["x"]), _p(inp["conv_w"]),
                                _p(inp["conv_cache"]), _p(inp["parent"]), _p(inp["slot"]),
                                _p(m), _p(out)), "lbxo_tree_conv")
    return out


def conv_lb(N, Hk, Hv, d, K, l2_eps, x_lb, w_l, cache, parent) -> np.ndarray:
    C = 2 * Hk * d + Hv * d
    out = np.zeros((N, C), dtype=np.float64)
    x_lb = np.ascontiguousarray(x_lb, dtype=np.uint16)
    w_l = np.ascontiguousarray(w_l, dtype=np.uint16)
    cache = np.ascontiguousarray(cache, dtype=np.float32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    _check(lib().lbxo_conv_lb(N, Hk, Hv, d, K, ctypes.c_double(l2_eps), _p(x_lb), _p(w_l),
                              _p(cache), _p(parent), _p(out)), "lbxo_conv_lb")
    return out


def deltanet_head(N, Hk, Hv, d, h, q_scale, form, qkv_lb, a_lb, b_lb, S0, parent,
                  accepted=-1, want_states=False):
    """Recurrence of one head.  Returns (o [N][d], node_states [N][d][d] or
    None, S_acc [d][d] or None)."""
    o = np.zeros((N, d), dtype=np.float64)
    ns = np.zeros((N, d, d), dtype=np.float64) if want_states else None
    sacc = np.zeros((d, d), dtype=np.float64) if accepted >= 0 else None
    args = [np.ascontiguousarray(qkv_lb, dtype=np.float64),
            np.ascontiguousarray(a_lb, dtype=np.uint16),
            np.ascontiguousarray(b_lb, dtype=np.uint16),
            np.ascontiguousarray(S0, dtype=np.float32),
            np.ascontiguousarray(parent, dtype=np.int32)]
    _check(lib().lbxo_deltanet_head(N, Hk, Hv, d, h, ctypes.c_double(q_scale), form,
                                    *[_p(x) for x in args], int(accepted), _p(o), _p(ns),
                                    _p(sacc)), "lbxo_deltanet_head")
    return o, ns, sacc


def tree_deltanet(w, qkv: np.ndarray, inp: dict, form: int = FORM_PATH,
                  want_states: bool = False):
    """Whole-batch recurrence from a conv output.  Returns (o, node_states)."""
    cfg = cfg_of(w)
    o = np.zeros((w.L, w.Bq, w.N, w.Hv, w.d), dtype=np.float64)
    ns = (np.zeros((w.L, w.Bq, w.N, w.Hv, w.d, w.d), dtype=np.float64)
          if want_states else None)
    qkv = np.ascontiguousarray(qkv, dtype=np.float64)
    _check(lib().lbxo_tree_deltanet(ctypes.byref(cfg), _p(qkv), _p(inp["a"]), _p(inp["b"]),
                                    _p(inp["state"]), _p(inp["parent"]), _p(inp["slot"]),
                                    form, _p(o), _p(ns)), "lbxo_tree_deltanet")
    return o, ns


def verify_heads(w, inp: dict, items: Sequence[Sequence[int]], form: int = FORM_PATH,
                 want_o: bool = True, want_state: bool = True, n_threads: int = 0):
    """Full verify step for a list of (layer, request, value head) items.

    Returns (o [n][N][d] or None, S_acc [n][d][d] or None, threads_used)."""
    it = np.ascontiguousarray(np.asarray(items, dtype=np.int32).reshape(-1, 3))
    n = it.shape[0]
    o = np.zeros((n, w.N, w.d), dtype=np.float64) if want_o else None
    s = np.zeros((n, w.d, w.d), dtype=np.float64) if want_state else None
    used = ctypes.c_int(0)
    cfg = cfg_of(w)
    _check(lib().lbxo_verify_heads(ctypes.byref(cfg), _p(inp["x"]), _p(inp["conv_w"]),
                                   _p(inp["a"]), _p(inp["b"]), _p(inp["state"]),
                                   _p(inp["conv_cache"]), _p(inp["parent"]), _p(inp["slot"]),
                                   _p(inp["accepted"]), _p(it), n, form, _p(o), _p(s),
                                   int(n_threads), ctypes.byref(used)), "lbxo_verify_heads")
    return o, s, used.value


def persist_conv_lb(N, C, K, x_lb, cache_old, parent, accepted) -> np.ndarray:
    out = np.zeros((K - 1, C), dtype=np.float32)
    x_lb = np.ascontiguousarray(x_lb, dtype=np.uint16)
    cache_old = np.ascontiguousarray(cache_old, dtype=np.float32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    _check(lib().lbxo_persist_conv_lb(N, C, K, _p(x_lb), _p(cache_old), _p(parent),
                                      int(accepted), _p(out)), "lbxo_persist_conv_lb")
    return out


def tree_persist(w, inp: dict, node_states: np.ndarray):
    """Unfused persist from fp32 snapshots; returns (state, conv_cache) copies."""
    cfg = cfg_of(w)
    state = inp["state"].copy()
    cache = inp["conv_cache"].copy()
    ns = np.ascontiguousarray(node_states, dtype=np.float32)
    _check(lib().lbxo_tree_persist(ctypes.byref(cfg), _p(inp["x"]), _p(ns), _p(inp["parent"]),
                                   _p(inp["slot"]), _p(inp["accepted"]), _p(state), _p(cache)),
           "lbxo_tree_persist")
    return state, cache


def verify_step_full(w, inp: dict, form: int = FORM_PATH, n_threads: int = 0):
    """Every head of a (small) workload: returns (o [L][Bq][N][Hv][d],
    new_state float64 [L][n_slots][Hv][d][d] (persisted slots replaced,
    others widened from the input), new_conv_cache float32)."""
    items = [(l, b, h) for l in range(w.L) for b in range(w.Bq) for h in range(w.Hv)]
    o_it, s_it, _ = verify_heads(w, inp, items, form=form, n_threads=n_threads)
    o = np.zeros((w.L, w.Bq, w.N, w.Hv, w.d), dtype=np.float64)
    state = inp["state"].astype(np.float64)
    for i, (l, b, h) in enumerate(items):
        o[l, b, :, h, :] = o_it[i]
        state[l, inp["slot"][b], h] = s_it[i]
    cache = inp["conv_cache"].copy()
    for l in range(w.L):
        for b in range(w.Bq):
            s = inp["slot"][b]
            cache[l, s] = persist_conv_lb(w.N, w.C, w.K, inp["x"][l, b], inp["conv_cache"][l, s],
                                          inp["parent"][b], inp["accepted"][b])
    return o, state, cache


def accept_walk(logits: np.ndarray, draft: np.ndarray, parent: np.ndarray):
    """Verify argmax and greedy acceptance walk (see lbx_oracle.c).

    logits float32 [Bq][N][V], draft and parent int32 [Bq][N].  Returns
    (argmax int32 [Bq][N], accepted int32 [Bq], next int32 [Bq])."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    Bq, N, V = lg.shape
    dr = np.ascontiguousarray(draft, dtype=np.int32).reshape(Bq, N)
    pa = np.ascontiguousarray(parent, dtype=np.int32).reshape(Bq, N)
    am = np.zeros((Bq, N), dtype=np.int32)
    acc = np.zeros(Bq, dtype=np.int32)
    nxt = np.zeros(Bq, dtype=np.int32)
    _check(lib().lbxo_accept_walk(ctypes.c_int(Bq), ctypes.c_int(N), ctypes.c_int(V), _p(lg),
                                  _p(dr), _p(pa), _p(am), _p(acc), _p(nxt)), "lbxo_accept_walk")
    return am, acc, nxt


def ddtree_build(logp: np.ndarray, tok: np.ndarray, root_tok: np.ndarray, B: int):
    """DDTree construction from draft top-K scores (see lbx_oracle.c).

    logp float32 [Bq][D][K], tok int32 [Bq][D][K], root_tok int32 [Bq].
    Returns (parent, token, depth int32 [Bq][B], score float32 [Bq][B],
    n_nodes int32 [Bq])."""
    lp = np.ascontiguousarray(logp, dtype=np.float32)
    Bq, D, K = lp.shape
    tk = np.ascontiguousarray(tok, dtype=np.int32).reshape(Bq, D, K)
    rt = np.ascontiguousarray(root_tok, dtype=np.int32).reshape(Bq)
    par = np.zeros((Bq, B), np.int32)
    tn = np.zeros((Bq, B), np.int32)
    dp = np.zeros((Bq, B), np.int32)
    sc = np.zeros((Bq, B), np.float32)
    nn = np.zeros(Bq, np.int32)
    _check(lib().lbxo_ddtree_build(ctypes.c_int(Bq), ctypes.c_int(D), ctypes.c_int(K),
                                   ctypes.c_int(B), _p(lp), _p(tk), _p(rt), _p(par), _p(tn),
                                   _p(dp), _p(sc), _p(nn)), "lbxo_ddtree_build")
    return par, tn, dp, sc, nn


def tree_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, k_tree: np.ndarray,
                   v_tree: np.ndarray, ctx_len: np.ndarray, parent: np.ndarray,
                   scale: float) -> np.ndarray:
    """Tree-masked attention of the full-attention layers (see lbx_oracle.c).

    q uint16 (bf16 bits) [L][Bq][N][Hq][dh]; k_cache, v_cache [L][Bq][T][Hkv][dh];
    k_tree, v_tree [L][Bq][N][Hkv][dh]; ctx_len int32 [Bq]; parent int32
    [Bq][N].  Returns o float64 [L][Bq][N][Hq][dh]."""
    L, Bq, N, Hq, dh = q.shape
    T, Hkv = k_cache.shape[2], k_cache.shape[3]
    arrs = [np.ascontiguousarray(a, dtype=np.uint16) for a in (q, k_cache, v_cache, k_tree, v_tree)]
    cl = np.ascontiguousarray(ctx_len, dtype=np.int32).reshape(Bq)
    pa = np.ascontiguousarray(parent, dtype=np.int32).reshape(Bq, N)
    o = np.zeros((L, Bq, N, Hq, dh), dtype=np.float64)
    _check(lib().lbxo_tree_attention(ctypes.c_int(L), ctypes.c_int(Bq), ctypes.c_int(N),
                                     ctypes.c_int(Hq), ctypes.c_int(Hkv), ctypes.c_int(dh),
                                     ctypes.c_int(T), _p(cl), ctypes.c_double(scale),
                                     *[_p(a) for a in arrs], _p(pa), _p(o)),
           "lbxo_tree_attention")
    return o
