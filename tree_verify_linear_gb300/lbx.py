"""Thin Python binding of the liblbx C ABI (include/lbx.h).

Argument marshalling only: every step of the verify path runs in the CUDA
kernels of liblbx.so.  The functions keep the C names and argument order and
take torch CUDA tensors (PyTorch supplies device memory and streams).  bf16
arguments may be ``torch.bfloat16`` or 16-bit integer tensors holding bf16 bit
patterns.  There is no CPU fallback: if the library cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblbx.so")

LBX_OK, LBX_EINVAL, LBX_ECUDA, LBX_ETREE, LBX_ETIMEOUT = 0, -1, -2, -3, -4
LBX_MAX_TREE_NODES = 64
LBX_CHAIN_CHUNK = 64
LBX_MAX_CONV_WIDTH = 4
LBX_MODE_AUTO, LBX_MODE_TREE, LBX_MODE_CHUNKED, LBX_MODE_TREE_CUDA_CORES = 0, 1, 2, 3

# Every function the header declares, in header order.
EXPORTS = ("lbx_strerror", "lbx_workspace_size", "lbx_tree_conv", "lbx_tree_deltanet",
           "lbx_tree_persist", "lbx_verify_step", "lbx_verify_step_noalloc",
           "lbx_accept_workspace_size", "lbx_accept_walk", "lbx_ddtree_build",
           "lbx_attn_workspace_size", "lbx_tree_attention")
LBX_ACCEPT_MAX_NODES = 4096
LBX_DDTREE_MAX_K, LBX_DDTREE_MAX_DEPTH = 8, 64
LBX_NOALLOC_MAX_GROUPS = 65536
LBX_ATTN_HEAD_DIM, LBX_ATTN_MAX_NODES = 256, 64


class LbxError(RuntimeError):
    def __init__(self, fn: str, rc: int):
        super().__init__(f"{fn} failed: {rc} ({strerror(rc)})")
        self.rc = rc


class lbx_cfg(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int), ("Bq", ctypes.c_int), ("N", ctypes.c_int),
                ("Hk", ctypes.c_int), ("Hv", ctypes.c_int), ("d", ctypes.c_int),
                ("K", ctypes.c_int), ("n_slots", ctypes.c_int), ("l2_eps", ctypes.c_float),
                ("q_scale", ctypes.c_float), ("mode", ctypes.c_int)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load liblbx.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"liblbx.so not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        lib.lbx_strerror.restype = ctypes.c_char_p
        lib.lbx_strerror.argtypes = [i32]
        lib.lbx_workspace_size.restype = ctypes.c_size_t
        lib.lbx_workspace_size.argtypes = [vp]
        lib.lbx_tree_conv.restype = i32
        lib.lbx_tree_conv.argtypes = [vp] * 9
        lib.lbx_tree_deltanet.restype = i32
        lib.lbx_tree_deltanet.argtypes = [vp] * 11
        lib.lbx_tree_persist.restype = i32
        lib.lbx_tree_persist.argtypes = [vp] * 10
        lib.lbx_verify_step.restype = i32
        lib.lbx_verify_step.argtypes = [vp] * 11 + [vp, ctypes.c_size_t, vp, vp]
        lib.lbx_verify_step_noalloc.restype = i32
        lib.lbx_verify_step_noalloc.argtypes = [vp] * 13
        lib.lbx_accept_workspace_size.restype = ctypes.c_size_t
        lib.lbx_accept_workspace_size.argtypes = [i32, i32, i32]
        lib.lbx_accept_walk.restype = i32
        lib.lbx_accept_walk.argtypes = [i32, i32, i32] + [vp] * 6 + [vp, ctypes.c_size_t, vp, vp]
        lib.lbx_ddtree_build.restype = i32
        lib.lbx_ddtree_build.argtypes = [i32, i32, i32, i32] + [vp] * 9
        lib.lbx_attn_workspace_size.restype = ctypes.c_size_t
        lib.lbx_attn_workspace_size.argtypes = [i32] * 7
        lib.lbx_tree_attention.restype = i32
        lib.lbx_tree_attention.argtypes = ([i32] * 7 + [ctypes.c_float] + [vp] * 8
                                           + [vp, ctypes.c_size_t, vp, vp])
        _lib = lib
    return _lib


def strerror(rc: int) -> str:
    return load().lbx_strerror(rc).decode()


def make_cfg(L, Bq, N, Hk, Hv, d, K=4, n_slots=None, l2_eps=1e-6, q_scale=1.0,
             mode=LBX_MODE_AUTO) -> lbx_cfg:
    return lbx_cfg(L=L, Bq=Bq, N=N, Hk=Hk, Hv=Hv, d=d, K=K,
                   n_slots=Bq if n_slots is None else n_slots, l2_eps=l2_eps, q_scale=q_scale,
                   mode=mode)


def cfg_of(w, mode=LBX_MODE_AUTO) -> lbx_cfg:
    """Config from an inputs.Workload."""
    return make_cfg(w.L, w.Bq, w.N, w.Hk, w.Hv, w.d, w.K, w.n_slots, w.l2_eps, w.q_scale, mode)


_BF16_OK = (torch.bfloat16, torch.int16, getattr(torch, "uint16", torch.int16))


def _ptr(t: Optional[torch.Tensor], dtypes=None, name="") -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: tensor must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    return t.data_ptr()


def _bf(t, name):
    return _ptr(t, _BF16_OK, name)


def _f32(t, name):
    return _ptr(t, (torch.float32,), name)


def _i32(t, name):
    return _ptr(t, (torch.int32,), name)


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, rc: int):
    if rc != LBX_OK:
        raise LbxError(fn, rc)


def lbx_workspace_size(cfg: lbx_cfg) -> int:
    return int(load().lbx_workspace_size(ctypes.byref(cfg)))


def lbx_tree_conv(cfg, x, conv_w, conv_cache, parent, slot, qkv_out, d_status=None, stream=None):
    _check("lbx_tree_conv", load().lbx_tree_conv(
        ctypes.byref(cfg), _bf(x, "x"), _bf(conv_w, "conv_w"), _f32(conv_cache, "conv_cache"),
        _i32(parent, "parent"), _i32(slot, "slot"), _f32(qkv_out, "qkv_out"),
        _i32(d_status, "d_status"), _stream(stream)))


def lbx_tree_deltanet(cfg, qkv, a, b, state, parent, slot, o, node_states=None, d_status=None,
                      stream=None):
    _check("lbx_tree_deltanet", load().lbx_tree_deltanet(
        ctypes.byref(cfg), _f32(qkv, "qkv"), _bf(a, "a"), _bf(b, "b"), _f32(state, "state"),
        _i32(parent, "parent"), _i32(slot, "slot"), _f32(o, "o"),
        _f32(node_states, "node_states"), _i32(d_status, "d_status"), _stream(stream)))


def lbx_tree_persist(cfg, x, node_states, parent, slot, accepted, state, conv_cache,
                     d_status=None, stream=None):
    _check("lbx_tree_persist", load().lbx_tree_persist(
        ctypes.byref(cfg), _bf(x, "x"), _f32(node_states, "node_states"), _i32(parent, "parent"),
        _i32(slot, "slot"), _i32(accepted, "accepted"), _f32(state, "state"),
        _f32(conv_cache, "conv_cache"), _i32(d_status, "d_status"), _stream(stream)))


def lbx_verify_step(cfg, x, conv_w, a, b, parent, slot, accepted, state, conv_cache, o,
                    workspace, d_status=None, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("lbx_verify_step", load().lbx_verify_step(
        ctypes.byref(cfg), _bf(x, "x"), _bf(conv_w, "conv_w"), _bf(a, "a"), _bf(b, "b"),
        _i32(parent, "parent"), _i32(slot, "slot"), _i32(accepted, "accepted"),
        _f32(state, "state"), _f32(conv_cache, "conv_cache"), _f32(o, "o"),
        _ptr(workspace, None, "workspace"), ws_bytes, _i32(d_status, "d_status"),
        _stream(stream)))


def lbx_verify_step_noalloc(cfg, x, conv_w, a, b, parent, slot, accepted, state, conv_cache, o,
                            d_status=None, stream=None):
    """lbx_verify_step for callers that cannot allocate: the arrival counters
    live in a fixed array inside the library (see include/lbx.h)."""
    _check("lbx_verify_step_noalloc", load().lbx_verify_step_noalloc(
        ctypes.byref(cfg), _bf(x, "x"), _bf(conv_w, "conv_w"), _bf(a, "a"), _bf(b, "b"),
        _i32(parent, "parent"), _i32(slot, "slot"), _i32(accepted, "accepted"),
        _f32(state, "state"), _f32(conv_cache, "conv_cache"), _f32(o, "o"),
        _i32(d_status, "d_status"), _stream(stream)))


def new_workspace(cfg: lbx_cfg, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of lbx_workspace_size(cfg) bytes."""
    n = lbx_workspace_size(cfg)
    if n == 0:
        raise LbxError("lbx_workspace_size", LBX_EINVAL)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def lbx_accept_workspace_size(Bq: int, N: int, V: int) -> int:
    return int(load().lbx_accept_workspace_size(Bq, N, V))


def new_accept_workspace(Bq: int, N: int, V: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of lbx_accept_workspace_size(Bq, N, V) bytes."""
    n = lbx_accept_workspace_size(Bq, N, V)
    if n == 0:
        raise LbxError("lbx_accept_workspace_size", LBX_EINVAL)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def lbx_accept_walk(logits, draft, parent, accepted_out, next_out, workspace, argmax_out=None,
                    d_status=None, stream=None):
    """Verify argmax and greedy acceptance walk; logits float32 [Bq][N][V]."""
    Bq, N, V = logits.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("lbx_accept_walk", load().lbx_accept_walk(
        Bq, N, V, _f32(logits, "logits"), _i32(draft, "draft"), _i32(parent, "parent"),
        _i32(argmax_out, "argmax_out"), _i32(accepted_out, "accepted_out"),
        _i32(next_out, "next_out"), _ptr(workspace, None, "workspace"), ws_bytes,
        _i32(d_status, "d_status"), _stream(stream)))


def lbx_ddtree_build(logp, tok, root_tok, B, parent_out, token_out, n_nodes_out,
                     depth_out=None, score_out=None, stream=None):
    """DDTree construction of budget B from logp float32 [Bq][D][K] and tok
    int32 [Bq][D][K]."""
    Bq, D, K = logp.shape
    _check("lbx_ddtree_build", load().lbx_ddtree_build(
        Bq, D, K, int(B), _f32(logp, "logp"), _i32(tok, "tok"), _i32(root_tok, "root_tok"),
        _i32(parent_out, "parent_out"), _i32(token_out, "token_out"),
        _i32(depth_out, "depth_out"), _f32(score_out, "score_out"),
        _i32(n_nodes_out, "n_nodes_out"), _stream(stream)))


def lbx_attn_workspace_size(L: int, Bq: int, N: int, Hq: int, Hkv: int, dh: int, T: int) -> int:
    return int(load().lbx_attn_workspace_size(L, Bq, N, Hq, Hkv, dh, T))


def new_attn_workspace(L, Bq, N, Hq, Hkv, dh, T, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of lbx_attn_workspace_size(...) bytes."""
    n = lbx_attn_workspace_size(L, Bq, N, Hq, Hkv, dh, T)
    if n == 0:
        raise LbxError("lbx_attn_workspace_size", LBX_EINVAL)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def lbx_tree_attention(scale, ctx_len, parent, q, k_cache, v_cache, k_tree, v_tree, o, workspace,
                       d_status=None, stream=None):
    """Tree-masked attention of the full-attention layers: q bf16
    [L][Bq][N][Hq][dh], k_cache / v_cache [L][Bq][T][Hkv][dh], k_tree / v_tree
    [L][Bq][N][Hkv][dh], o float32 like q; shapes are read from the tensors."""
    L, Bq, N, Hq, dh = q.shape
    T, Hkv = k_cache.shape[2], k_cache.shape[3]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("lbx_tree_attention", load().lbx_tree_attention(
        L, Bq, N, Hq, Hkv, dh, T, float(scale), _i32(ctx_len, "ctx_len"), _i32(parent, "parent"),
        _bf(q, "q"), _bf(k_cache, "k_cache") if T > 0 else None,
        _bf(v_cache, "v_cache") if T > 0 else None, _bf(k_tree, "k_tree"), _bf(v_tree, "v_tree"),
        _f32(o, "o"), _ptr(workspace, None, "workspace"), ws_bytes, _i32(d_status, "d_status"),
        _stream(stream)))
