"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
CUDA path through the C ABI, and compare with the fp64 oracle.

Tolerances (per workload): max |o_gpu - o_ref| <= 2e-3 * max |o_ref|;
state relative Frobenius error <= 1e-4 for every (layer, slot, head);
bit-exact conv-cache persist and untouched unreferenced slots.
"""
import numpy as np
import torch

import oracle
from tree_verify_linear_gb300 import lbx

O_TOL = 2e-3
STATE_TOL = 1e-4


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_inputs(inp: dict) -> dict:
    return {k: to_dev(v) for k, v in inp.items()}


def run_verify(w, inp, mode=lbx.LBX_MODE_AUTO, steps=1, ws=None):
    """Run lbx_verify_step `steps` times in place.  Returns numpy copies of
    (o, state, conv_cache, status, workspace)."""
    d = dev_inputs(inp)
    cfg = lbx.cfg_of(w, mode)
    o = torch.full((w.L, w.Bq, w.N, w.Hv, w.d), float("nan"), device="cuda")
    ws = lbx.new_workspace(cfg) if ws is None else ws
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(steps):
        lbx.lbx_verify_step(cfg, d["x"], d["conv_w"], d["a"], d["b"], d["parent"], d["slot"],
                            d["accepted"], d["state"], d["conv_cache"], o, ws, status)
    torch.cuda.synchronize()
    return (o.cpu().numpy(), d["state"].cpu().numpy(), d["conv_cache"].cpu().numpy(),
            int(status.item()), ws.cpu().numpy())


def uses_tensor_cores(w, mode=lbx.LBX_MODE_AUTO) -> bool:
    """Whether lbx_verify_step runs the tensor-core step (tree mode, d = 128,
    N <= 64), whose workspace holds the prep kernel's records instead of
    arrival counters."""
    if mode == lbx.LBX_MODE_AUTO:
        mode = lbx.LBX_MODE_TREE if w.N <= lbx.LBX_MAX_TREE_NODES else lbx.LBX_MODE_CHUNKED
    return mode == lbx.LBX_MODE_TREE and w.d == 128 and w.N <= 64


def counters_cleared(w, ws: np.ndarray, mode=lbx.LBX_MODE_AUTO) -> bool:
    """The CUDA-core kernels leave their arrival counters at zero; the
    tensor-core step's workspace holds records and is not checked."""
    return uses_tensor_cores(w, mode) or not ws.any()


def o_error(o_gpu: np.ndarray, o_ref: np.ndarray) -> float:
    """max |o_gpu - o_ref| / max |o_ref|."""
    return float(np.abs(o_gpu.astype(np.float64) - o_ref).max() / np.abs(o_ref).max())


def state_rel(s_gpu: np.ndarray, s_ref: np.ndarray) -> float:
    return float(np.linalg.norm(s_gpu.astype(np.float64) - s_ref) / np.linalg.norm(s_ref))


def check_verify(w, inp, o_gpu, state_gpu, cache_gpu, items=None, form=oracle.FORM_PATH,
                 n_threads=0, batch_bytes=1 << 28):
    """Compare one fused verify step with the oracle.

    items: (layer, request, head) triples to check against the oracle (all
    heads when None), taken in batches whose oracle outputs hold about
    batch_bytes; the o bound is over all of them (max |diff| / max |ref|).
    Every (layer, request) conv window is checked bit-exactly, and every
    slot no request names byte-for-byte."""
    if items is None:
        items = [(l, b, h) for l in range(w.L) for b in range(w.Bq) for h in range(w.Hv)]
    per_item = (w.N * w.d + w.d * w.d) * 8
    step = max(1, batch_bytes // per_item)
    diff, ref_max, worst = 0.0, 0.0, 0.0
    for i0 in range(0, len(items), step):
        chunk = items[i0:i0 + step]
        o_ref, s_ref, _ = oracle.verify_heads(w, inp, chunk, form=form, n_threads=n_threads)
        og = np.stack([o_gpu[l, b, :, h, :] for (l, b, h) in chunk]).astype(np.float64)
        diff = max(diff, float(np.abs(og - o_ref).max()))
        ref_max = max(ref_max, float(np.abs(o_ref).max()))
        for i, (l, b, h) in enumerate(chunk):
            worst = max(worst, state_rel(state_gpu[l, inp["slot"][b], h], s_ref[i]))
    err_o = diff / ref_max
    assert err_o <= O_TOL, f"o error {err_o:.3e} > {O_TOL}"
    assert worst <= STATE_TOL, f"state rel error {worst:.3e} > {STATE_TOL}"
    K = w.K
    for l in range(w.L):
        for b in range(w.Bq):
            s = inp["slot"][b]
            exp = oracle.persist_conv_lb(w.N, w.C, K, inp["x"][l, b], inp["conv_cache"][l, s],
                                         inp["parent"][b], inp["accepted"][b])
            assert exp.view(np.uint32).tobytes() == cache_gpu[l, s].view(np.uint32).tobytes(), \
                f"conv window mismatch at layer {l} request {b}"
    used = set(int(s) for s in inp["slot"])
    for s in range(w.n_slots):
        if s not in used:
            assert state_gpu[:, s].tobytes() == inp["state"][:, s].tobytes(), f"slot {s} touched"
            assert cache_gpu[:, s].tobytes() == inp["conv_cache"][:, s].tobytes(), \
                f"conv slot {s} touched"
    return err_o, worst
