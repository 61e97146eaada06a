"""Benchmark of the fused tree-verify step (lbx_verify_step) on GB300.

Default workload: the full verify step of a 27B-class hybrid target -- 48
gated-DeltaNet layers, 16 key / 48 value heads, d = 128, conv width 4, one
request, a 22-node DDTree draft tree (budget 22).  One step = one call of
lbx_verify_step over all layers (conv + recurrence + persist).

Prints one JSON line.  `value` is node-head updates per second (L*Bq*N*Hv per
step) with inputs resident in HBM; `e2e` is the same metric through the C ABI
with the step's inputs copied from pinned host memory and o copied back inside
the timed region.  `--impl reference` times the fp64 CPU oracle instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lbx|reference]
                       [--workload NAME] [--op verify|unfused|accept|ddtree|attn]
`--op unfused` times lbx_tree_conv -> lbx_tree_deltanet (node states) ->
lbx_tree_persist on --workload, `--op accept` times lbx_accept_walk (verify argmax + greedy acceptance walk)
on a 5-request serving batch instead, `--op ddtree` lbx_ddtree_build, `--op
attn` lbx_tree_attention on --attn-workload (each a separate JSON line of its
own).
Under torchrun each rank runs an independent replica (the path needs no
exchange between GPUs); value is the sum over ranks of the work done divided
by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tree_verify_linear_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402

METRIC = "µs per DDTree verify step & node-head updates/s; HBM GB/s vs ~8 TB/s roofline"
UNIT = "node-head updates/s"


def step_kernels(w):
    """The kernels one lbx_verify_step call launches for this workload (the
    library's own selection rule, default mode): tree mode (N <= 64) with
    d = 128 is a prep kernel per key head followed by the
    tensor-core step kernel; chunked mode (longer chains) with d = 128 is the
    tensor-core chain kernel; the other configurations run one CUDA-core
    kernel."""
    if w.d == 128 and w.N <= 64:
        return ("gdn_qk_prep_kernel", "gdn_step_tc_kernel")
    if w.d == 128 and w.N > 64:
        return ("gdn_chain_tc_kernel",)
    return ("gdn_step_kernel",)


def step_dtype(w) -> str:
    """Arithmetic of the path the step runs: the tensor-core kernels take
    their products as three bf16 passes (hi*hi + hi*lo + lo*hi) with fp32
    accumulation, the CUDA-core kernel plain fp32."""
    if w.d == 128:
        return "f32 (tensor-core products as 3-pass bf16 hi/lo splits, fp32 accumulate)"
    return "f32"


def algorithmic_bytes(w) -> int:
    """Bytes one fused step must move at minimum: state and conv window read
    and written once per (layer, request), conv weights once per layer, the
    bf16 inputs and gates, the tree indices (parent, slot, accepted) and o."""
    C = w.C
    per_lb = (2 * w.Hv * w.d * w.d * 4          # state read + write
              + 2 * (w.K - 1) * C * 4           # conv window read + write
              + w.N * C * 2                     # x
              + 2 * w.N * w.Hv * 2              # a, b
              + (w.N + 2) * 4                   # parent, slot, accepted
              + w.N * w.Hv * w.d * 4)           # o
    return w.L * (w.Bq * per_lb + C * w.K * 2)  # conv_w once per layer


def describe(w) -> str:
    tree = {"ddtree": f"budget-{w.N} DDTree-shaped tree", "uniform": f"{w.N}-node uniform tree",
            "chain": f"{w.N}-token chain"}[w.tree]
    return (f"{w.name}: {w.L} GDN layers, {w.Bq} request(s), {tree}, Hk={w.Hk}, Hv={w.Hv}, "
            f"d={w.d}, conv width {w.K}")


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# Sources of kernels that the verify step never launches; a change to them
# leaves the recorded traffic of the verify workloads valid.
OTHER_OPS = ("accept_walk.cu", "ddtree_build.cu", "tree_attn.cu")


def kernel_source_hash(op: str = "verify") -> str:
    """Hash of the CUDA sources the op's kernels are built from: every file
    under csrc/ except the other ops' kernels (verify), or the attention
    kernel and the PTX wrappers it includes (attn)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tree_verify_linear_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if op == "verify" and name in OTHER_OPS:
            continue
        if op == "attn" and name not in ("tree_attn.cu", "tc_ptx.cuh"):
            continue
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, op: str = "verify"):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    e = j.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash(op):
        return None
    return int(e["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.rows = []
        self.proc = None
        self.gpu_id = gpu_id
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, on: bool):
        if on:
            self.t_on = time.time()
        else:
            self.t_off = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = [r for t, r in self.rows if self.t_on and self.t_off and self.t_on <= t <= self.t_off]
        if not rows:
            rows = [r for _, r in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 4 + i and r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup(n_gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if os.environ.get("LBX_BENCH_GLOO") is None else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline and the reference arm).
# ---------------------------------------------------------------------------
def oracle_rate(w, inp, budget_s: float, n_threads: int = 0):
    """Time the fp64 oracle (full verify step: conv, recurrence, accepted
    state) on whole (layer, request) slices until about budget_s seconds of
    work; returns (updates/s, threads, description)."""
    import oracle
    oracle.lib()
    done_heads = 0
    used = 1
    t0 = time.perf_counter()
    slices = [(l, b) for l in range(w.L) for b in range(w.Bq)]
    for (l, b) in slices:
        items = [(l, b, h) for h in range(w.Hv)]
        _, _, used = oracle.verify_heads(w, inp, items, n_threads=n_threads)
        done_heads += len(items)
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    rate = done_heads * w.N / dt
    n_slices = done_heads // w.Hv
    return rate, used, f"{n_slices} of {len(slices)} (layer, request) slices, all {w.Hv} heads"


def run_reference(args, w):
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    import oracle
    oracle.lib()
    inp = make_inputs(w)
    items_all = [(l, b, h) for l in range(w.L) for b in range(w.Bq) for h in range(w.Hv)]
    # size each step so the whole run takes about a minute
    t = time.perf_counter()
    _, _, used = oracle.verify_heads(w, inp, items_all[:w.Hv])
    per_head = (time.perf_counter() - t) / w.Hv
    total = args.steps + args.warmup
    heads_per_step = int(max(1, min(len(items_all), 60.0 / max(total, 1) / max(per_head, 1e-9))))
    k = 0
    times = []
    for s in range(total):
        items = [items_all[(k + i) % len(items_all)] for i in range(heads_per_step)]
        k += heads_per_step
        t = time.perf_counter()
        _, _, used = oracle.verify_heads(w, inp, items)
        dt = time.perf_counter() - t
        if s >= args.warmup:
            times.append(dt)
    sec = sum(times)
    value = heads_per_step * w.N * len(times) / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(w)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": f"each step: {heads_per_step} (layer, request, head) items of "
                                   f"the workload, full conv + recurrence + accepted state"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# The GPU arm.
# ---------------------------------------------------------------------------
def run_lbx(args, w):
    import torch
    from tree_verify_linear_gb300 import lbx

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lbx.load()
    inp = make_inputs(w, seed=w.seed + 7919 * rank)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    d = {k: to_dev(v) for k, v in inp.items()}
    cfg = lbx.cfg_of(w)
    o = torch.empty((w.L, w.Bq, w.N, w.Hv, w.d), device=dev)
    ws = lbx.new_workspace(cfg, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        lbx.lbx_verify_step(cfg, d["x"], d["conv_w"], d["a"], d["b"], d["parent"], d["slot"],
                            d["accepted"], d["state"], d["conv_cache"], o, ws, status, stream)

    # ---- device-resident timing ----
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", ""))
    gpu_id = (uuid if uuid.startswith("GPU-") else "GPU-" + uuid) if uuid else str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    barrier(world)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    barrier(world)
    ms_local = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms_local, world, dev)
    sampler.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    units = w.L * w.Bq * w.N * w.Hv
    value = units * args.steps * world / (ms / 1e3)
    ms_per_step = ms / args.steps

    # ---- end to end: host buffers through the C ABI ----
    names_in = ("x", "a", "b", "parent", "slot", "accepted")
    host = {k: d[k].cpu().pin_memory() for k in names_in}
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h2d = sum(host[k].numel() * host[k].element_size() for k in names_in)
    d2h = o_host.numel() * o_host.element_size()
    e2e_steps = max(3, min(args.steps, 200))

    def e2e_step():
        for k in names_in:
            d[k].copy_(host[k], non_blocking=True)
        step()
        o_host.copy_(o, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = units * e2e_steps * world / (e2e_ms / 1e3)

    if rank != 0:
        return

    peak, peak_kind = read_peaks()
    alg = algorithmic_bytes(w)
    kernels = step_kernels(w)
    achieved = alg / (ms_per_step / 1e3) / 1e9
    traffic = recorded_traffic(w.name)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        rate, cores, sample = oracle_rate(w, inp, budget_s=args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_step": 1e3 * ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": step_dtype(w),
        "data": "synthetic",
        "config": {"workload": describe(w), "L": w.L, "Bq": w.Bq, "N": w.N, "Hk": w.Hk,
                   "Hv": w.Hv, "d": w.d, "K": w.K, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({alg / 1e6:.1f} MB moved per step)"},
        "hbm_gbs": achieved,
        # achieved = the step's algorithmic bytes over the time of the whole
        # call (every kernel it launches), so it is a lower bound for the
        # dominant kernel alone
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
                     "algorithmic_bytes": alg, "kernel": "+".join(kernels),
                     "timed": "whole lbx_verify_step call"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps * len(kernels),
        "clocks": sampler.summary(),
    }
    print(json.dumps(line))


def run_accept(args):
    """Times lbx_accept_walk (verify argmax + greedy acceptance walk) on a
    5-request serving batch of budget-22 trees and a 152K vocabulary.  Three
    logits buffers are used in turn (3 x 67 MB > L2), so each call reads its
    logits from HBM."""
    import torch
    from tree_verify_linear_gb300 import lbx
    from tree_verify_linear_gb300.inputs import ACCEPT_VOCAB, make_accept_inputs

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lbx.load()
    Bq, N, V = 5, 22, ACCEPT_VOCAB
    sets = [make_accept_inputs(Bq, N, V, seed=3001 + 97 * rank + i) for i in range(3)]
    lg = [torch.from_numpy(x["logits"]).to(dev) for x in sets]
    dr = [torch.from_numpy(x["draft"]).to(dev) for x in sets]
    pa = [torch.from_numpy(x["parent"]).to(dev) for x in sets]
    acc = torch.zeros(Bq, dtype=torch.int32, device=dev)
    nxt = torch.zeros(Bq, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = lbx.new_accept_workspace(Bq, N, V, dev)
    stream = torch.cuda.current_stream(dev)

    def call(i):
        k = i % 3
        lbx.lbx_accept_walk(lg[k], dr[k], pa[k], acc, nxt, ws, d_status=status, stream=stream)

    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", ""))
    gpu_id = (uuid if uuid.startswith("GPU-") else "GPU-" + uuid) if uuid else str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    barrier(world)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    ev0.record(stream)
    for i in range(args.steps):
        call(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    sampler.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    us = 1e3 * ms / args.steps

    # end to end: the draft tokens and parents from pinned host memory, the
    # accepted nodes and next tokens back (the logits are produced on the
    # device by the target's forward and stay there)
    hd = [x["draft"] for x in sets]
    h_dr = torch.from_numpy(hd[0]).pin_memory()
    h_pa = torch.from_numpy(sets[0]["parent"]).pin_memory()
    h_acc = torch.zeros(Bq, dtype=torch.int32).pin_memory()
    h_nxt = torch.zeros(Bq, dtype=torch.int32).pin_memory()
    e2e_steps = max(3, min(args.steps, 200))

    def e2e(i):
        dr[0].copy_(h_dr, non_blocking=True)
        pa[0].copy_(h_pa, non_blocking=True)
        lbx.lbx_accept_walk(lg[i % 3], dr[0], pa[0], acc, nxt, ws, d_status=status, stream=stream)
        h_acc.copy_(acc, non_blocking=True)
        h_nxt.copy_(nxt, non_blocking=True)

    for i in range(3):
        e2e(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        e2e(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_us = 1e3 * max_over_ranks(e0.elapsed_time(e1), world, dev) / e2e_steps
    if rank != 0:
        return
    import oracle  # CPU baseline leg only
    cpu = None
    if not args.no_cpu_baseline:
        t0, n = time.time(), 0
        while time.time() - t0 < min(args.cpu_seconds, 10.0):
            oracle.accept_walk(sets[n % 3]["logits"], sets[n % 3]["draft"], sets[n % 3]["parent"])
            n += 1
        cpu = {"value": 1e6 * (time.time() - t0) / n, "unit": "us per call", "cores": 1,
               "kind": "oracle", "sample": f"{n} whole calls (5 x 22 x {V} logits)"}
    peak, peak_kind = read_peaks()
    alg = Bq * N * V * 4 + 2 * Bq * N * 4 + 2 * Bq * 4
    achieved = alg / (us / 1e6) / 1e9
    line = {
        "metric": "us per verify argmax + acceptance walk", "value": us, "unit": "us per call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"acceptance walk: {Bq} requests, budget-{N} DDTree-shaped "
                               f"trees, vocabulary {V}",
                   "Bq": Bq, "N": N, "V": V, "parallelism": f"replicas x{world}",
                   "l2": "three logits buffers in turn (3 x 67 MB > L2)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind, "traffic": None,
                     "algorithmic_bytes": alg, "kernel": "accept_walk_kernel",
                     "timed": "whole lbx_accept_walk call"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_us, "unit": "us per call",
                "h2d_bytes_per_step": 2 * Bq * N * 4, "d2h_bytes_per_step": 2 * Bq * 4,
                "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line))


def run_ddtree(args):
    """Times lbx_ddtree_build: budget-22 trees for 5 requests from a
    16-position draft block with top-8 tokens per position.  The kernel is a
    chain of 21 dependent selection rounds per request (one warp each): it
    is bound by latency, not by bytes or arithmetic, so no roofline fraction
    is given."""
    import torch
    from tree_verify_linear_gb300 import lbx
    from tree_verify_linear_gb300.inputs import ACCEPT_VOCAB, make_draft_topk

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lbx.load()
    Bq, D, K, B = 5, 16, 8, 22
    d = make_draft_topk(Bq, D, K, ACCEPT_VOCAB, seed=5001 + rank)
    lp = torch.from_numpy(d["logp"]).to(dev)
    tk = torch.from_numpy(d["tok"]).to(dev)
    rt = torch.from_numpy(d["root_tok"]).to(dev)
    par = torch.zeros((Bq, B), dtype=torch.int32, device=dev)
    tn = torch.zeros((Bq, B), dtype=torch.int32, device=dev)
    nn = torch.zeros(Bq, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        lbx.lbx_ddtree_build(lp, tk, rt, B, par, tn, nn, stream=stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    barrier(world)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        call()
    ev1.record(stream)
    torch.cuda.synchronize()
    us = 1e3 * max_over_ranks(ev0.elapsed_time(ev1), world, dev) / args.steps
    if rank != 0:
        return
    import oracle  # CPU baseline leg only
    cpu = None
    if not args.no_cpu_baseline:
        t0, n = time.time(), 0
        while time.time() - t0 < 2.0:
            oracle.ddtree_build(d["logp"], d["tok"], d["root_tok"], B)
            n += 1
        cpu = {"value": 1e6 * (time.time() - t0) / n, "unit": "us per call", "cores": 1,
               "kind": "oracle", "sample": f"{n} whole calls"}
    line = {
        "metric": "us per DDTree construction", "value": us, "unit": "us per call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"DDTree build: {Bq} requests, budget {B}, draft block {D}, "
                               f"top-{K}", "Bq": Bq, "D": D, "K": K, "B": B,
                   "parallelism": f"replicas x{world}", "l2": "inputs of 5 KB (latency-bound)"},
        "roofline": {"bound": "latency", "achieved": None, "peak": None, "unit": None,
                     "frac": None, "kernel": "ddtree_build_kernel",
                     "timed": "whole lbx_ddtree_build call"},
        "cpu_baseline": cpu,
        "gpu_launches": args.steps,
    }
    print(json.dumps(line))


def attn_algorithmic_bytes(w, ctx_len) -> int:
    """Bytes one tree-attention call must move: each request's cached keys
    and values up to its context length, q, the tree's keys and values, o
    (fp32), the context lengths and parent arrays."""
    kv = int(np.asarray(ctx_len, dtype=np.int64).sum()) * w.L * w.Hkv * w.dh * 2 * 2
    q = w.L * w.Bq * w.N * w.Hq * w.dh * 2
    tree = 2 * w.L * w.Bq * w.N * w.Hkv * w.dh * 2
    o = w.L * w.Bq * w.N * w.Hq * w.dh * 4
    return kv + q + tree + o + w.Bq * 4 + w.Bq * w.N * 4


def run_attn(args):
    """Times lbx_tree_attention (the full-attention layers of the verify
    forward) on --attn-workload; the default, attn27b, reads 268 MB of KV
    cache per call (> L2)."""
    import torch
    from tree_verify_linear_gb300 import lbx
    from tree_verify_linear_gb300.inputs import ATTN_WORKLOADS, make_attn_inputs

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lbx.load()
    w = ATTN_WORKLOADS[args.attn_workload]
    inp = make_attn_inputs(w, seed=w.seed + 7919 * rank)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    d = {k: to_dev(v) for k, v in inp.items()}
    o = torch.empty((w.L, w.Bq, w.N, w.Hq, w.dh), device=dev)
    ws = lbx.new_attn_workspace(w.L, w.Bq, w.N, w.Hq, w.Hkv, w.dh, w.T, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        lbx.lbx_tree_attention(w.scale, d["ctx_len"], d["parent"], d["q"], d["k_cache"],
                               d["v_cache"], d["k_tree"], d["v_tree"], o, ws, status, stream)

    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", ""))
    gpu_id = (uuid if uuid.startswith("GPU-") else "GPU-" + uuid) if uuid else str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    barrier(world)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    ev0.record(stream)
    for _ in range(args.steps):
        call()
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    sampler.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    us = 1e3 * ms / args.steps

    # end to end: the step's queries, tree keys / values, context lengths and
    # parents from pinned host memory, o back (the KV cache stays resident)
    names_in = ("q", "k_tree", "v_tree", "ctx_len", "parent")
    host = {k: d[k].cpu().pin_memory() for k in names_in}
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h2d = sum(host[k].numel() * host[k].element_size() for k in names_in)
    d2h = o_host.numel() * o_host.element_size()
    e2e_steps = max(3, min(args.steps, 200))

    def e2e():
        for k in names_in:
            d[k].copy_(host[k], non_blocking=True)
        call()
        o_host.copy_(o, non_blocking=True)

    for _ in range(3):
        e2e()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_us = 1e3 * max_over_ranks(e0.elapsed_time(e1), world, dev) / e2e_steps
    if rank != 0:
        return
    import oracle  # CPU baseline leg only
    cpu = None
    if not args.no_cpu_baseline:
        # one (layer) slice of the call, scaled to the whole call
        t0 = time.time()
        sl = {k: (np.ascontiguousarray(v[:1]) if k not in ("ctx_len", "parent") else v)
              for k, v in inp.items()}
        oracle.tree_attention(sl["q"], sl["k_cache"], sl["v_cache"], sl["k_tree"], sl["v_tree"],
                              sl["ctx_len"], sl["parent"], w.scale)
        dt = time.time() - t0
        cpu = {"value": 1e6 * dt * w.L, "unit": "us per call", "cores": 1, "kind": "oracle",
               "sample": f"layer 0 of {w.L} (all requests, nodes and heads), timed and scaled "
                         f"by {w.L}"}
    peak, peak_kind = read_peaks()
    alg = attn_algorithmic_bytes(w, inp["ctx_len"])
    achieved = alg / (us / 1e6) / 1e9
    line = {
        "metric": "us per tree-masked attention call", "value": us, "unit": "us per call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.L} full-attention layers, {w.Bq} request(s), "
                               f"budget-{w.N} tree, Hq={w.Hq}, Hkv={w.Hkv}, dh={w.dh}, "
                               f"context {w.T} ({w.ctx})",
                   "L": w.L, "Bq": w.Bq, "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "dh": w.dh,
                   "T": w.T, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({alg / 1e6:.1f} MB per call)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": recorded_traffic(w.name, "attn"),
                     "algorithmic_bytes": alg, "kernel": "tree_attn_kernel",
                     "timed": "whole lbx_tree_attention call"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_us, "unit": "us per call", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line))


def run_unfused(args, w):
    """Times the three unfused entry points chained on one stream --
    lbx_tree_conv -> lbx_tree_deltanet (with per-node state snapshots) ->
    lbx_tree_persist -- on --workload, each kernel between CUDA events, with
    its own algorithmic bytes and roofline fraction; the snapshot write of
    lbx_tree_deltanet (N states per head) dominates."""
    import torch
    from tree_verify_linear_gb300 import lbx

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lbx.load()
    inp = make_inputs(w, seed=w.seed + 7919 * rank)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    d = {k: to_dev(v) for k, v in inp.items()}
    cfg = lbx.cfg_of(w)
    qkv = torch.empty((w.L, w.Bq, w.N, w.C), device=dev)
    o = torch.empty((w.L, w.Bq, w.N, w.Hv, w.d), device=dev)
    ns = torch.empty((w.L, w.Bq, w.N, w.Hv, w.d, w.d), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    calls = [
        lambda: lbx.lbx_tree_conv(cfg, d["x"], d["conv_w"], d["conv_cache"], d["parent"],
                                  d["slot"], qkv, status, stream),
        lambda: lbx.lbx_tree_deltanet(cfg, qkv, d["a"], d["b"], d["state"], d["parent"],
                                      d["slot"], o, ns, status, stream),
        lambda: lbx.lbx_tree_persist(cfg, d["x"], ns, d["parent"], d["slot"], d["accepted"],
                                     d["state"], d["conv_cache"], status, stream),
    ]
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", ""))
    gpu_id = (uuid if uuid.startswith("GPU-") else "GPU-" + uuid) if uuid else str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    for _ in range(args.warmup):
        for c in calls:
            c()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    barrier(world)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler.mark(True)
    for k in range(args.steps):
        ev[k][0].record(stream)
        for i, c in enumerate(calls):
            c()
            ev[k][i + 1].record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    barrier(world)
    sampler.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    per = [1e3 * sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(args.steps)) / args.steps
           for i in range(3)]
    per = [max_over_ranks(x, world, dev) for x in per]
    us = sum(per)

    # ---- end to end: the step's inputs from pinned host memory and o back,
    # inside the timed region (states, caches and snapshots stay resident) ----
    names_in = ("x", "a", "b", "parent", "slot", "accepted")
    host = {k: d[k].cpu().pin_memory() for k in names_in}
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h2d = sum(host[k].numel() * host[k].element_size() for k in names_in)
    d2h = o_host.numel() * o_host.element_size()
    e2e_steps = max(3, min(args.steps, 50))

    def e2e_step():
        for k in names_in:
            d[k].copy_(host[k], non_blocking=True)
        for c in calls:
            c()
        o_host.copy_(o, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    e2e_us = max_over_ranks(1e3 * e0.elapsed_time(e1) / e2e_steps, world, dev)
    if rank != 0:
        return
    L, Bq, N, Hv, dd, C, K = w.L, w.Bq, w.N, w.Hv, w.d, w.C, w.K
    slab = dd * dd * 4
    alg = [
        # conv: x, weights, the slots' cached rows, parents; qkv out
        L * Bq * N * C * 2 + L * C * K * 2 + L * Bq * (K - 1) * C * 4 + Bq * N * 4
        + L * Bq * N * C * 4,
        # deltanet: qkv, gates, S0, parents; o and every node's state out
        L * Bq * N * C * 4 + 2 * L * Bq * N * Hv * 2 + L * Bq * Hv * slab + Bq * N * 4
        + L * Bq * N * Hv * dd * 4 + L * Bq * N * Hv * slab,
        # persist: the accepted node's state in, the slot's state out, the conv
        # window (at most K-1 rows read and written)
        2 * L * Bq * Hv * slab + 2 * L * Bq * (K - 1) * C * 4 + Bq * N * 4 + 2 * Bq * 4,
    ]
    peak, peak_kind = read_peaks()
    names = ("tree_conv_kernel", "gdn_step_kernel (unfused, node states)", "tree_persist_kernel")
    kernels = {n: {"us": t, "algorithmic_bytes": a, "GB/s": a / (t / 1e6) / 1e9,
                   "frac": a / (t / 1e6) / 1e9 / peak}
               for n, t, a in zip(names, per, alg)}
    import oracle  # CPU baseline leg only
    cpu = None
    if not args.no_cpu_baseline:
        # layer 0 of every request: conv, every head's recurrence with node
        # states, the conv window; scaled by L
        t0 = time.time()
        mask = np.zeros((L, Bq), np.uint8)
        mask[0, :] = 1
        q0 = oracle.tree_conv(w, inp, lb_mask=mask)
        for b in range(Bq):
            s0 = int(inp["slot"][b])
            for h in range(Hv):
                oracle.deltanet_head(N, w.Hk, Hv, dd, h, w.q_scale, oracle.FORM_PATH, q0[0, b],
                                     inp["a"][0, b], inp["b"][0, b], inp["state"][0, s0, h],
                                     inp["parent"][b], accepted=int(inp["accepted"][b]),
                                     want_states=True)
            oracle.persist_conv_lb(N, C, K, inp["x"][0, b], inp["conv_cache"][0, s0],
                                   inp["parent"][b], inp["accepted"][b])
        dt = time.time() - t0
        cpu = {"value": 1e6 * dt * L, "unit": "us per step", "cores": 1, "kind": "oracle",
               "sample": f"layer 0 of {L} (all requests and heads, node states), scaled by {L}"}
    line = {
        "metric": "us per unfused verify step (lbx_tree_conv + lbx_tree_deltanet with node "
                  "states + lbx_tree_persist)",
        "value": us, "unit": "us per step", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": describe(w), "L": L, "Bq": Bq, "N": N, "Hk": w.Hk, "Hv": Hv,
                   "d": dd, "K": K, "parallelism": f"replicas x{world}",
                   "l2": "node states of one step > L2"},
        "roofline": {"bound": "hbm", "achieved": kernels[names[1]]["GB/s"], "peak": peak,
                     "unit": "GB/s", "frac": kernels[names[1]]["frac"], "peak_kind": peak_kind,
                     "traffic": recorded_traffic(f"{w.name}_unfused"),
                     "algorithmic_bytes": alg[1], "kernel": names[1],
                     "timed": "lbx_tree_deltanet call between CUDA events"},
        "kernels": kernels,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_us, "unit": "us per step", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": 3 * args.steps,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("lbx", "reference"), default="lbx")
    ap.add_argument("--workload", default="step27b", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", choices=("verify", "unfused", "accept", "ddtree", "attn"),
                    default="verify",
                    help="verify: lbx_verify_step on --workload (the headline); unfused: "
                         "lbx_tree_conv -> lbx_tree_deltanet -> lbx_tree_persist on --workload; "
                         "accept: lbx_accept_walk on a serving batch; ddtree: "
                         "lbx_ddtree_build; attn: lbx_tree_attention on --attn-workload")
    ap.add_argument("--attn-workload", default="attn27b")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = WORKLOADS[args.workload]
    if args.op in ("unfused", "accept", "ddtree", "attn"):
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              f"--op {args.op} times the library only; its oracle is the "
                              "cpu_baseline field"}))
            return
        if args.op == "unfused":
            run_unfused(args, w)
        else:
            {"accept": run_accept, "ddtree": run_ddtree, "attn": run_attn}[args.op](args)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_lbx(args, w)


if __name__ == "__main__":
    main()
