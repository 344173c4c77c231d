"""Benchmark: causal decayed linear attention (retention) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on rank 0.  A "step" is one chunkwise forward (la_chunk_fwd)
over the headline workload, the largest that fits one GPU: RetNet multi-scale
retention, B=8, H=16, T=8192, d_k=128, d_v=256, bf16 inputs, gamma_h =
1 - 2^(-5-h), no feature map, no normaliser.  The same line carries
sub-measurements of the other workloads (normalised linear attention, long
sequences, the floored normaliser, per-token decay, the Taylor feature map,
the backward pass and the recurrent decode step), each timed the same way.

Timing: CUDA events on the launching stream; W untimed warm-up steps; the K
timed steps cycle through enough input copies that their footprint exceeds
3x the L2 cache, so every step reads its inputs from HBM.  N > 1 (torchrun):
each rank runs its own shard of a batch N times larger (weak scaling, no
collective on the data path); the time is the max over ranks.

``--impl reference`` times the fp64 CPU oracle on the host cores on a
bounded sample of the same workload (the comparison arm).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = ("retention fwd tokens/s & TFLOP/s (% bf16 TC peak); decode steps/s & HBM GB/s")

# DRAM bytes (read + write) per launch of the headline's dominant kernel, from
# an ncu capture of that kernel on the headline workload (its summary sits under
# profiles/, named for the kernel and workload).  It holds only for the kernel
# sources that capture measured (their SHA-256 below); any later change to them
# makes the reported traffic null until the kernel is captured again.
KERNEL_SOURCES = ("chunk_tc_ws.cuh", "chunk_tc_ws.cu", "chunk_tc_common.cuh", "tc_ptx.cuh",
                  "chunk_tc.cu", "common.cuh", "launch.h")
TRAFFIC = {
    # (workload, kernel): bytes per launch
    ("msr_retention_bf16", "chunk_tc_ws_kernel/full"): {
        "bytes": 1_076_144_896 + 517_590_016,
        "sources_sha256": "6e82be391a8cddc6f69c03d83b4979e7daa8d1411b3698bfca889a817c65fd63",
    },
}
HEADLINE = "msr_retention_bf16"
# the prefill workloads timed beside the headline
SUB_PREFILL = ("linear_attention_bf16", "long_retention_bf16", "retention_floor_bf16",
               "gated_retention_bf16", "taylor_linear_attention_bf16")
# the backward pass of normalised linear attention with phi (tensor-core composite)
BWD_NORM = "linear_attention_bf16"
# the backward pass on the tensor cores: plain retention, d_k = d_v = 128
BWD_TC = "long_retention_bf16"
# the second-order Taylor feature map (273 features from d = 16)
TAYLOR = "taylor_linear_attention_bf16"
L2_BYTES = 129 * 1024 * 1024
C_REF = 64  # chunk length fixed for counting useful intra-chunk flops


# ----------------------------------------------------------------------------- accounting

def feature_dim(c: dict) -> int:
    """Rows of the state: d_k, or 1 + d_k + d_k^2 with the Taylor feature map."""
    return 1 + c["dk"] + c["dk"] ** 2 if c["phi"] == "taylor" else c["dk"]


def alg_bytes(c: dict) -> int:
    """Bytes the method must move: read Q, K, V (and the per-token log decays),
    write O, write S_T (and z_T) in fp32."""
    es = 2 if c["dtype"] == "bf16" else 4
    nbh = c["B"] * c["H"]
    df = feature_dim(c)
    io = nbh * c["T"] * ((2 * c["dk"] + 2 * c["dv"]) * es + (4 if c.get("gate") else 0))
    state = nbh * df * c["dv"] * 4 + (nbh * df * 4 if c["normalize"] else 0)
    return io + state


def alg_flops(c: dict) -> int:
    """Useful flops: 4 d_phi d_v per head-token (state update + read-out, the right
    order of "Moving the parentheses") plus the causal lower triangle of C_REF-long
    intra-chunk squares, C_REF (d_phi + d_v) per head-token; d_phi = d_k, or 273
    features with the Taylor map."""
    nbh = c["B"] * c["H"]
    df = feature_dim(c)
    return nbh * c["T"] * (4 * df * c["dv"] + C_REF * (df + c["dv"]))


def decode_bytes(c: dict) -> int:
    """Per decode step: read + write the fp32 state, read q, k, v, write o."""
    nbh = c["B"] * c["H"]
    es = 2 if c["dtype"] == "bf16" else 4
    return nbh * (2 * c["dk"] * c["dv"] * 4 + (2 * c["dk"] + 2 * c["dv"]) * es)


def decode_flops(c: dict) -> int:
    """About 4 d_k d_v flops per head per token ("Decoding, training, ...")."""
    return c["B"] * c["H"] * 4 * c["dk"] * c["dv"]


def describe(name: str, c: dict) -> str:
    bits = [f"{name}: B={c['B']} H={c['H']} T={c['T']} d_k={c['dk']} d_v={c['dv']}",
            c["dtype"], {True: "phi=elu+1", False: "phi=identity",
                         "taylor": f"phi=Taylor (2nd order, {feature_dim(c)} features)"}[c["phi"]]]
    if c.get("gate"):
        bits.append("per-token decay")
    bits += [
            ("floored normaliser" if c.get("floor") else "normalised") if c["normalize"]
            else "no normaliser"]
    return ", ".join(bits)


def kernel_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "retnet_retention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(workload: str, kernel: str) -> int | None:
    t = TRAFFIC.get((workload, kernel))
    if t is None or t["sources_sha256"] != kernel_sources_sha256():
        return None
    return t["bytes"]


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained",
                                                      d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.25)
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self) -> dict | None:
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                 power=float(parts[3]) if parts[3] not in ("[N/A]", "") else 0.0,
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        busy = [r for r in rows if r["power"] > 0.25 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(r["sm"] for r in busy),
                    sm_max_mhz=max(r["smax"] for r in rows), reasons=sorted(reasons),
                    samples=len(rows))


# ----------------------------------------------------------------------------- our arm

def time_region(fn, steps: int, stream) -> float:
    """Device milliseconds for `steps` calls of fn(i), bracketed by events on `stream`."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        fn(i)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def graph_replay_ms(step_on, n_sets: int, steps: int) -> float | None:
    """Device milliseconds a step when the same steps are replayed from CUDA graphs
    (one captured step per input set, on a side stream): the launches then cost no
    host work.  None if capturing fails."""
    side = torch.cuda.Stream()
    try:
        graphs = []
        torch.cuda.synchronize()
        for i in range(n_sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                step_on(i, side)
            graphs.append(g)
        with torch.cuda.stream(side):
            for g in graphs:
                g.replay()
            ms = time_region(lambda i: graphs[i % n_sets].replay(), steps, side)
        return ms / steps
    except RuntimeError:
        torch.cuda.synchronize()
        return None


def kernel_breakdown(la, fn, steps: int, stream) -> dict:
    """Per-kernel device time of the same timed loop, from the library's launch
    trace (CUDA events recorded on the launching stream around each kernel)."""
    la.trace_enable(max(64, steps * 8))
    try:
        time_region(fn, steps, stream)
        recs = la.trace_collect(max(64, steps * 8))
    finally:
        la.trace_enable(0)
    out = {}
    for name, ms in recs:
        d = out.setdefault(name, {"launches": 0, "total_ms": 0.0})
        d["launches"] += 1
        d["total_ms"] += ms
    tot = sum(d["total_ms"] for d in out.values()) or 1.0
    for d in out.values():
        d["avg_ms"] = d["total_ms"] / d["launches"]
        d["ms_per_step"] = d["total_ms"] / steps
        d["share"] = d["total_ms"] / tot
    return out


def prefill_measure(la, name: str, steps: int, warmup: int, rank: int, world: int,
                    e2e: bool = False, batch: int | None = None) -> dict:
    c = dict(workloads.CONFIGS[name])
    if batch:
        c["B"] = batch
    B = c["B"]
    pairs = workloads.shard_pairs(rank, world, B, c["H"])
    cw = dict(c)
    cw["B"] = B * world
    x = workloads.make_inputs(cw, pairs=pairs)
    shape_qk = (B, c["H"], c["T"], c["dk"])
    shape_v = (B, c["H"], c["T"], c["dv"])
    q = x["q"].reshape(shape_qk)
    k = x["k"].reshape(shape_qk)
    v = x["v"].reshape(shape_v)
    gamma = x["gamma"]
    gated = bool(c.get("gate"))
    log_a = x["log_a"].reshape(B, c["H"], c["T"]) if gated else None
    dev = torch.device("cuda")
    per_set = alg_bytes(c)
    n_sets = max(1, min(16, (3 * L2_BYTES + per_set - 1) // per_set))
    sets = []
    for _ in range(n_sets):
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        O = torch.empty(shape_v, dtype=qd.dtype, device=dev)
        S = torch.empty(B, c["H"], feature_dim(c), c["dv"], device=dev)
        z = torch.empty(B, c["H"], feature_dim(c), device=dev) if c["normalize"] else None
        lad = log_a.to(dev) if gated else None
        sets.append((qd, kd, vd, O, S, z, lad))
    ws_n = la.workspace_size(B, c["H"], c["T"], c["dk"], c["dv"], qd.dtype, c["phi"],
                             c["normalize"], gated=gated, floor=c.get("floor", False))
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step_on(i, s):
        qd, kd, vd, O, S, z, lad = sets[i % n_sets]
        la.chunk_fwd(qd, kd, vd, None if gated else gamma, phi=c["phi"],
                     normalize=c["normalize"], floor=c.get("floor", False), out=O, S_out=S,
                     z_out=z, workspace=ws, stream=s, log_a=lad)

    def step(i):
        step_on(i, stream)

    for i in range(warmup):
        step(i)
    ms = time_region(step, steps, stream)
    kernels = kernel_breakdown(la, step, steps, stream)
    graph_ms = graph_replay_ms(step_on, n_sets, steps)
    flags = ((la.LA_PHI_TAYLOR if c["phi"] == "taylor" else la.LA_PHI_ELU1 if c["phi"] else 0)
             | (la.LA_NORMALIZE if c["normalize"] else 0)
             | (la.LA_NORM_FLOOR if c.get("floor") else 0) | (la.LA_GATED if gated else 0))
    launches = la.library().la_chunk_fwd_launches(B, c["H"], c["T"], c["dk"], c["dv"],
                                                  1 if c["dtype"] == "bf16" else 0, flags, 0)
    res = dict(name=name, config=c, ms=ms / steps, tokens=B * c["T"], n_sets=n_sets,
               graph_ms=graph_ms,
               alg_bytes=alg_bytes(c), alg_flops=alg_flops(c), launches=launches,
               kernels=kernels)
    if e2e:
        # through the C ABI's host-buffer entry point (la_chunk_fwd_host): pinned
        # inputs in, results out, every copy inside the timed region (device time,
        # CUDA events); the batch goes in one piece per batch row, pipelined
        qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
        Oh = torch.empty(shape_v, dtype=q.dtype, pin_memory=True)
        Sh = torch.empty(B, c["H"], c["dk"], c["dv"], pin_memory=True)
        zh = torch.empty(B, c["H"], c["dk"], pin_memory=True) if c["normalize"] else None
        arena = torch.empty(la.host_arena_size(B, c["H"], c["T"], c["dk"], c["dv"], q.dtype,
                                               c["phi"], c["normalize"], pieces=B),
                            dtype=torch.uint8, device=dev)

        def step_host(times):
            la.chunk_fwd_host(qh, kh, vh, gamma, phi=c["phi"], normalize=c["normalize"], pieces=B,
                              out=Oh, S_out=Sh, z_out=zh, timing=times, arena=arena)

        for _ in range(warmup):
            step_host(None)
        times = []
        for _ in range(steps):
            step_host(times)
        es = q.element_size()
        res["e2e_ms"] = sum(times) / len(times)
        res["h2d"] = (q.numel() + k.numel() + v.numel()) * es
        res["d2h"] = Oh.numel() * es + Sh.numel() * 4 + (zh.numel() * 4 if zh is not None else 0)
    del sets
    torch.cuda.empty_cache()
    return res


def bwd_bytes(c: dict) -> int:
    """Backward pass: read Q, K, V, dO, write dQ, dK, dV, and the initial state's
    gradient; with the normaliser the per-token denominators are written and
    read once (8 + 8 bytes per head-token)."""
    es = 2 if c["dtype"] == "bf16" else 4
    nbh = c["B"] * c["H"]
    per_tok = (2 * c["dk"] + 2 * c["dv"]) * es + (2 * c["dk"] + c["dv"]) * es
    if c["normalize"]:
        per_tok += 16
    return nbh * c["T"] * per_tok + nbh * c["dk"] * c["dv"] * 4


def bwd_measure(la, name: str, steps: int, warmup: int, rank: int, world: int) -> dict:
    """The backward pass (la_chunk_bwd) of a workload, with a seeded N(0,1) dO."""
    c = dict(workloads.CONFIGS[name])
    B, H, T = c["B"], c["H"], c["T"]
    pairs = workloads.shard_pairs(rank, world, B, H)
    cw = dict(c)
    cw["B"] = B * world
    x = workloads.make_inputs(cw, pairs=pairs)
    dev = torch.device("cuda")
    q = x["q"].reshape(B, H, T, c["dk"]).to(dev)
    k = x["k"].reshape(B, H, T, c["dk"]).to(dev)
    v = x["v"].reshape(B, H, T, c["dv"]).to(dev)
    dO = torch.from_numpy(workloads.normal_bhtd(c["seed"] + 100, workloads.V_ID, B, H, T, c["dv"],
                                                1.0)).to(q.dtype).to(dev)
    gamma = x["gamma"]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(16, la.library().la_bwd_workspace_size(
        B, H, T, c["dk"], c["dv"], 1 if c["dtype"] == "bf16" else 0,
        la.LA_NORMALIZE if c["normalize"] else 0)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        la.chunk_bwd(q, k, v, dO, gamma, phi=c["phi"], normalize=c["normalize"], dq=dq, dk=dk,
                     dv=dv, workspace=ws, stream=stream)

    for i in range(warmup):
        step(i)
    ms = time_region(step, steps, stream)
    res = dict(name=name, config=c, ms=ms / steps, tokens=B * T, bytes=bwd_bytes(c),
               kernels=kernel_breakdown(la, step, steps, stream))
    del q, k, v, dO, dq, dk, dv
    torch.cuda.empty_cache()
    return res


def decode_measure(la, steps_total: int, warmup: int, rank: int, world: int) -> dict:
    name = "decode_bf16"
    c = dict(workloads.CONFIGS[name])
    B, H = c["B"], c["H"]
    pairs = workloads.shard_pairs(rank, world, B, H)
    cw = dict(c)
    cw["B"] = B * world
    x = workloads.make_inputs(cw, pairs=pairs)
    dev = torch.device("cuda")
    q = x["q"].reshape(B, H, c["T"], c["dk"]).to(dev)
    k = x["k"].reshape(B, H, c["T"], c["dk"]).to(dev)
    v = x["v"].reshape(B, H, c["T"], c["dv"]).to(dev)
    gamma = x["gamma"]
    _, S, _ = la.chunk_fwd(q, k, v, gamma)
    torch.cuda.synchronize()
    del q, k, v, x
    torch.cuda.empty_cache()
    # every decode step's own inputs, resident before timing
    d = workloads.decode_inputs_all(cw, steps_total)
    bsl = slice(rank * B, (rank + 1) * B)
    dq = d["q"][:, bsl].contiguous().to(dev)
    dk = d["k"][:, bsl].contiguous().to(dev)
    dv = d["v"][:, bsl].contiguous().to(dev)
    o = torch.empty(steps_total, B, H, c["dv"], dtype=dq.dtype, device=dev)
    stream = torch.cuda.current_stream()
    S_warm = S.clone()

    for i in range(warmup):  # warm-up on a scratch copy of the state
        la.recurrent_step(dq[i], dk[i], dv[i], gamma, S_warm, out=o[i], stream=stream)
    del S_warm

    def step(i):
        la.recurrent_step(dq[i], dk[i], dv[i], gamma, S, out=o[i], stream=stream)

    ms = time_region(step, steps_total, stream)
    res = dict(name=name, config=c, ms=ms / steps_total, steps=steps_total,
               bytes=decode_bytes(c), flops=decode_flops(c))
    # (the traced repeat continues the same recurrence; only its timing is used)
    res["kernels"] = kernel_breakdown(la, step, min(steps_total, 64), stream)
    res["graph"] = decode_graph(la, dq, dk, dv, o, S, gamma, steps_total)
    del dq, dk, dv, o, S
    torch.cuda.empty_cache()
    return res


def bwd_path(kernels: dict) -> str:
    """The backward pass's path, from the kernels its traced step launched."""
    if "aug_prep_kernel" in kernels:
        return "CUDA cores (dq, per-token dd and du) and tensor cores (dk, dv: reversed-time passes)"
    if any(k.startswith("chunk_tc_ws_kernel") for k in kernels):
        return "tensor cores (three forward passes)"
    return "CUDA cores"


def decode_graph(la, dq, dk, dv, o, S, gamma, steps_total: int) -> dict:
    """The same decode steps captured once in a CUDA graph and replayed: the
    launches cost no host work.  The graph runs the recurrence on its own copy of
    the state.  Reported beside the stream-launched timing, not instead of it."""
    S_g = S.clone()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    try:
        with torch.cuda.graph(g, stream=side):
            for i in range(steps_total):
                la.recurrent_step(dq[i], dk[i], dv[i], gamma, S_g, out=o[i], stream=side)
    except RuntimeError as e:
        del S_g
        return {"unavailable": str(e).splitlines()[0][:200]}
    stream = torch.cuda.current_stream()
    g.replay()  # warm-up replay
    ms = time_region(lambda i: g.replay(), 1, stream)
    del g, S_g
    return {"ms_per_step": ms / steps_total, "steps": steps_total, "launches": steps_total}


def oracle_baseline(name: str, budget_s: float = 12.0) -> dict:
    """The fp64 oracle on the host cores, on whole (b, h) sequences of the workload."""
    import oracle
    c = workloads.CONFIGS[name]
    H = c["H"]
    pairs = workloads.sample_pairs(c["B"], H, max(1, min(c["B"] * H, oracle.num_threads())))
    x = workloads.make_inputs(c, pairs=pairs)
    g = x["gamma_pairs"]
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.recurrent(x["q"][None], x["k"][None], x["v"][None], g, phi=c["phi"],
                         normalize=c["normalize"])
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            break
    tok = reps * len(pairs) * c["T"] / H  # token = one position of all H heads
    return dict(value=tok / el, unit="tokens/s", cores=oracle.num_threads(), kind="oracle",
                sample=(f"{reps} x {len(pairs)} whole (b, h) sequences of T={c['T']} "
                        f"({describe(name, c)}); tokens counted per position of all {H} heads"),
                seconds=el)


def run_ours(args) -> dict | None:
    import retnet_retention_gb300 as la
    from retnet_retention_gb300 import _build
    _build.build()
    la.library()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x: float) -> float:
        if dist is None:
            return x
        t = torch.tensor([x], dtype=torch.float64, device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    pk = peaks()
    only = args.only
    if only == "decode":  # profiling aid: the decode workload alone
        dec = decode_measure(la, args.decode_steps, args.warmup, rank, world)
        if rank == 0:
            print(json.dumps({"only": "decode", "ms_per_step": dec["ms"],
                              "hbm_gbs": dec["bytes"] / (dec["ms"] * 1e-3) / 1e9,
                              "graph": dec["graph"]}))
        return None
    if only in ("backward", "backward_" + BWD_TC):  # profiling aid: one backward pass alone
        r = bwd_measure(la, BWD_NORM if only == "backward" else BWD_TC, args.steps, args.warmup,
                        rank, world)
        if rank == 0:
            print(json.dumps({"only": only, "ms": r["ms"],
                              "alg_gbs": r["bytes"] / (r["ms"] * 1e-3) / 1e9,
                              "kernel_ms_per_step": {k: round(v["total_ms"] / args.steps, 5)
                                                     for k, v in r["kernels"].items()}}))
        return None
    if only in (HEADLINE,) + SUB_PREFILL:  # profiling aid: one prefill workload alone
        r = prefill_measure(la, only, args.steps, args.warmup, rank, world, batch=args.batch)
        if rank == 0:
            print(json.dumps({"only": only, "ms_per_step": r["ms"],
                              "alg_gbs": r["alg_bytes"] / (r["ms"] * 1e-3) / 1e9,
                              "graph_ms_per_step": r["graph_ms"]}))
        return None
    barrier()
    sampler = ClockSampler(local)
    with sampler:
        head = prefill_measure(la, HEADLINE, args.steps, args.warmup, rank, world, e2e=True)
    barrier()
    head_ms = max_over_ranks(head["ms"])
    e2e_ms = max_over_ranks(head["e2e_ms"])
    others = {}
    headline_only = args.headline_only or only == "headline"
    if not headline_only:
        for name in SUB_PREFILL:
            r = prefill_measure(la, name, max(3, args.steps // 2), args.warmup, rank, world)
            r["ms"] = max_over_ranks(r["ms"])
            others[name] = r
        dec = decode_measure(la, args.decode_steps, args.warmup, rank, world)
        dec["ms"] = max_over_ranks(dec["ms"])
        bwds = {}
        for name in (BWD_NORM, BWD_TC):
            r = bwd_measure(la, name, 3, args.warmup, rank, world)
            r["ms"] = max_over_ranks(r["ms"])
            bwds[name] = r
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    c = head["config"]
    tokens_all = head["tokens"] * world
    value = tokens_all / (head_ms * 1e-3)
    dom_name, dom = max(head["kernels"].items(), key=lambda kv: kv[1]["total_ms"])
    # the dominant kernel processes the whole workload once per launch
    achieved_gbs = head["alg_bytes"] / (dom["avg_ms"] * 1e-3) / 1e9
    useful_tflops = head["alg_flops"] / (head["ms"] * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) inputs, see workloads/)",
        "config": {
            "workload": describe(HEADLINE, c),
            "global_batch": c["B"] * world,
            "seq_len": c["T"],
            "parallelism": "replicas" if world == 1 else f"batch-sharded x{world}",
            "l2": f"inputs rotate over {head['n_sets']} copies ({head['n_sets'] * head['alg_bytes'] / 1e6:.0f} MB > L2)",
        },
        "tflops_useful": useful_tflops,
        "pct_bf16_peak": 100.0 * useful_tflops / pk["bf16_tflops"],
        "roofline": {
            "bound": "hbm",
            "achieved": achieved_gbs,
            "peak": pk["hbm_gbs"],
            "unit": "GB/s",
            "frac": achieved_gbs / pk["hbm_gbs"],
            "traffic": measured_traffic(HEADLINE, dom_name),
            "kernel": dom_name,
            "kernel_avg_ms": dom["avg_ms"],
            "peak_source": pk["source"],
        },
        "kernels": head["kernels"],
        # the same steps replayed from CUDA graphs (no host work per launch); context
        "graph_ms_per_step": head.get("graph_ms"),
        "e2e": {
            "value": tokens_all / (e2e_ms * 1e-3),
            "unit": "tokens/s",
            "h2d_bytes_per_step": head["h2d"],
            "d2h_bytes_per_step": head["d2h"],
        },
        "gpu_launches": args.steps * head["launches"],
    }
    if not headline_only:
        sub = {}
        for name, r in others.items():
            rc = r["config"]
            gbs = r["alg_bytes"] / (r["ms"] * 1e-3) / 1e9
            tf = r["alg_flops"] / (r["ms"] * 1e-3) / 1e12
            # the dominant kernel's launches of a step (one, or the two builds of a split
            # walk) process the workload once
            dn, dk_ = max(r["kernels"].items(), key=lambda kv: kv[1]["total_ms"])
            kgbs = r["alg_bytes"] / (dk_["ms_per_step"] * 1e-3) / 1e9
            ktf = r["alg_flops"] / (dk_["ms_per_step"] * 1e-3) / 1e12
            # the bound: whichever of the algorithmic bytes and flops takes longer at peak
            tensor = r["alg_flops"] / (pk["bf16_tflops"] * 1e12) > r["alg_bytes"] / (pk["hbm_gbs"] * 1e9)
            sub[name] = dict(workload=describe(name, rc), tokens_per_s=r["tokens"] * world /
                             (r["ms"] * 1e-3), ms=r["ms"], alg_gbs=gbs,
                             step_roofline_frac=gbs / pk["hbm_gbs"], tflops_useful=tf,
                             pct_bf16_peak=100.0 * tf / pk["bf16_tflops"],
                             dominant_kernel=dn, kernel_gbs=kgbs, kernel_tflops=ktf,
                             bound="tensor" if tensor else "hbm",
                             roofline_frac=(ktf / pk["bf16_tflops"]) if tensor else kgbs / pk["hbm_gbs"],
                             graph_ms=r.get("graph_ms"), kernels=r["kernels"])
        dc = dec["config"]
        gbs = dec["bytes"] / (dec["ms"] * 1e-3) / 1e9
        for name, bwd in bwds.items():
            bc = bwd["config"]
            bgbs = bwd["bytes"] / (bwd["ms"] * 1e-3) / 1e9
            sub["backward_" + name] = dict(
                workload="backward of " + describe(name, bc) + " (gradients of Q, K, V and of "
                         "the initial state for a seeded N(0,1) dO)",
                path=bwd_path(bwd["kernels"]),
                tokens_per_s=bwd["tokens"] * world / (bwd["ms"] * 1e-3), ms=bwd["ms"],
                alg_gbs=bgbs, roofline_frac=bgbs / pk["hbm_gbs"], kernels=bwd["kernels"])
        sub["decode_bf16"] = dict(
            workload=f"decode_bf16: B={dc['B']} H={dc['H']} d_k={dc['dk']} d_v={dc['dv']} fp32 "
                     f"state after a {dc['T']}-token prefill, {dec['steps']} steps",
            steps_per_s=1e3 / dec["ms"], ms_per_step=dec["ms"], hbm_gbs=gbs,
            roofline_frac=gbs / pk["hbm_gbs"], kernel="decode_step_kernel",
            kernels=dec["kernels"], graph=dec["graph"])
        line["workloads"] = sub
    clocks = sampler.summary()
    if clocks is not None:
        line["clocks"] = clocks
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(HEADLINE)
    if dist is not None:
        dist.destroy_process_group()
    return line


def run_reference(args) -> dict | None:
    """The oracle as it stands, on the host cores, on bounded samples of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    c = workloads.CONFIGS[HEADLINE]
    H = c["H"]
    n = max(1, min(c["B"] * H, oracle.num_threads()))
    pairs = workloads.sample_pairs(c["B"], H, n)
    x = workloads.make_inputs(c, pairs=pairs)
    g = x["gamma_pairs"]

    def one():
        oracle.recurrent(x["q"][None], x["k"][None], x["v"][None], g, phi=c["phi"],
                         normalize=c["normalize"])

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    tok_per_step = len(pairs) * c["T"] / H
    value = args.steps * tok_per_step / el
    sample = (f"each step: {len(pairs)} whole (b, h) sequences of T={c['T']} of "
              f"{describe(HEADLINE, c)}; tokens counted per position of all {H} heads")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(HEADLINE, c), "global_batch": c["B"],
                   "seq_len": c["T"], "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--headline-only", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=("headline", HEADLINE) + SUB_PREFILL +
                    ("decode", "backward", "backward_" + BWD_TC),
                    default=None,
                    help="profiling aid: run one workload only")
    ap.add_argument("--batch", type=int, default=None,
                    help="profiling aid (with --only and a prefill workload): a smaller batch B")
    ap.add_argument("--decode-steps", type=int,
                    default=workloads.CONFIGS["decode_bf16"]["decode_steps"],
                    help="decode steps to time (the workload has 1024)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
