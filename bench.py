#!/usr/bin/env python
"""Benchmark of the speculative-sampling verify step on GB300.

One step = one spv_verify_chain call (accept test, first-rejection stop,
residual or bonus draw) over one batch of the sweep workload at the metric's
shape: B = 64 sequences, gamma = 4, V = 151,936, fp32 logits, T = 1
(synthetic, seeded; see speculative_decoding_token_spv_gb300.workloads).
A call is two kernel launches (streaming grid + dependent finalize grid);
the timed steps are issued from a CUDA graph of consecutive calls (the eager
loop is timed too and reported as eager_ms_per_step).

Prints ONE JSON line.  value = verified target rows per second
(B * (gamma + 1) per step) over all ranks; the roofline object gives the HBM
bandwidth the kernel reaches with the ALGORITHMIC bytes of a step (every
target and draft logit once, plus the tokens, uniforms, keys and outputs)
against the measured copy peak.  Inputs (2 sets, 350 MB each) exceed the
129 MB L2, and consecutive steps alternate between the sets.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 launch under torchrun: every rank verifies its own batch (weak
scaling, no data-path collective; the barrier and the max-over-ranks timing
are the only communication).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(name="sweep", B=64, gamma=4, V=151936, dtype="float32", T=1.0)
METRIC = "verified logit rows/s (V=151936, gamma=4)"


# ----------------------------------------------------------------- algorithmic bytes
def chain_bytes(B, gamma, V, elem_bytes, T):
    """Bytes the method reads and writes once: every logit row once, draft
    tokens, r, keys, and the outputs (accept count + gamma+1 ids)."""
    if T == 0:
        return B * (gamma + 1) * V * elem_bytes + B * gamma * 4 + B * (gamma + 2) * 4
    return B * (2 * gamma + 1) * V * elem_bytes + B * gamma * 8 + B * 8 + B * (gamma + 2) * 4


def tree_bytes(B, N, internal, V, elem_bytes, T):
    """Tree verify: every target row once, the draft rows of the nodes with
    children once (a leaf's draft row is not read), parents and tokens, and
    at T > 0 r and keys; outputs: accept count, N ids and N nodes."""
    rows = N if T == 0 else N + internal
    extra = 0 if T == 0 else B * N * 4 + B * 8
    return B * rows * V * elem_bytes + B * N * 8 + extra + B * (2 * N + 1) * 4


def fanout_bytes(B, K1, V, elem_bytes, sumF):
    return B * K1 * V * elem_bytes + B * K1 * 4 + B * sumF * 4


# ----------------------------------------------------------------- distributed helpers
def dist_init():
    """(rank, world); initialises torch.distributed only under torchrun."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("SPV_BENCH_BACKEND") or ("nccl" if _cuda_ok() else "gloo")
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
    return rank, world


def _cuda_ok():
    import torch
    return torch.cuda.is_available()


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        if dist.get_backend() == "nccl":
            import torch
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def dist_max(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(rows_local: float, ms_local: float, world: int):
    """Whole-job throughput: rows of all ranks over the slowest rank's time."""
    ms_max = dist_max(ms_local, world)
    total_rows = dist_sum(rows_local, world)
    return total_rows / (ms_max * 1e-3), ms_max, total_rows


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_token_spv_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(tag: str):
    """DRAM bytes per launch recorded under profiles/ for this exact kernel
    source (None once the sources changed since the capture)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_source_hash()
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == tag and parts[1] == want:
                return float(parts[2])
    return None


def make_chain_inputs(dev, B, gamma, V, dtype, T, sets=2):
    import torch

    from speculative_decoding_token_spv_gb300 import workloads
    dt = getattr(torch, dtype)
    out = []
    for s in range(sets):
        w = workloads.sweep(B=B, dtype=dt, device=dev, temperature=T, V=V, gamma=gamma)
        if s:
            # a second, distinct set: different uniforms/keys, logits rolled by one row
            w.target = torch.roll(w.target, 1, 0).contiguous()
            w.draft = torch.roll(w.draft, 1, 0).contiguous()
        out.append(w)
    return out


def time_replays(replay, replays, stream):
    """Device ms of each of `replays` consecutive graph replays (CUDA events
    between them on `stream`) and of all of them together."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(replays + 1)]
    ev[0].record(stream)
    for i in range(replays):
        replay(i)
        ev[i + 1].record(stream)
    ev[-1].synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(replays)]
    return per, ev[0].elapsed_time(ev[-1])


def parity_against_oracle(got, ref, B, g):
    """Compare the timed call's outputs with the oracle's on the same inputs:
    sequences that differ with an oracle decision margin >= 1e-6 (must be 0),
    near-tie sequences (margin < 1e-6) and the largest relative error of
    p_i(x_i), q_i(x_i)."""
    import numpy as np
    k_got = got["accept_count"].cpu().numpy()
    t_got = got["out_tokens"].cpu().numpy()
    same = (k_got == ref["accept_count"]) & (t_got == ref["out_tokens"]).all(axis=1) & \
        (got["row_status"].cpu().numpy() == ref["status"])
    near = ref["margin"] < 1e-6
    ok = ref["status"] == 0
    pq = got["pq"].float().cpu().numpy()[ok]
    rel = np.abs(pq - ref["pq"][ok]) / np.maximum(np.abs(ref["pq"][ok]), 1e-30)
    return {"sequences": int(B), "positions": int(B * (g + 1)), "far_mismatches": int((~same & ~near).sum()),
            "near_ties": int(near.sum()), "near_tie_mismatches": int((~same & near).sum()),
            "pq_max_rel_err": float(rel.max()) if rel.size else 0.0,
            "checked": "outputs of the timed graph replays (input set 0) against the oracle, same run"}


def time_device(fn, steps, warmup, stream):
    """Average ms per call over `steps` calls (CUDA events on `stream`)."""
    import torch
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        fn(i)
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / steps


# ----------------------------------------------------------------- our arm
def run_spv(args, rank, world):
    import numpy as np
    import torch

    import speculative_decoding_token_spv_gb300 as spv
    from speculative_decoding_token_spv_gb300 import build as spv_build

    if rank == 0 or not os.path.exists(spv.LIB_PATH):
        spv_build.build_library()
    dist_barrier(world)
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    W = dict(WORKLOAD)
    B, g, V, T = W["B"], W["gamma"], W["V"], W["T"]
    eb = 4 if W["dtype"] == "float32" else 2
    sets = make_chain_inputs(dev, B, g, V, W["dtype"], T)
    ws = spv.new_workspace(spv.spv_chain_workspace_bytes(B, g, V), dev)
    outs = [spv.spv_verify_chain(s.target, s.draft, s.tokens, s.r, s.keys, T, workspace=ws, want_pq=True)
            for s in sets]
    torch.cuda.synchronize()

    def step(i):
        s = sets[i % 2]
        spv.spv_verify_chain(s.target, s.draft, s.tokens, s.r, s.keys, T, workspace=ws, out=outs[i % 2])

    algo = chain_bytes(B, g, V, eb, T)
    # The timed steps are issued from a CUDA graph of consecutive calls
    # (alternating input sets): K calls in all, as `replays` (at least 5 when
    # K allows) replays of a graph holding `graph_calls` of them, each replay
    # timed on its own for the median and the best.  The eager call loop is
    # timed too and reported beside it.
    cap_calls = max(1, min(200, args.steps // 5))
    graph_calls = next(c for c in range(cap_calls, 0, -1) if args.steps % c == 0)
    replays = args.steps // graph_calls
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for i in range(4):
            step(i)
        cap.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(graph_calls):
                step(i)
    torch.cuda.synchronize()

    def replay(_):
        graph.replay()

    # ---- timed region (device) with clock sampling
    dist_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        per_replay, total_ms = time_replays(replay, replays, stream)
    ms = total_ms / args.steps
    timed_out = {k: v.clone() for k, v in outs[0].items()}  # the timed calls' outputs on input set 0
    per_call = sorted(x / graph_calls for x in per_replay)
    ms_eager = time_device(step, args.steps, args.warmup, stream)
    dist_barrier(world)
    rows = B * (g + 1)
    value, ms_max, total_rows = aggregate(float(rows), ms, world)
    clocks = clk.summary()
    assert spv.spv_workspace_status(ws) == spv.SPV_OK

    # ---- end to end through the public API with host buffers
    host = []
    for s in sets:
        h = {k: getattr(s, k).cpu().pin_memory() for k in ("target", "draft", "tokens", "r", "keys")}
        host.append(h)
    dbuf = {k: torch.empty_like(getattr(sets[0], k)) for k in ("target", "draft", "tokens", "r", "keys")}
    hout = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs[0].items()}
    h2d = sum(v.numel() * v.element_size() for v in host[0].values())
    d2h = sum(v.numel() * v.element_size() for v in hout.values())

    def e2e_step(i):
        h = host[i % 2]
        for k, v in h.items():
            dbuf[k].copy_(v, non_blocking=True)
        o = spv.spv_verify_chain(dbuf["target"], dbuf["draft"], dbuf["tokens"], dbuf["r"], dbuf["keys"], T,
                                 workspace=ws, out=outs[0])
        for k, v in o.items():
            hout[k].copy_(v, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20))
    dist_barrier(world)
    ms_e2e = time_device(e2e_step, e2e_steps, 2, stream)
    ms_e2e_max = dist_max(ms_e2e, world)

    peak, peak_kind = measured_peaks()
    achieved = algo / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "timing": f"CUDA graph of {graph_calls} calls replayed {replays}x; eager call loop {ms_eager * 1e3:.2f} us/step",
        "replay_ms_per_step": {"replays": replays, "calls_per_replay": graph_calls,
                               "median": statistics.median(per_call), "best": per_call[0], "worst": per_call[-1]},
        "eager_ms_per_step": ms_eager,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; sweep workload distributions)",
        "config": {"workload": f"chain verify B={B} gamma={g} V={V} fp32 T=1", "B": B, "gamma": g, "V": V,
                   "logits": W["dtype"], "temperature": T, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (2 sets x 350 MB, alternating)"},
        "gb_per_s": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": ncu_traffic("chain_f32_B64"), "algorithmic_bytes": algo,
                     "frac_of_8000": achieved / 8000.0},
        "clocks": clocks,
        "e2e": {"value": total_rows / (ms_e2e_max * 1e-3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e_max},
        "gpu_launches": 2 * args.steps,
    }
    if rank == 0 and not args.no_variants:
        line["variants"] = run_variants(spv, dev, stream, args)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"], ref = cpu_baseline(sets[0], B, g, V, T)
        line["parity"] = parity_against_oracle(timed_out, ref, B, g)
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_graph(fn, n_inner=20, n_outer=10):
    """Average device ms per call of `fn` replayed from a CUDA graph that holds
    `n_inner` calls (launch overhead of the host removed)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(n_inner):
                fn()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(n_outer):
        g.replay()
    b.record(st)
    b.synchronize()
    return a.elapsed_time(b) / (n_outer * n_inner)


def run_variants(spv, dev, stream, args):
    """Every hot-path row on its own workload: device time per call, replayed
    from a CUDA graph (small calls are otherwise bound by host launch cost)."""
    import torch

    from speculative_decoding_token_spv_gb300 import workloads
    peak, _ = measured_peaks()
    res = []

    def add(name, ms, algo, rows):
        gbs = algo / (ms * 1e-3) / 1e9
        res.append({"workload": name, "ms": round(ms, 5), "rows_per_s": rows / (ms * 1e-3), "gb_per_s": round(gbs, 1),
                    "frac_measured": round(gbs / peak, 4), "frac_8000": round(gbs / 8000.0, 4),
                    "algorithmic_bytes": algo, "timing": "cuda graph replay"})

    cases = [("sweep B=64 fp32 T=0", lambda: workloads.sweep(B=64, dtype=torch.float32, device=dev, temperature=0.0)),
             ("sweep B=64 bf16 T=1", lambda: workloads.sweep(B=64, dtype=torch.bfloat16, device=dev)),
             ("sweep B=128 fp32 T=1", lambda: workloads.sweep(B=128, dtype=torch.float32, device=dev)),
             ("sweep B=256 fp32 T=1", lambda: workloads.sweep(B=256, dtype=torch.float32, device=dev)),
             ("sweep B=256 bf16 T=1", lambda: workloads.sweep(B=256, dtype=torch.bfloat16, device=dev)),
             ("sweep B=256 fp32 T=0", lambda: workloads.sweep(B=256, dtype=torch.float32, device=dev, temperature=0.0)),
             ("sweep B=8 fp32 T=1", lambda: workloads.sweep(B=8, dtype=torch.float32, device=dev)),
             ("sweep B=1 fp32 T=1", lambda: workloads.sweep(B=1, dtype=torch.float32, device=dev)),
             ("tiny B=1 g=4 V=1000 fp32 T=1", lambda: workloads.tiny(device=dev)),
             ("spd B=64 g=1 bf16 T=1", lambda: workloads.spd(device=dev)),
             ("spd B=64 g=1 bf16 T=0", lambda: workloads.spd(device=dev, temperature=0.0)),
             ("eagle B=32 g=7 bf16 T=1", lambda: workloads.eagle(gamma=7, device=dev)),
             ("eagle B=32 g=15 bf16 T=1", lambda: workloads.eagle(gamma=15, device=dev)),
             ("eagle B=32 g=15 bf16 T=0", lambda: workloads.eagle(gamma=15, device=dev, temperature=0.0))]
    for name, mk in cases:
        w = mk()
        eb = w.target.element_size()
        ws = spv.new_workspace(spv.spv_chain_workspace_bytes(w.B, w.gamma, w.V), dev)
        o = spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, w.temperature, workspace=ws)
        ms = time_graph(lambda: spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, w.temperature,
                                                     workspace=ws, out=o))
        add(name, ms, chain_bytes(w.B, w.gamma, w.V, eb, w.temperature), w.B * (w.gamma + 1))
        del w, o, ws
    fw = workloads.fanout(device=dev)
    ws = spv.new_workspace(spv.spv_fanout_workspace_bytes(8, 4, fw.draft.shape[2], max(fw.fanout)), dev)
    o = spv.spv_fanout_topk(fw.draft, fw.exclude, fw.fanout, workspace=ws)
    ms = time_graph(lambda: spv.spv_fanout_topk(fw.draft, fw.exclude, fw.fanout, workspace=ws, out=o))
    add("fanout B=8 K=4 fp32 F=[8,7,6,5,4]", ms, fanout_bytes(8, 5, fw.draft.shape[2], 4, sum(fw.fanout)), 8 * 5)
    del fw, o, ws
    # Verify on top-k / top-p filtered distributions (the SPD sampling setup:
    # top-k 50, top-p 1.0 at T = 1); same logit bytes as the unfiltered call.
    fcases = [("filtered spd B=64 g=1 bf16 T=1 top-k 50", lambda: workloads.spd(device=dev, top_k=50), 50, 1.0),
              ("filtered sweep B=64 fp32 T=1 top-k 50", lambda: workloads.sweep(B=64, device=dev, top_k=50), 50, 1.0),
              ("filtered sweep B=64 bf16 T=1 top-k 50",
               lambda: workloads.sweep(B=64, dtype=torch.bfloat16, device=dev, top_k=50), 50, 1.0),
              ("filtered sweep B=256 fp32 T=1 top-k 50", lambda: workloads.sweep(B=256, device=dev, top_k=50), 50, 1.0),
              ("filtered eagle B=32 g=15 bf16 T=1 top-k 50 top-p 0.9",
               lambda: workloads.eagle(gamma=15, device=dev, top_k=50, top_p=0.9), 50, 0.9)]
    for name, mk, fk, fp in fcases:
        w = mk()
        ws = spv.new_workspace(spv.spv_filtered_workspace_bytes(w.B, w.gamma, w.V), dev)
        o = spv.spv_verify_chain_filtered(w.target, w.draft, w.tokens, w.r, w.keys, 1.0, fk, fp, workspace=ws)
        ms = time_graph(lambda: spv.spv_verify_chain_filtered(w.target, w.draft, w.tokens, w.r, w.keys, 1.0, fk, fp,
                                                              workspace=ws, out=o))
        add(name, ms, chain_bytes(w.B, w.gamma, w.V, w.target.element_size(), 1.0), w.B * (w.gamma + 1))
        del w, o, ws
    # Verify fused with the speculation-cache lookup; the cache is the fan-out
    # of the draft rows at positions 0..gamma.  The hit rate is a property of
    # the synthetic workload (reported over 32 draws of the sampling keys).
    for T in (1.0, 0.0):
        w = workloads.sweep(B=64, device=dev, temperature=T, bonus_draft=True)
        F = spv.fanout_sizes(8, 0.8, 0.5, w.gamma, w.V)
        d, ex = workloads.cache_fanout_inputs(w)
        lists = spv.spv_fanout_topk(d, ex, F)["ids"]
        del d
        ws = spv.new_workspace(spv.spv_chain_workspace_bytes(w.B, w.gamma, w.V), dev)
        o = spv.spv_verify_chain_cached(w.target, w.draft, w.tokens, w.r, w.keys, T, lists, F, workspace=ws)
        ms = time_graph(lambda: spv.spv_verify_chain_cached(w.target, w.draft, w.tokens, w.r, w.keys, T, lists, F,
                                                            workspace=ws, out=o))
        hits, n = 0, 0
        gen = torch.Generator(device=dev).manual_seed(77)
        for _ in range(32 if T > 0 else 1):
            keys = torch.randint(-(2 ** 63), 2 ** 63 - 1, (w.B,), generator=gen, device=dev, dtype=torch.int64)
            r = 1.0 - torch.rand(w.B, w.gamma, generator=gen, device=dev)
            oo = spv.spv_verify_chain_cached(w.target, w.draft, w.tokens, r, keys, T, lists, F, workspace=ws)
            hits += int((oo["cache_slot"] >= 0).sum())
            n += w.B
        add(f"cached verify sweep B=64 fp32 T={T:g} F={F}", ms,
            chain_bytes(w.B, w.gamma, w.V, 4, T) + w.B * (sum(F) + 1) * 4, w.B * (w.gamma + 1))
        res[-1]["cache_hit_rate"] = round(hits / n, 4)
        res[-1]["cache_hit_sample"] = f"{n} verify outcomes"
        del w, o, ws, lists
    # Saguaro sampling: drafts drawn with the cached candidates' probability
    # divided by C; acceptance falls and the cache hit rate rises with C.
    w = workloads.sweep(B=64, device=dev, bonus_draft=True)
    F = [8, 7, 6, 5, 4]
    d, _ = workloads.cache_fanout_inputs(w)
    lists = spv.spv_fanout_topk(d, torch.full((w.B, w.gamma + 1), -1, dtype=torch.int32, device=dev), F)["ids"]
    del d
    ws = spv.new_workspace(spv.spv_chain_workspace_bytes(w.B, w.gamma, w.V), dev)
    for C in (1.0, 2.0, 4.0, 8.0):
        gen = torch.Generator(device=dev).manual_seed(91)
        hits, acc, n = 0, 0, 0
        for rep in range(16):
            tok = workloads.saguaro_tokens(w, lists, F, C, seed=100 + rep)
            keys = torch.randint(-(2 ** 63), 2 ** 63 - 1, (w.B,), generator=gen, device=dev, dtype=torch.int64)
            r = 1.0 - torch.rand(w.B, w.gamma, generator=gen, device=dev)
            oo = spv.spv_verify_chain_saguaro(w.target, w.draft, tok, r, keys, 1.0, lists, F, C, workspace=ws)
            hits += int((oo["cache_slot"] >= 0).sum())
            acc += int(oo["accept_count"].sum())
            n += w.B
        o = spv.spv_verify_chain_saguaro(w.target, w.draft, tok, w.r, w.keys, 1.0, lists, F, C, workspace=ws)
        ms = time_graph(lambda: spv.spv_verify_chain_saguaro(w.target, w.draft, tok, w.r, w.keys, 1.0, lists, F, C,
                                                             workspace=ws, out=o))
        add(f"saguaro verify sweep B=64 fp32 T=1 C={C:g} F={F}", ms,
            chain_bytes(w.B, w.gamma, w.V, 4, 1.0) + w.B * (sum(F) + 1) * 4, w.B * (w.gamma + 1))
        res[-1]["cache_hit_rate"] = round(hits / n, 4)
        res[-1]["mean_accepted"] = round(acc / n, 4)
        res[-1]["sample"] = f"{n} verify outcomes"
    del w, ws, lists
    # Tree verify (multi-round speculative sampling over a draft tree per
    # sequence): the 21-node tree, the width-4 tree and a 63-node binary tree
    # on the spd rows.
    tcases = [("k21", 1.0, torch.bfloat16), ("k21", 0.0, torch.bfloat16), ("w4", 1.0, torch.bfloat16),
              ("k21", 1.0, torch.float32), ("b63", 1.0, torch.bfloat16)]
    for shape, T, dt in tcases:
        w = workloads.tree(B=64, shape=shape, dtype=dt, temperature=T, device=dev)
        ws = spv.new_workspace(spv.spv_tree_workspace_bytes(w.B, w.N, w.V), dev)
        o = spv.spv_verify_tree(w.target, w.draft, w.parent, w.tokens, w.r, w.keys, T, workspace=ws)
        ms = time_graph(lambda: spv.spv_verify_tree(w.target, w.draft, w.parent, w.tokens, w.r, w.keys, T,
                                                    workspace=ws, out=o))
        internal = len(set(workloads.tree_parents(workloads.TREE_SHAPES[shape])[1:]))
        add(f"tree verify {shape} (N={w.N}) B=64 {str(dt).replace('torch.', '')} T={T:g}", ms,
            tree_bytes(w.B, w.N, internal, w.V, w.target.element_size(), T), w.B * w.N)
        res[-1]["mean_accepted"] = round(float(o["accept_count"].float().mean()), 4)
        del w, ws, o
    torch.cuda.synchronize()
    return res


def cpu_baseline(w, B, g, V, T, budget_s=1.5, single_budget_s=1.0):
    """The oracle, as it stands, on the host cores: the full batch of the
    workload, repeated until `budget_s` of wall time (about 10-30 s of CPU
    work on a 16-core host), then on one core over the first sequences of the
    batch until `single_budget_s`.  Returns (the baseline object, the oracle's
    outputs on the batch, for the parity check of the timed call)."""
    import numpy as np

    import oracle
    oracle.build()
    t = w.target.float().cpu().numpy()
    d = w.draft.float().cpu().numpy()
    tok = w.tokens.cpu().numpy()
    r = w.r.cpu().numpy()
    keys = w.keys.cpu().numpy().view(np.uint64)
    cores = len(os.sched_getaffinity(0))
    reps, t0 = 0, time.perf_counter()
    ref = None
    while True:
        o = oracle.verify_chain(t, d, tok, r, keys, T, threads=cores)
        if ref is None:
            ref = o
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    n1, t1 = 0, time.perf_counter()
    while True:  # one core, one sequence at a time
        b = n1 % B
        oracle.verify_chain(t[b:b + 1], d[b:b + 1], tok[b:b + 1], r[b:b + 1], keys[b:b + 1], T, threads=1)
        n1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= single_budget_s:
            break
    base = {"value": B * (g + 1) * reps / el, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} pass(es) over the full B={B} batch (gamma={g}, V={V}), {el:.1f} s wall",
            "single_thread": {"value": n1 * (g + 1) / el1, "unit": "rows/s", "cores": 1,
                              "sample": f"{n1} sequence(s) of the batch one at a time, {el1:.1f} s wall"}}
    return base, ref


# ----------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The oracle as the reference arm: same workload, metric and unit, on the
    host cores; each step is one pass over a bounded sample of the batch."""
    import numpy as np

    import oracle
    if rank != 0:
        return
    oracle.build()
    import torch

    from speculative_decoding_token_spv_gb300 import workloads
    W = dict(WORKLOAD)
    B, g, V, T = W["B"], W["gamma"], W["V"], W["T"]
    w = workloads.sweep(B=B, dtype=torch.float32, device="cpu", temperature=T, V=V, gamma=g)
    nb = B  # every step verifies the full batch (about 50 ms on 16 host cores)
    t = w.target[:nb].numpy()
    d = w.draft[:nb].numpy()
    tok = w.tokens[:nb].numpy()
    r = w.r[:nb].numpy()
    keys = w.keys[:nb].numpy().view(np.uint64)
    cores = len(os.sched_getaffinity(0))
    for _ in range(args.warmup):
        oracle.verify_chain(t, d, tok, r, keys, T, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify_chain(t, d, tok, r, keys, T, threads=cores)
    el = time.perf_counter() - t0
    value = nb * (g + 1) * args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; sweep workload distributions)",
            "config": {"workload": f"chain verify B={B} gamma={g} V={V} fp32 T=1", "B": B, "gamma": g, "V": V,
                       "logits": "float32", "temperature": T, "parallelism": "cpu oracle"},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                             "sample": f"the full batch of {B} sequences per step, {args.steps} steps"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def profile_case(args):
    """Run one workload `--iters` times with no timing (a small command for ncu)."""
    import torch

    import speculative_decoding_token_spv_gb300 as spv
    from speculative_decoding_token_spv_gb300 import build as spv_build
    from speculative_decoding_token_spv_gb300 import workloads
    spv_build.build_library()
    dev = torch.device("cuda", 0)
    name, dt, B, T = args.profile_case, getattr(torch, args.dtype), args.B, args.T
    if name == "fanout":
        fw = workloads.fanout(device=dev)
        ws = spv.new_workspace(spv.spv_fanout_workspace_bytes(fw.draft.shape[0], 4, fw.draft.shape[2], 8), dev)
        for _ in range(args.iters):
            spv.spv_fanout_topk(fw.draft, fw.exclude, fw.fanout, workspace=ws)
    elif name.startswith("tree"):
        w = workloads.tree(B=B, shape=name[5:] or "k21", dtype=dt, temperature=T, device=dev)
        ws = spv.new_workspace(spv.spv_tree_workspace_bytes(w.B, w.N, w.V), dev)
        for _ in range(args.iters):
            spv.spv_verify_tree(w.target, w.draft, w.parent, w.tokens, w.r, w.keys, T, workspace=ws)
    else:
        fk = dict(top_k=args.top_k, top_p=args.top_p) if args.top_k else {}
        if name == "sweep":
            w = workloads.sweep(B=B, dtype=dt, device=dev, temperature=T, **fk)
        elif name == "spd":
            w = workloads.spd(device=dev, temperature=T, **fk)
        else:
            w = workloads.eagle(gamma=int(name[5:] or 7), device=dev, temperature=T, **fk)
        if args.top_k:
            ws = spv.new_workspace(spv.spv_filtered_workspace_bytes(w.B, w.gamma, w.V), dev)
            for _ in range(args.iters):
                spv.spv_verify_chain_filtered(w.target, w.draft, w.tokens, w.r, w.keys, w.temperature, args.top_k,
                                              args.top_p, workspace=ws)
        else:
            ws = spv.new_workspace(spv.spv_chain_workspace_bytes(w.B, w.gamma, w.V), dev)
            for _ in range(args.iters):
                spv.spv_verify_chain(w.target, w.draft, w.tokens, w.r, w.keys, w.temperature, workspace=ws)
    torch.cuda.synchronize()
    print("profile case done:", name, args.dtype, B, T, args.iters)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="spv", choices=["spv", "reference"])
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", default=None, help="sweep | spd | eagle7 | eagle15 | fanout | tree_k21 | tree_w4")
    ap.add_argument("--dtype", default="float32")
    ap.add_argument("--B", type=int, default=64)
    ap.add_argument("--T", type=float, default=1.0)
    ap.add_argument("--top-k", type=int, default=0, help="profile case: filtered verify with this top_k")
    ap.add_argument("--top-p", type=float, default=1.0)
    ap.add_argument("--iters", type=int, default=4)
    args = ap.parse_args(argv)
    if args.profile_case:
        profile_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    rank, world = dist_init()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_spv(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
