#!/usr/bin/env python3
"""Benchmark of the decode-step MoE layer tail on GB300: microseconds per call and achieved
HBM GB/s, for the 8-row, 256-expert top-8 workload with ~40% repeated picks
(r8_h7168_e256k8_similar: H 7168, I 2048, shared inter 2048).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one full call of the tail (add+RMSNorm, router, top-k, dedup, routed MXFP4
experts, bf16 shared expert, combine) on its own 8-row input set.  Consecutive steps run on
different copies of the layer's weights (L = max(4, ceil(4 x L2 / bytes per call)) copies,
one library handle each, like consecutive decoder layers), so no step finds its weights in
L2 and no flush is needed.  Besides the K timed steps the line carries the protocol
statistic: a CUDA graph of L calls replayed 7 trials x 50 replays in 2 rounds, median per
call.  --workload picks another of the five workloads.

Prints one JSON line (rank 0).  Multi-GPU runs (torchrun) are independent replicas: the
path has no cross-GPU exchange; value = all ranks' calls / max-over-ranks time.

--impl reference times the CPU oracle (plain C, fp64) on the host cores instead, each step
one bounded sample (one row of a call), scaled to microseconds per call.

--attnres-mix ROWS measures the second workload instead: the AttnRes residual mix over a
187-call decoder sequence (H 7168) on ROWS rows, one CUDA-graph replay of the sequence per
step, microseconds per call (with --impl reference: the oracle, one call per step).
"""
import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from moe_layer_tail_gb300 import inputs as gen  # noqa: E402

METRIC = "us_per_call"
UNIT = "us/call"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=gen.BENCH_WORKLOAD)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-protocol", action="store_true",
                   help="skip the CUDA-graph protocol statistic (7 trials x 50 replays x 2 "
                        "rounds)")
    p.add_argument("--experts", type=int, default=0,
                   help="profiling aid: the workload with this many experts instead (a "
                        "smaller case of the same kernels, e.g. for an ncu capture); the "
                        "line's config says so")
    p.add_argument("--weight-copies", type=int, default=0,
                   help="profiling aid: rotate over this many weight copies instead of "
                        "max(4, ceil(4 L2 / bytes per call)); the line's config says so")
    p.add_argument("--out-proj", type=int, default=0, metavar="HA",
                   help="the workload with an attention output projection of width HA in "
                        "front (moe_tail_run_attn); the line's config says so (no e2e leg)")
    p.add_argument("--shared-gate", action="store_true",
                   help="the workload with the shared expert's sigmoid gate; the line's config "
                        "says so")
    p.add_argument("--timeline", action="store_true",
                   help="also record the per-call milestone timeline (MOE_TAIL_DEBUG_TIMELINE "
                        "on a separate handle, 20 calls after the timed region; medians in "
                        "microseconds after the norm launch's start)")
    p.add_argument("--mma-sync", action="store_true",
                   help="the expert stages on the CUDA-core dequantisation + mma.sync "
                        "streaming kernels (MOE_TAIL_DEBUG_MMA_SYNC) instead of the default "
                        "tcgen05 kernels; the line's config says so")
    p.add_argument("--persistent", action="store_true",
                   help="the workload in the single persistent launch (MOE_TAIL_MODE_PERSISTENT); "
                        "the line's config says so")
    p.add_argument("--attnres-mix", type=int, default=0, metavar="ROWS",
                   help="the second workload instead: the AttnRes residual mix over a "
                        "187-call decoder sequence on ROWS rows (H 7168), one CUDA graph "
                        "replay per step")
    p.add_argument("--mix-family", default="unit", choices=["unit", "scaled"])
    p.add_argument("--no-pdl", action="store_true",
                   help="with --attnres-mix: plain launches instead of programmatic "
                        "dependent ones")
    p.add_argument("--no-extras", action="store_true",
                   help="the default line without its 'also_measured' entries (the AttnRes "
                        "mix at 8 rows and the workload with the attention out_proj in front)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def max_over_ranks(value: float) -> float:
    """Max of a per-rank number over all ranks (identity without a process group).  The
    tensor lives on the GPU under NCCL and on the CPU under gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_call(max_elapsed_ms: float, steps: int, world: int) -> float:
    """Whole-job microseconds per call: every rank ran `steps` calls in at most
    max_elapsed_ms, so the job processed steps*world calls in that time."""
    return max_elapsed_ms * 1000.0 / (steps * world)


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stage_bytes(shape, D, R):
    """Algorithmic bytes of the gate/up and down launches (weights once + activations)."""
    H, I, Is = shape.H, shape.I, shape.Is
    gu = D * 2 * I * (H // 2 + H // 32) + 2 * Is * H * 2 + R * H * 2 * 2
    dn = D * H * (I // 2 + I // 32) + H * Is * 2 + D * I * 2
    return gu, dn


def ncu_traffic(kernel_tag, src_hash, algorithmic_bytes):
    """Per-launch DRAM bytes of a kernel, from the committed ncu summary if it was taken on
    the current source (else None).  The capture runs a smaller case of the same kernel; its
    measured DRAM bytes over its algorithmic bytes (traffic grows with the weight bytes
    streamed) scale this launch's algorithmic bytes."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(kernel_tag)
    if not rec or rec.get("source_hash") != src_hash:
        return None
    return int(rec["dram_over_algorithmic"] * algorithmic_bytes)


# --------------------------------------------------------------------- our arm ----

L2_BYTES = 126 * 1024 * 1024  # GB300 L2 as the driver reports it (cudaDevAttrL2CacheSize)
PROTOCOL_TRIALS, PROTOCOL_REPLAYS, PROTOCOL_ROUNDS = 7, 50, 2
MAX_COPIES = 1024


def weight_copies(bytes_per_call: float) -> int:
    """Layers (weight copies) a timed sequence rotates over: max(4, ceil(4 L2 / B)), so that
    the weights streamed between two calls on the same copy exceed the L2 four times."""
    return int(min(MAX_COPIES, max(4, -(-4 * L2_BYTES // max(1, int(bytes_per_call))))))


def run_ours(args, rank, world, local_rank):
    import torch
    import moe_layer_tail_gb300 as mt

    torch.cuda.set_device(local_rank)
    wl = gen.WORKLOADS[args.workload]
    shape = wl.shape
    if args.experts:
        shape = dataclasses.replace(shape, E=args.experts)
    if args.out_proj:
        shape = dataclasses.replace(shape, Ha=args.out_proj)
    R = shape.R
    K, W = args.steps, args.warmup
    nsets = K + W
    host_w = gen.make_weights(shape, wl.seed)
    if args.shared_gate:
        host_w["ws_gate"] = gen.make_weight(shape, wl.seed, "ws_gate")
    if args.out_proj:
        host_w["w_o"] = gen.make_weight(shape, wl.seed, "w_o")
    # L copies of the layer's weights (same bits, separate device memory), one handle each:
    # consecutive calls run on different copies, like consecutive decoder layers, so no
    # call finds its weights in L2 from the call before
    est = gen.algorithmic_bytes(shape, min(shape.E, R * shape.k), gated=args.shared_gate,
                                out_proj=bool(args.out_proj))
    L = args.weight_copies if args.weight_copies > 0 else weight_copies(est)
    dev_w = [mt.weights_to_device(host_w)]
    for _ in range(L - 1):
        dev_w.append({k: v.clone() for k, v in dev_w[0].items()})
    # one input set per step: correlated rows (~40% repeated picks), seeds wl.seed + 1000*i
    xs, rs = [], []
    c = gen.similar_c() if wl.kind == "similar" else None
    for i in range(nsets):
        a = gen.make_activations(shape, wl.seed + 1000 * i, wl.kind, c)
        xs.append(gen.make_attention_output(shape, wl.seed + 1000 * i) if args.out_proj
                  else a["x"])
        rs.append(a["residual"])
    x_all = mt.acts_to_device(np.stack(xs))  # the attention outputs with --out-proj
    res0 = mt.acts_to_device(np.stack(rs))
    res = res0.clone()
    out = torch.empty_like(res0)
    mode = mt.MODE_PERSISTENT if args.persistent else mt.MODE_MULTI_KERNEL
    flags = mt.DEBUG_MMA_SYNC if args.mma_sync else 0
    tails = [mt.MoeTail(shape, dw, max_rows=R, mode=mode, debug_flags=flags) for dw in dev_w]
    nst = tails[0].launches_per_run(R) + (1 if args.out_proj else 0)
    stream = torch.cuda.current_stream()

    def call(i, stream=None):
        t = tails[i % L]
        (t.run_attn if args.out_proj else t.run)(x_all[i], res[i], out[i], stream=stream)

    # warm-up
    for i in range(W):
        call(i)
    torch.cuda.synchronize()

    # per-step stage events (recorded by the library around each launch, on our stream)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nst)] for _ in range(K)]
    # torch creates events lazily: record once so each handle exists
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    ev_handles = [[e.cuda_event for e in row] for row in evs]

    # timed region: K calls (step i on input set W + i and weight copy (W + i) mod L),
    # nothing else on the stream
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        call(W + i, stream=stream)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1))

    # the measurement protocol: a CUDA graph of L calls (one per weight copy, input sets
    # 0..L-1), timed per replay with events on its stream; the residuals the calls update are
    # restored before each replay, outside the events; 7 trials x 50 replays, two rounds
    # (graph over the copies in order, then in reverse order, alternating)
    proto = None
    if not args.persistent and not args.no_protocol:
        Lg = min(L, nsets)
        graphs = []
        cap = torch.cuda.Stream()
        for order in (list(range(Lg)), list(range(Lg))[::-1]):
            res.copy_(res0)
            torch.cuda.synchronize()
            cap.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                for j in order:
                    t = tails[j]
                    (t.run_attn if args.out_proj else t.run)(x_all[j], res[j], out[j],
                                                             stream=cap)
            graphs.append(g)
        pristine = res0[:Lg].clone()
        per_call = []
        pe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(PROTOCOL_REPLAYS)]
        for rnd in range(PROTOCOL_ROUNDS):
            for trial in range(PROTOCOL_TRIALS):
                g = graphs[(rnd * PROTOCOL_TRIALS + trial) % 2]
                for rep in range(PROTOCOL_REPLAYS):
                    res[:Lg].copy_(pristine)
                    pe[rep][0].record(stream)
                    g.replay()
                    pe[rep][1].record(stream)
                torch.cuda.synchronize()
                ms = sum(a.elapsed_time(b) for a, b in pe)
                per_call.append(ms * 1000.0 / (PROTOCOL_REPLAYS * Lg))
        res.copy_(res0)
        torch.cuda.synchronize()
        del graphs
        proto = {"median_us_per_call": round(statistics.median(per_call), 3),
                 "min_us": round(min(per_call), 3), "max_us": round(max(per_call), 3),
                 "trials": len(per_call), "replays_per_trial": PROTOCOL_REPLAYS,
                 "calls_per_replay": Lg,
                 "how": "CUDA graph of %d calls on %d weight copies, events around each "
                        "replay; residuals restored between replays outside the events; "
                        "median of %d trials x %d replays in %d rounds, the graph's call "
                        "order alternating between trials" % (Lg, Lg, PROTOCOL_TRIALS,
                                                               PROTOCOL_REPLAYS,
                                                               PROTOCOL_ROUNDS)}
    clk = clocks.stop()

    # stage-timed pass: the same K calls again (residuals restored), with the library
    # recording an event pair around each launch on the launching stream
    res.copy_(res0)
    torch.cuda.synchronize()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for i in range(K):
        t = tails[(W + i) % L]
        t.set_stage_events(ev_handles[i])
        call(W + i, stream=stream)
        t.set_stage_events(None)
    s1.record(stream)
    torch.cuda.synchronize()
    staged_ms = s0.elapsed_time(s1)
    status = max(t.status() for t in tails)

    stage_ms = np.array([[row[2 * s].elapsed_time(row[2 * s + 1]) for s in range(nst)]
                         for row in evs])  # [K, stages]

    # distinct experts of every timed set (replayed untimed from pristine residuals)
    Ds = []
    res.copy_(res0)
    for i in range(K):
        call(W + i)
        _, _, nd = tails[(W + i) % L].routing(R)
        Ds.append(nd)
    Ds = np.array(Ds)
    res.copy_(res0)
    bytes_per = np.array([gen.algorithmic_bytes(shape, int(d), gated=args.shared_gate,
                                                 out_proj=bool(args.out_proj)) for d in Ds])
    total_bytes = float(bytes_per.sum())
    us_per_call = job_us_per_call(elapsed_ms, K, world)
    gbps = total_bytes * world / (elapsed_ms * 1e-3) / 1e9

    # dominant kernel: the stage with the largest total time
    names = (["out_proj"] if args.out_proj else []) + ["add_rmsnorm", "router_topk",
                                                       "stream_gate_up", "stream_down", "combine"]
    if args.persistent:
        names = ["tail_persistent"]
    if nst != len(names):
        names = ["stage%d" % s for s in range(nst)]
    tot = stage_ms.sum(axis=0)
    dom = int(np.argmax(tot))
    gu_b, dn_b = zip(*[stage_bytes(shape, int(d), R) for d in Ds])
    dom_bytes = {"stream_gate_up": np.mean(gu_b), "stream_down": np.mean(dn_b),
                 "tail_persistent": float(bytes_per.mean())}.get(names[dom])
    peak, peak_kind = peaks()
    roof = None
    if dom_bytes is not None:
        dur_s = tot[dom] / K * 1e-3
        achieved = dom_bytes / dur_s / 1e9
        if args.mma_sync:
            src = source_hash(["moe_layer_tail_gb300/csrc/k_stream.cu",
                               "moe_layer_tail_gb300/csrc/k_stream_common.cuh",
                               "moe_layer_tail_gb300/csrc/moe_tail_internal.cuh"])
            tag = names[dom] + "_mma_sync"
        else:
            src = source_hash(["moe_layer_tail_gb300/csrc/k_stream_tc.cu",
                               "moe_layer_tail_gb300/csrc/k_stream_common.cuh",
                               "moe_layer_tail_gb300/csrc/moe_tail_internal.cuh"])
            tag = names[dom]
        tr = ncu_traffic(tag, src, dom_bytes) if not args.persistent else None
        roof = {"bound": "hbm", "kernel": names[dom], "achieved": round(achieved, 1),
                "measured": "CUDA events around each launch on its stream, second pass of the "
                            "same %d calls (events serialise the launches: %.1f us/call)"
                            % (K, staged_ms * 1000 / K),
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": tr,
                "algorithmic_bytes_per_launch": int(dom_bytes),
                "launch_us": round(tot[dom] / K * 1000, 2)}

    result = {
        "metric": METRIC, "value": round(us_per_call, 3), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(elapsed_ms / K, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "mxfp4xbf16->f32", "data": "synthetic",
        "config": {"workload": wl.name + ("" if not args.experts else " with %d experts" % shape.E)
                               + (" with shared-expert gate" if args.shared_gate else "")
                               + (" with out_proj from %d" % shape.Ha if args.out_proj else "")
                               + (" in one persistent launch" if args.persistent else "")
                               + (" on the mma.sync expert kernels" if args.mma_sync else ""),
                   "rows": R, "hidden": shape.H, "experts": shape.E,
                   "top_k": shape.k, "expert_inter": shape.I, "shared_inter": shape.Is,
                   "weights": "MXFP4 routed experts, bf16 router and shared expert",
                   "arithmetic": ("MXFP4 weights x bf16 activations (fed to mma.sync as f16 "
                                  "with power-of-two scales), fp32 accumulation"
                                  if args.mma_sync or args.persistent else
                                  "MXFP4 weights x bf16 activations as four E2M1 planes "
                                  "(tcgen05 block-scaled MMAs), bf16 shared expert (tcgen05 "
                                  "bf16 MMAs), fp32 accumulation in tensor memory"),
                   "distinct_experts_mean": round(float(Ds.mean()), 2),
                   "repeat_fraction_mean": round(float(1 - Ds.mean() / (R * shape.k)), 3),
                   "bytes_per_call_mean": int(bytes_per.mean()),
                   "input_sets": nsets,
                   "weight_copies": L,
                   "l2": "no flush: consecutive calls rotate over %d copies of the weights "
                         "(one handle each), each call streaming ~%.0f MB of its own copy's "
                         "weights, larger than the 126 MB L2" % (L, bytes_per.mean() / 1e6),
                   "parallelism": "replicas" if world > 1 else "single"},
        "gbps": round(gbps, 1),
        "hbm_frac_of_%s_peak" % peak_kind: round(gbps / peak, 4),
        "stages_us": {n: round(float(tot[i] / K * 1000), 2) for i, n in enumerate(names)},
        "roofline": roof,
        "protocol": proto,
        "clocks": clk,
        "gpu_launches": int(K * nst),
        "device_status": status,
    }

    # end to end through the C ABI with host buffers (host-device traffic inside the timed
    # region): per step one pinned host block [x; residual; out], read and written in place
    if not args.no_e2e and not args.out_proj:
        ke = min(K, 200)
        blocks = []
        for i in range(ke):
            hb = torch.empty((3, R, shape.H), dtype=torch.bfloat16).pin_memory()
            hb[0].copy_(torch.from_numpy(xs[W + i].view(np.int16)).view(torch.bfloat16))
            hb[1].copy_(torch.from_numpy(rs[W + i].view(np.int16)).view(torch.bfloat16))
            blocks.append(hb)
        # the C ABI called with prebuilt arguments (no Python tensor work inside the loop)
        import ctypes
        lib = mt.load_library()
        st_e2e = torch.cuda.Stream()
        sh = ctypes.c_void_p(st_e2e.cuda_stream)
        act = R * shape.H * 2
        calls = [(tails[(W + i) % L].handle, ctypes.c_void_p(hb.data_ptr()),
                  ctypes.c_void_p(hb.data_ptr() + act), ctypes.c_void_p(hb.data_ptr() + 2 * act),
                  R, sh) for i, hb in enumerate(blocks)]
        warm = blocks[0].clone().pin_memory()
        for t in tails:  # one untimed call per handle
            t.run_host(warm[0], warm[1], warm[2], stream=st_e2e)
        torch.cuda.synchronize()
        fn = lib.moe_tail_run_host
        ts = time.perf_counter()
        for a in calls:
            if fn(*a) != 0:
                raise RuntimeError("moe_tail_run_host failed")
        te = time.perf_counter()
        e2e_us = (te - ts) * 1e6 / ke
        result["e2e"] = {"value": round(e2e_us / world, 3), "unit": UNIT,
                         "h2d_bytes_per_step": 2 * R * shape.H * 2,
                         "d2h_bytes_per_step": 2 * R * shape.H * 2, "steps": ke,
                         "api": "moe_tail_run_host on one pinned host block [x; residual; out] "
                                "per step on a non-default stream: the call's kernels read x and "
                                "residual from, and write out and residual to, the page-locked "
                                "block in place (mapped host memory over NVLink-C2C)"}

    if args.timeline:
        tt = mt.MoeTail(shape, dev_w[0], max_rows=R, mode=mode,
                        debug_flags=flags | mt.DEBUG_TIMELINE)
        marks = []
        for i in range(min(20, nsets)):
            (tt.run_attn if args.out_proj else tt.run)(x_all[i], res[i], out[i])
            marks.append(tt.timeline())
        res.copy_(res0)
        tt.close()
        result["timeline_us"] = {
            n: (round(float(np.median([m[n] for m in marks])), 2)
                if all(m[n] is not None for m in marks) else None)
            for n in mt.TL_NAMES}
        result["timeline_us"]["how"] = ("%%globaltimer stamps of each launch's milestones, one "
                                        "call at a time on a separate handle (its per-call "
                                        "reset serialises the calls), median of %d calls"
                                        % len(marks))

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(shape, host_w, xs[W], rs[W],
                                              attn=bool(args.out_proj))
    for t in tails:
        t.close()
    return result


# The pages' own per-call figures for their split mix over a 187-call decoder sequence in a
# CUDA graph, by row count (RTX PRO 6000; another machine and kernel: context only).
PAGE_MIX_US = {1: 3.38, 8: 3.44, 16: 3.66}


def run_mix(args, rank, world, local_rank):
    """The AttnRes mix: one step = one replay of a CUDA graph holding the 187-call decoder
    sequence (a block committed every 24 calls, 2 to 9 sources per call) on ROWS rows of
    H 7168; us per call = replay time / 187.  The sequence's state (prefix, blocks) is
    restored and L2 flushed (a 256 MB write) between replays, outside the timed events."""
    import torch
    import moe_layer_tail_gb300 as mt

    torch.cuda.set_device(local_rank)
    seq = gen.MixSequence(R=args.attnres_mix)
    L, R, H = seq.L, seq.R, seq.H
    K, W = args.steps, args.warmup
    host = gen.make_mix_sequence(seq, 2026, args.mix_family)
    dd = {k: mt.acts_to_device(v) for k, v in host.items()}
    pre0, blk0 = dd["prefix"].clone(), dd["blocks"].clone()
    mix = torch.empty((L, R, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(mix)
    flags = 0 if args.no_pdl else mt.ATTNRES_MIX_PDL
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def sequence(stream=None):
        for l in range(L):
            mt.attnres_mix(dd["sub"][l], dd["prefix"], dd["blocks"], seq.n_blocks(l),
                           seq.commit(l), dd["q"][l], dd["gamma"][l], mix[l], y[l], eps=seq.eps,
                           flags=flags, stream=stream)

    def reset():
        dd["prefix"].copy_(pre0)
        dd["blocks"].copy_(blk0)
        flush.zero_()

    sequence()  # eager once (loads the kernel)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    reset()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=cap):
        sequence()
    stream = torch.cuda.current_stream()
    for _ in range(W):
        reset()
        g.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    for i in range(K):
        reset()
        evs[i][0].record(stream)
        g.replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    replay_ms = [a.elapsed_time(b) for a, b in evs]
    elapsed_ms = max_over_ranks(float(np.sum(replay_ms)))
    us_per_call = elapsed_ms * 1e3 / (K * L) / world
    bytes_seq = sum(gen.mix_call_bytes(R, H, seq.n_blocks(l), seq.commit(l)) for l in range(L))
    peak, peak_kind = peaks()
    achieved = bytes_seq / L / (us_per_call * world * 1e-6) / 1e9
    result = {
        "metric": METRIC, "value": round(us_per_call, 3), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(elapsed_ms / K, 5),
        "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16->f32", "data": "synthetic",
        "config": {"workload": "attnres_mix_h7168_187calls_r%d" % R, "rows": R, "hidden": H,
                   "calls_per_step": L, "block_calls": seq.block_calls,
                   "sources_per_call": "%d..%d" % (seq.n_blocks(0) + 1,
                                                   seq.n_blocks(L - 1) + 1),
                   "family": args.mix_family,
                   "ctas_per_row": mt.attnres_mix_ctas_per_row(H, seq.n_blocks(L - 1)),
                   "launch": "CUDA graph, " + ("plain launches" if args.no_pdl else
                                               "programmatic dependent launches"),
                   "l2": "flushed (256 MB write) between replays, outside the timed events",
                   "context": "the pages quote %s us per call at %d rows for their split mix "
                              "on an RTX PRO 6000 (another machine and another kernel: "
                              "context, not a baseline)" % (PAGE_MIX_US.get(R, "no figure"), R),
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "kernel": "attnres_mix", "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "algorithmic_bytes_per_launch": int(bytes_seq / L),
                     "measured": "CUDA events around each graph replay on its stream",
                     "note": "latency-bound: ~%.0f KB per call" % (bytes_seq / L / 1e3)},
        "clocks": clk,
        "gpu_launches": int(K * L),
    }
    # end to end: per call, the sublayer output from pinned host memory, the call, y back
    if not args.no_e2e:
        hs = torch.from_numpy(host["sub"].view(np.int16)).view(torch.bfloat16).pin_memory()
        hy = torch.empty((L, R, H), dtype=torch.bfloat16).pin_memory()
        dsub = torch.empty((R, H), dtype=torch.bfloat16, device="cuda")
        reset()
        torch.cuda.synchronize()
        ts = time.perf_counter()
        for l in range(L):
            dsub.copy_(hs[l], non_blocking=True)
            mt.attnres_mix(dsub, dd["prefix"], dd["blocks"], seq.n_blocks(l), seq.commit(l),
                           dd["q"][l], dd["gamma"][l], mix[l], y[l], eps=seq.eps, flags=flags)
            hy[l].copy_(y[l], non_blocking=True)
        torch.cuda.synchronize()
        te = time.perf_counter()
        result["e2e"] = {"value": round((te - ts) * 1e6 / L / world, 3), "unit": UNIT,
                         "h2d_bytes_per_step": L * R * H * 2, "d2h_bytes_per_step": L * R * H * 2,
                         "steps": 1,
                         "api": "moe_attnres_mix, eager, per call the sublayer output copied "
                                "in from pinned host memory and y copied back"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = mix_cpu_baseline(seq, host)
    return result


def mix_cpu_baseline(seq, host, budget_s=20.0):
    """The oracle's mix, as it stands (one host thread), over the decoder sequence until the
    budget is used; us per call."""
    import oracle
    per_call = []
    t_start = time.perf_counter()
    pre, blk = host["prefix"], host["blocks"]
    for l in range(seq.L):
        t = time.perf_counter()
        m = oracle.attnres_mix(host["sub"][l], pre, blk, seq.n_blocks(l), seq.commit(l),
                               host["q"][l], host["gamma"][l], seq.eps)
        per_call.append(time.perf_counter() - t)
        pre, blk = m["prefix"], m["blocks"]
        if time.perf_counter() - t_start > budget_s:
            break
    us = float(np.mean(per_call)) * 1e6
    return {"value": round(us, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "the first %d calls of the same sequence, mean" % len(per_call)}


def cpu_baseline(shape, host_w, x, r, budget_s=20.0, attn=False):
    """The oracle, as it stands, on the host cores: whole calls of the workload until the
    budget is used (at least one).  attn: x is the attention output to project first."""
    import oracle
    cores = oracle.host_cores()
    d = dict(host_w)
    d["attn" if attn else "x"] = x
    d["residual"] = r
    times = []
    t_start = time.perf_counter()
    while not times or (time.perf_counter() - t_start < budget_s and len(times) < 5):
        t = time.perf_counter()
        oracle.moe_tail(d, shape.k, shape.eps, nthreads=cores)
        times.append(time.perf_counter() - t)
    us = statistics.median(times) * 1e6
    return {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d whole call(s) of the same workload (8 rows), median" % len(times)}


# --------------------------------------------------------------- reference arm ----

def run_reference(args, rank, world):
    """The oracle on the host cores, each step one row of the workload through the whole
    tail (routing, its k experts, shared expert, combine); microseconds per call = per-row
    time x rows."""
    import oracle
    wl = gen.WORKLOADS[args.workload]
    shape = wl.shape
    if args.experts:
        shape = dataclasses.replace(shape, E=args.experts)
    R = shape.R
    cores = oracle.host_cores()
    host_w = gen.make_weights(shape, wl.seed)
    if args.shared_gate:
        host_w["ws_gate"] = gen.make_weight(shape, wl.seed, "ws_gate")
    c = gen.similar_c() if wl.kind == "similar" else None
    K, W = args.steps, args.warmup
    a = gen.make_activations(shape, wl.seed, wl.kind, c)
    samples = []
    for i in range(W + K):
        rr = i % R
        d = dict(host_w)
        d["x"] = a["x"][rr:rr + 1]
        d["residual"] = a["residual"][rr:rr + 1]
        t = time.perf_counter()
        oracle.moe_tail(d, shape.k, shape.eps, nthreads=cores)
        if i >= W:
            samples.append(time.perf_counter() - t)
    step_s = float(np.mean(samples))
    us_per_call = step_s * R * 1e6
    return {"impl": "reference", "metric": METRIC, "value": round(us_per_call, 1), "unit": UNIT,
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(step_s * 1e3, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "rows": R, "hidden": shape.H, "experts": shape.E,
                       "top_k": shape.k, "expert_inter": shape.I, "shared_inter": shape.Is},
            "cpu_baseline": {"value": round(us_per_call, 1), "unit": UNIT, "cores": cores,
                             "kind": "oracle",
                             "sample": "each step: one row of the workload through the whole "
                                       "tail; us per call = mean row time x %d rows" % R},
            "e2e": {"value": round(us_per_call, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_reference_mix(args, world):
    """The oracle's mix on the host (one thread), each step one call of the decoder
    sequence, in sequence order."""
    seq = gen.MixSequence(R=args.attnres_mix)
    host = gen.make_mix_sequence(seq, 2026, args.mix_family)
    import oracle
    K, W = args.steps, args.warmup
    pre, blk = host["prefix"], host["blocks"]
    samples = []
    for i in range(W + K):
        l = i % seq.L
        if l == 0:
            pre, blk = host["prefix"], host["blocks"]
        t = time.perf_counter()
        m = oracle.attnres_mix(host["sub"][l], pre, blk, seq.n_blocks(l), seq.commit(l),
                               host["q"][l], host["gamma"][l], seq.eps)
        if i >= W:
            samples.append(time.perf_counter() - t)
        pre, blk = m["prefix"], m["blocks"]
    us = float(np.mean(samples)) * 1e6
    return {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT,
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(us / 1e3, 4),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "attnres_mix_h7168_187calls_r%d" % seq.R, "rows": seq.R,
                       "hidden": seq.H, "calls_per_step": 1, "family": args.mix_family},
            "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "each step one call of the decoder sequence"},
            "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def extras(args):
    """Two more workloads of the same build, measured in the same run and reported beside the
    headline line (not part of its value): the AttnRes mix at 8 rows (one step = one graph
    replay of the 187-call sequence) and the headline workload with the attention output
    projection (Ha 16384) in front of the tail, 100 calls."""
    import copy
    out = {}
    a = copy.copy(args)
    a.attnres_mix, a.steps, a.warmup, a.no_cpu_baseline = 8, 50, 5, True
    m = run_mix(a, 0, 1, 0)
    out["attnres_mix_8_rows"] = {
        "metric": m["metric"], "value": m["value"], "unit": m["unit"], "steps": a.steps,
        "roofline_frac": (m.get("roofline") or {}).get("frac"),
        "e2e_value": (m.get("e2e") or {}).get("value"), "clocks": m.get("clocks"),
        "config": m.get("config")}
    b = copy.copy(args)
    b.out_proj, b.steps, b.warmup = 16384, 100, 5
    b.no_cpu_baseline, b.no_e2e, b.no_protocol, b.timeline = True, True, True, False
    o = run_ours(b, 0, 1, 0)
    out["out_proj_16384_in_front"] = {
        "metric": o["metric"], "value": o["value"], "unit": o["unit"], "steps": b.steps,
        "stages_us": o.get("stages_us"), "roofline": o.get("roofline"),
        "clocks": o.get("clocks")}
    return out


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        res = run_reference_mix(args, world) if args.attnres_mix else run_reference(args, rank,
                                                                                     world)
        print(json.dumps(res), flush=True)
        return 0
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = (run_mix if args.attnres_mix else run_ours)(args, rank, world, local_rank)
    if (rank == 0 and world == 1 and not args.no_extras and not args.attnres_mix
            and not args.out_proj and not args.persistent and not args.mma_sync
            and not args.experts and args.workload == gen.BENCH_WORKLOAD):
        res["also_measured"] = extras(args)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
