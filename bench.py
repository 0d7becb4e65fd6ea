#!/usr/bin/env python3
"""Benchmark: one MoE decode layer shaped like Mixtral-8x7B (d=4096, f=14336, 8 experts,
top-2, one decode token), INT2 up projection, fp16 gate/down, sparse SwiGLU experts.

A step is one pass of the whole hot path on one token: router GEMV + softmax top-k,
the two selected sparse experts (INT2 up-GEMV, threshold mask, gathered gate and
down rows), the weighted combination and the RMSNorm that hands the hidden state to
the next layer.  Steps replay a CUDA graph of `moe_layer_decode` over 8 distinct
layer copies back to back (different weights and tokens), the way a stack of layers
runs, so every step streams its weights from HBM (the 8 copies hold 16 GB; a copy is
reused only after 7 others).  The same steps with one graph launch per layer are
reported beside it.

Prints one JSON line.  `--impl reference` times the CPU oracle on the same
workload instead (its own line, impl = "reference").
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

WORKLOAD = dict(name="mixtral-8x7b-moe-layer-decode", d=4096, f=14336, E=8, k=2, B=1,
                calib_tokens=1024)
SPARSITIES = (0, 50, 70, 90)
INF_PCT = 101  # --sparsity 101: t = +inf (nothing kept: only the up projection's bytes)

# Further layer shapes, timed with --workload (one JSON line per point; the default run
# above is the headline).  Shared experts have the routed experts' d and f.
WORKLOADS = {
    "mixtral-8x7b-batch": dict(d=4096, f=14336, E=8, k=2, shared=0, tokens=(1, 2, 4, 8, 16, 32),
                               sparsities=(70,), calib_tokens=1024, copies=8, chained=False),
    "deepseek-v2-lite": dict(d=2048, f=1408, E=64, k=6, shared=2, tokens=(1, 2, 4, 8, 16, 32, 64),
                             sparsities=(0, 50, 90), calib_tokens=1024, copies=8, chained=False),
    "mixtral-8x22b-stack": dict(d=6144, f=16384, E=8, k=2, shared=0, tokens=(1, 8), sparsities=(70,),
                                calib_tokens=256, copies=56, chained=True),
    # FloE's on-the-fly setting: gate/down rows in page-locked host memory, only the kept
    # rows fetched over the host link
    "mixtral-8x7b-host-rows": dict(d=4096, f=14336, E=8, k=2, shared=0, tokens=(1, 2),
                                   sparsities=(0, 50, 70, 90), calib_tokens=1024, copies=2, chained=False,
                                   host_rows=True),
    # MoE-Infinity's expert activation matrix collection and expert cache (host code):
    # per-query time at 1K stored matrices of the Mixtral-8x7B shape (32 MoE layers x 8)
    "eamc-lookup": dict(L=32, E=8, capacity=1000, host_only=True),
}
# the further configurations the default run also times (every sparsity of the workload)
FURTHER_POINTS = (("mixtral-8x7b-batch", (1, 2, 4, 8, 16, 32)),
                  ("deepseek-v2-lite", (1, 2, 8, 64)),
                  ("mixtral-8x22b-stack", (1, 8)))
HEADLINE_PCT = 70
N_LAYER_COPIES = 8
METRIC = "MoE decode layer expert-tokens/s (Mixtral-8x7B-shaped layer, 1 token, 70% sparsity)"

# ncu DRAM bytes per launch of the dominant kernel, keyed by the source file hash it was
# taken on; reported only while the kernel source is unchanged.
NCU_TRAFFIC = {
    # decode_gather_kernel: 147.50 MB (read + write) captured on layer copy 0 at 70% (the
    # 1-copy small case, 143.97 MB algorithmic), scaled to the 8-copy mean of 139.12 MB
    ("decode_gather_kernel", "345fe56b4667b2fa"): 147.50e6 * 139.12 / 143.97,
    # decode_layer_kernel: 180.87 MB read + 3.10 MB written (dram__bytes_read.sum,
    # dram__bytes_write.sum) captured on layer copy 0 at 70% (the 1-copy case, 180.75 MB
    # algorithmic), scaled to the 8-copy mean of 175.90 MB (re-keyed after two unused fields
    # of the control block were renamed; the compiled kernel is unchanged)
    ("decode_layer_kernel", "6652570ccd95b6ef"): (180871936 + 3104768) * 175.90 / 180.75,
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sparsity", type=int, default=HEADLINE_PCT,
                    help="0/50/70/90 (the calibrated points) or 101 for t = +inf")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--copies", type=int, default=N_LAYER_COPIES,
                    help="rotating layer copies (fewer: a small case for profiling; below 8 the "
                         "weights no longer exceed L2 by a wide margin)")
    ap.add_argument("--no-sweep", action="store_true", help="time only the headline sparsity")
    ap.add_argument("--no-further", action="store_true",
                    help="skip the further configurations in the default run's line")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=None,
                    help="time one of the further layer shapes instead of the headline")
    ap.add_argument("--tokens", type=int, default=None, help="with --workload: only this batch size")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if torch.cuda.is_available():
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:  # host-only ranks (the multi-process tests of the rank reductions)
            dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float, device) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(world, value: float, device) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload set-up (synthetic weights, device-side packing, GPU calibration)
# ---------------------------------------------------------------------------

def build_layers(dev, R):
    import sparse_expert_swiglu_gb300 as ses
    from sparse_expert_swiglu_gb300 import synth
    W = WORKLOAD
    layers = []
    for r in range(R):
        de = synth.experts(W["E"], W["d"], W["f"], 100 + r, device=dev, layer=r)
        ex = ses.Experts.from_dense(de.w_up, de.gate_t, de.down,
                                    torch.zeros(W["E"], dtype=torch.float32, device=dev),
                                    interleave=True)
        del de
        wr = synth.router(W["d"], W["E"], 100 + r, device=dev, layer=r)
        layers.append(ses.Layer(wr, ex, W["k"], True))
    torch.cuda.empty_cache()
    return layers


def calibrate(layers, dev):
    """Per-expert thresholds: nearest-rank percentiles of |v| over calibration tokens,
    with v from the library's own up-projection kernel (set-up only)."""
    import sparse_expert_swiglu_gb300 as ses
    from sparse_expert_swiglu_gb300 import synth
    W = WORKLOAD
    xcal = synth.calibration_tokens(W["calib_tokens"], W["d"], 7, device=dev)
    table = {p: [] for p in SPARSITIES}
    for layer in layers:
        ex = layer.routed
        ex.thr.fill_(float("inf"))  # nothing kept: only v is computed
        ws = ses.Workspace(ses.expert_workspace_bytes(W["calib_tokens"], W["d"], W["f"]), dev)
        thr = {p: torch.zeros(W["E"], dtype=torch.float32, device=dev) for p in SPARSITIES}
        for e in range(W["E"]):
            _, dbg = ses.expert_sparse_swiglu(xcal, ex, e, ws=ws, debug=True)
            a = torch.sort(dbg["v"].abs().flatten()).values
            n = a.numel()
            for p in SPARSITIES:
                if p > 0:
                    thr[p][e] = a[(p * n + 99) // 100 - 1]
        for p in SPARSITIES:
            table[p].append(thr[p])
        table.setdefault(INF_PCT, []).append(torch.full((W["E"],), float("inf"), dtype=torch.float32, device=dev))
    return table


def pct_label(pct):
    return "t=+inf" if pct == INF_PCT else f"{pct}%"


def config_dict(pct, R, world):
    """The workload both arms report (identical keys and values)."""
    W = WORKLOAD
    d, f, E = W["d"], W["f"], W["E"]
    copy_gb = E * (4 * d * f + d * f * 5 / 16) / 1e9  # gate + down fp16, packed INT2 up
    return {"workload": W["name"], "d": d, "f": f, "experts": E, "top_k": W["k"],
            "tokens_per_step": W["B"], "sparsity_pct": pct, "up_projection": "int2 g64 fp16 scale/zero",
            "gate_down": "fp16", "rmsnorm": True, "parallelism": f"replicas x{world}",
            "calibration_tokens": W["calib_tokens"],
            "l2": f"inputs larger than L2: {R} rotating layer copies ({R * copy_gb:.1f} GB), "
                  f"each reused only after {R - 1} others",
            "graphs": f"the {R} layer copies back to back in one CUDA graph, as a stack of "
                      "layers runs (PDL between all kernels); each copy keeps its own token"}


def set_thresholds(layers, table, pct):
    for r, layer in enumerate(layers):
        layer.routed.thr.copy_(table[pct][r])


def count_bytes(idx, words, d, f, E, k, B, up_bytes):
    """Bytes one layer step must move, from its routing (idx [B][k]) and its masks (words
    [B][k][ceil(f / 32)] uint32, bit c of word c / 32 = column c kept): per active expert
    the packed up projection plus 4 d bytes per column kept for any of its tokens (gate row
    + down row, read once), the router weight (2 d E), x in and y out (2 B d each).  Also
    per kernel."""
    words = np.asarray(words, dtype=np.uint32)
    bits = ((words[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(B, k, -1)[..., :f]
    experts = sorted(set(np.asarray(idx).ravel().tolist()))
    kept_cols, up_total = 0, 0
    for e in experts:
        rws, cls = np.nonzero(np.asarray(idx) == e)
        union = np.any(bits[rws, cls].astype(bool), axis=0)
        kept_cols += int(union.sum())
        up_total += up_bytes
    gather = 4 * d * kept_cols
    return dict(up=up_total + 2 * B * d, gather=gather, route=2 * d * E + 2 * B * d,
                total=up_total + gather + 2 * d * E + 2 * B * d * 2,
                kept_frac=kept_cols / (f * len(experts)), pairs=B * k)


def algorithmic_bytes(layers, xs, ws_list):
    """count_bytes of every layer copy at the current thresholds, from the masks the
    layer itself returns."""
    import sparse_expert_swiglu_gb300 as ses
    W = WORKLOAD
    d, f, E, k, B = W["d"], W["f"], W["E"], W["k"], W["B"]
    up_bytes = ses.packed_bytes(d, f)
    rows = []
    for layer, x, ws in zip(layers, xs, ws_list):
        _, dbg = ses.layer_decode(x, layer, rmsnorm=True, ws=ws, debug=True)
        rows.append(count_bytes(dbg["topk_idx"].cpu().numpy(), dbg["mask"].cpu().numpy(), d, f, E, k, B, up_bytes))
    return rows


def capture_graphs(layers, xs, ys, ws_list, events_list=None):
    import sparse_expert_swiglu_gb300 as ses
    graphs = []
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for r, layer in enumerate(layers):  # warm-up outside capture
            ses.layer_decode(xs[r], layer, rmsnorm=True, ws=ws_list[r], out=ys[r])
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    for r, layer in enumerate(layers):
        g = torch.cuda.CUDAGraph()
        c_layer = layer.c_struct()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            ev = events_list[r] if events_list is not None else None
            ses.layer_decode(xs[r], layer, rmsnorm=True, ws=ws_list[r], out=ys[r], c_layer=c_layer,
                             events=ev)
        graphs.append(g)
    torch.cuda.synchronize()
    return graphs, stream


def capture_stack(layers, xs, ys, ws_list, stream):
    """One CUDA graph of every layer copy back to back on one stream, as a stack of
    layers runs: each layer's first kernel waits for the previous layer's last kernel
    (programmatic dependent launch), the inputs stay the copies' own tokens."""
    import sparse_expert_swiglu_gb300 as ses
    g = torch.cuda.CUDAGraph()
    c_layers = [layer.c_struct() for layer in layers]
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for r, layer in enumerate(layers):
            ses.layer_decode(xs[r], layer, rmsnorm=True, ws=ws_list[r], out=ys[r], c_layer=c_layers[r])
    torch.cuda.synchronize()
    return g


def capture_stack_e2e(layers, x_all, y_all, ws_list, stream, x_pin, y_pin):
    """The stacked graph with the steps' host copies inside it: the R tokens come in
    from pinned host memory in one copy before the first layer and the R results go
    out to pinned host memory in one copy after the last (x_all, y_all hold them as
    rows).  Reading a result back between layers would end the programmatic launch
    overlap of the next layer, which costs more than the copies."""
    import sparse_expert_swiglu_gb300 as ses
    g = torch.cuda.CUDAGraph()
    c_layers = [layer.c_struct() for layer in layers]
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        x_all.copy_(x_pin, non_blocking=True)
        for r, layer in enumerate(layers):
            ses.layer_decode(x_all[r], layer, rmsnorm=True, ws=ws_list[r], out=y_all[r], c_layer=c_layers[r])
        y_pin.copy_(y_all, non_blocking=True)
    torch.cuda.synchronize()
    return g


def capture_stack_prefetch(layers, xs, ys, ws_list, stream, pred):
    """The stacked graph with the inter-expert prefetch hook: while layer copy r runs, a
    second stream prefetches into L2 the packed up projections of the experts predicted
    for copy r + 1 (the next replay's copy 0 after the last).  The side branch waits
    only for layer r - 1, so the layers' dependent launches are unchanged; it rejoins
    at the end of the graph."""
    import sparse_expert_swiglu_gb300 as ses
    R = len(layers)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    c_layers = [layer.c_struct() for layer in layers]
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for r, layer in enumerate(layers):
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                ses.prefetch_experts(layers[(r + 1) % R].routed, pred[(r + 1) % R])
            ses.layer_decode(xs[r], layer, rmsnorm=True, ws=ws_list[r], out=ys[r], c_layer=c_layers[r])
        stream.wait_stream(side)
    torch.cuda.synchronize()
    return g


def time_stack(stack, stream, R, steps, warmup):
    """Microseconds per layer over whole replays of a stacked graph."""
    reps = max(1, steps // R)
    with torch.cuda.stream(stream):
        for _ in range(max(1, warmup // R)):
            stack.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            stack.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * R)


def prefetch_hook_times(layers, xs, ys, ws_list, stream, steps, warmup):
    """Layer time in the stacked graph without the prefetch hook, with it on an exact
    prediction (each copy's own router on its own token: the copies are not chained, so
    this is the best a predictor can do) and with it on a prediction that misses every
    routed expert."""
    import sparse_expert_swiglu_gb300 as ses
    W = WORKLOAD
    R, E, k = len(layers), W["E"], W["k"]
    exact = [ses.route_topk(xs[r], layers[r].w_router, k)[0].reshape(-1).contiguous() for r in range(R)]
    miss = []
    for r in range(R):
        chosen = set(exact[r].tolist())
        miss.append(torch.tensor([e for e in range(E) if e not in chosen][:k], dtype=torch.int32,
                                 device=xs[r].device))
    plain = capture_stack(layers, xs, ys, ws_list, stream)
    with_exact = capture_stack_prefetch(layers, xs, ys, ws_list, stream, exact)
    with_miss = capture_stack_prefetch(layers, xs, ys, ws_list, stream, miss)
    out = {}
    for name, g in (("without", plain), ("exact_prediction", with_exact), ("missed_prediction", with_miss)):
        out[f"layer_us_{name}"] = time_stack(g, stream, R, steps, warmup)
    out["prefetch_bytes_per_layer"] = k * ses.packed_bytes(W["d"], W["f"])
    out["how"] = ("stacked graph of the layer copies; a second stream L2-prefetches the packed up "
                  "projections of the experts predicted for the next copy while a copy runs "
                  "(moe_prefetch_experts); exact = each copy's own router on its own token, "
                  "missed = k experts that copy does not route to")
    return out


def time_steps(graphs, stream, steps, warmup, world, dev, stack=None):
    """Device time of `steps` layer passes: whole replays of the stacked graph (R layers
    each), the remainder from the single-layer graphs."""
    R = len(graphs)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            graphs[i % R].replay()
    torch.cuda.synchronize()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    full = steps // R if stack is not None else 0
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(full):
            stack.replay()
        for i in range(full * R, steps):
            graphs[i % R].replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return start.elapsed_time(end) / 1e3  # seconds


def step_distribution(stack, stream, R, replays):
    """Spread of the step time: an event after every replay of the stacked graph (R layer
    steps each), each replay's time / R, as p10 / median / p90 in microseconds."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(replays + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(replays):
            stack.replay()
            evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per_step = np.array([evs[i].elapsed_time(evs[i + 1]) * 1e3 / R for i in range(replays)])
    return {"p10": float(np.percentile(per_step, 10)), "p50": float(np.median(per_step)),
            "p90": float(np.percentile(per_step, 90)), "replays": replays, "steps_per_replay": R,
            "how": "event after every replay of the stacked graph; replay time / steps per replay"}


def per_kernel_times(prof_graphs, events_list, stream, steps, path):
    """Average device time of each kernel, from events recorded around it inside the
    graphs (replayed R at a time, read back before the events are re-recorded).  On the
    decode path the router runs inside the up kernel and the combination inside the
    gather kernel: events 0 and 1 (and 3 and 4) are back to back, and their interval is
    the cost of an event pair, reported as event_pair_us."""
    R = len(prof_graphs)
    acc = np.zeros(4)
    n = 0
    blocks = max(1, steps // R)
    for _ in range(blocks):
        with torch.cuda.stream(stream):
            for g in prof_graphs:
                g.replay()
        torch.cuda.synchronize()
        for evs in events_list:
            for j in range(4):
                acc[j] += evs[j].elapsed_time(evs[j + 1])
            n += 1
    t = [acc[j] / n * 1e3 for j in range(4)]  # microseconds
    if path == "decode_fused":
        return {"decode_layer_kernel": t[1], "event_pair_us": t[0]}
    if path == "decode":
        return {"decode_up_kernel": t[1], "decode_gather_kernel": t[2], "event_pair_us": t[0]}
    return {"route_kernel": t[0], "up_kernel": t[1], "gather_kernel": t[2], "combine_kernel": t[3]}


def source_hash(kernel="decode_gather_kernel"):
    """Hash of the sources a kernel is built from (the traffic table is keyed by it)."""
    import hashlib
    h = hashlib.sha256()
    files = (["decode.cu", "common.cuh", "params.cuh"] if kernel.startswith("decode_")
             else ["up.cu", "gather.cu", "combine.cu", "route.cu", "common.cuh", "params.cuh"])
    for fn in files:
        with open(os.path.join(ROOT, "sparse_expert_swiglu_gb300", "csrc", fn), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# CPU oracle on the same workload
# ---------------------------------------------------------------------------

def oracle_prepare(dev, n_tokens, pct_table, pct):
    """Layer copy 0 in the oracle's form, for the experts that n_tokens sample tokens use."""
    from oracle import moe_oracle as orc
    from sparse_expert_swiglu_gb300 import synth
    W = WORKLOAD
    d, f, E, k = W["d"], W["f"], W["E"], W["k"]
    wr = synth.router(d, E, 100, device=dev, layer=0).cpu().numpy()
    xs = synth.tokens(n_tokens, d, 555, device=dev).cpu().numpy()
    idx, _, _ = orc.route_topk(xs, wr, k)
    need = sorted(set(idx.ravel().tolist()))
    de = synth.experts(E, d, f, 100, device=dev, layer=0)
    thr = pct_table[pct][0].cpu().numpy()
    experts = [None] * E
    for e in need:
        q, s, z = orc.quantize_int2(de.w_up[e].cpu().numpy())
        experts[e] = dict(w_gate=de.gate_t[e].cpu().numpy().T, w_up_deq=orc.dequantize_int2(q, s, z),
                          w_down=de.down[e].cpu().numpy(), thr=float(thr[e]))
    del de
    torch.cuda.empty_cache()
    return xs, wr, experts


def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def time_oracle(xs, wr, experts, steps, warmup):
    from oracle import moe_oracle as orc
    W = WORKLOAD
    for i in range(warmup):
        orc.moe_layer(xs[i % len(xs):i % len(xs) + 1], wr, experts, W["k"], True, rmsnorm_out=True)
    t0 = time.perf_counter()
    for i in range(steps):
        orc.moe_layer(xs[i % len(xs):i % len(xs) + 1], wr, experts, W["k"], True, rmsnorm_out=True)
    return time.perf_counter() - t0


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args, world, rank, local):
    if rank != 0:
        return
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    W = WORKLOAD
    from oracle import moe_oracle as orc
    from sparse_expert_swiglu_gb300 import synth
    d, f, E, k = W["d"], W["f"], W["E"], W["k"]
    xs_n = 4
    wr = synth.router(d, E, 100, device=dev, layer=0).cpu().numpy()
    # the GPU arm's tokens of its first layer copies (one token each), on layer copy 0
    xs = np.concatenate([synth.tokens(W["B"], d, 1000 + i, device=dev).cpu().numpy() for i in range(xs_n)])
    idx, _, _ = orc.route_topk(xs, wr, k)
    need = sorted(set(idx.ravel().tolist()))
    de = synth.experts(E, d, f, 100, device=dev, layer=0)
    # thresholds as the GPU arm sets them: the nearest-rank percentile of |v| over the same
    # calibration tokens (here with the oracle's own fp64 v)
    xcal = synth.calibration_tokens(W["calib_tokens"], d, 7, device=dev).cpu().numpy()
    experts = [None] * E
    for e in need:
        q, s, z = orc.quantize_int2(de.w_up[e].cpu().numpy())
        wdeq = orc.dequantize_int2(q, s, z)
        t = np.inf if args.sparsity == INF_PCT else orc.quantile_threshold(orc.expert_up(xcal, wdeq), args.sparsity)
        experts[e] = dict(w_gate=de.gate_t[e].cpu().numpy().T, w_up_deq=wdeq,
                          w_down=de.down[e].cpu().numpy(), thr=float(np.float32(t)))
    del de
    # a step is 1/n of a single-token layer decode: the oracle on the token, with both
    # routed experts cut to one of n column slices of their intermediate dimension (the
    # n slices together are the layer's expert work); n is chosen from one full decode so
    # that the --steps run takes about two minutes
    x0 = xs[0:1]
    t0 = time.perf_counter()
    orc.moe_layer(x0, wr, experts, k, True, rmsnorm_out=True)
    t_full = time.perf_counter() - t0
    n = max(1, min(64, math.ceil(args.steps * t_full / 120.0)))
    cuts = np.array_split(np.arange(f), n)
    sliced = [[None if ex is None else dict(w_gate=np.ascontiguousarray(ex["w_gate"][:, c]),
                                            w_up_deq=np.ascontiguousarray(ex["w_up_deq"][:, c]),
                                            w_down=np.ascontiguousarray(ex["w_down"][c, :]), thr=ex["thr"])
               for ex in experts] for c in cuts]
    for i in range(args.warmup):
        orc.moe_layer(xs[i % xs_n:i % xs_n + 1], wr, sliced[i % n], k, True)
    t0 = time.perf_counter()
    for i in range(args.steps):
        orc.moe_layer(xs[i % xs_n:i % xs_n + 1], wr, sliced[i % n], k, True)
    secs = time.perf_counter() - t0
    value = W["B"] * k * args.steps / n / secs
    cores = oracle_threads()
    line = {
        "impl": "reference", "metric": METRIC.replace("70%", pct_label(args.sparsity)), "value": value,
        "unit": "expert-tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(args.sparsity, max(1, args.copies), args.gpus),
        "cpu_baseline": {"value": value, "unit": "expert-tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} steps, each 1/{n} of a single-token layer decode (routing, then both "
                                   f"routed experts on one of {n} column slices of f), over {xs_n} tokens of "
                                   f"layer copy 0 (fp64 numpy oracle, {pct_label(args.sparsity)} thresholds from "
                                   f"{W['calib_tokens']} calibration tokens; a full decode took "
                                   f"{t_full * 1e3:.0f} ms)"},
        "e2e": {"value": value, "unit": "expert-tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import sparse_expert_swiglu_gb300 as ses
    from sparse_expert_swiglu_gb300 import synth
    ses.build_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    W = WORKLOAD
    d, f, E, k, B = W["d"], W["f"], W["E"], W["k"], W["B"]
    R = max(1, args.copies)
    layers = build_layers(dev, R)
    table = calibrate(layers, dev)
    # the copies' tokens and results as rows of one buffer each (one host copy moves all)
    x_all = torch.stack([synth.tokens(B, d, 1000 + r + 100 * rank, device=dev) for r in range(R)])
    y_all = torch.empty_like(x_all)
    xs, ys = list(x_all.unbind(0)), list(y_all.unbind(0))
    ws_list = [ses.Workspace(ses.layer_workspace_bytes(layers[0], B), dev) for _ in range(R)]
    peak, peak_kind = measured_peaks()

    # per-sparsity sweep (the headline is re-timed below with the clock sampler)
    graphs, stream = capture_graphs(layers, xs, ys, ws_list)
    stack = capture_stack(layers, xs, ys, ws_list, stream)
    sweep = []
    for pct in (() if args.no_sweep else SPARSITIES):
        set_thresholds(layers, table, pct)
        byts = algorithmic_bytes(layers, xs, ws_list)
        nsteps = max(200, args.steps // 4)
        secs = time_steps(graphs, stream, nsteps, args.warmup, world, dev, stack=stack)
        us = secs / nsteps * 1e6
        mean_bytes = float(np.mean([b["total"] for b in byts]))
        sweep.append(dict(sparsity_pct=pct, layer_us=us, expert_tokens_per_s=B * k / (us * 1e-6),
                          hbm_gbs=mean_bytes / (us * 1e-6) / 1e9,
                          frac_of_measured_hbm=mean_bytes / (us * 1e-6) / 1e9 / peak,
                          bytes_per_step=mean_bytes,
                          kept_fraction=float(np.mean([b["kept_frac"] for b in byts]))))
        if rank == 0:
            print(f"sweep {sweep[-1]}", file=sys.stderr, flush=True)

    pct = args.sparsity
    set_thresholds(layers, table, pct)
    byts = algorithmic_bytes(layers, xs, ws_list)
    with ClockSampler(local) as clk:
        t_start = time.perf_counter()
        secs = time_steps(graphs, stream, args.steps, args.warmup, world, dev, stack=stack)
        # keep the same load running until the sampler has seen >= 1 s of it
        while time.perf_counter() - t_start < 1.2:
            time_steps(graphs, stream, 2000, 0, 1, dev, stack=stack)
    secs = max_over_ranks(world, secs, dev)
    # the same steps with one graph launch per layer (no dependent launch across layers)
    secs_single = max_over_ranks(world, time_steps(graphs, stream, args.steps, 0, world, dev), dev)
    pairs = sum_over_ranks(world, B * k * args.steps, dev)
    value = pairs / secs
    ms_per_step = secs / args.steps * 1e3
    mean_bytes = float(np.mean([b["total"] for b in byts]))
    dist = step_distribution(stack, stream, R, max(20, args.steps // R))

    # per-kernel device times (events around each kernel inside graphs)
    events_list = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(R)]
    for evs in events_list:  # create the events before they are captured
        for ev in evs:
            ev.record()
    torch.cuda.synchronize()
    path = ses.layer_path(layers[0], B)
    prof_graphs, pstream = capture_graphs(layers, xs, ys, ws_list, events_list)
    kt = per_kernel_times(prof_graphs, events_list, pstream, max(R * 50, args.steps // 10), path)
    up_b = float(np.mean([b["up"] for b in byts]))
    ga_b = float(np.mean([b["gather"] for b in byts]))
    rt_b = float(np.mean([b["route"] for b in byts]))
    if path == "decode_fused":
        # one kernel: router, up projection, kept rows, combination
        kernel_bytes = {"decode_layer_kernel": up_b + rt_b + ga_b}
    elif path == "decode":
        # the up kernel also reads the router weight and the tokens
        kernel_bytes = {"decode_up_kernel": up_b + rt_b, "decode_gather_kernel": ga_b}
    else:
        kernel_bytes = {"up_kernel": up_b, "gather_kernel": ga_b, "route_kernel": rt_b}
    dominant = max((k for k in kernel_bytes if k in kt and k != "route_kernel"), key=lambda kname: kt[kname])
    achieved = kernel_bytes[dominant] / (kt[dominant] * 1e-6) / 1e9
    traffic = NCU_TRAFFIC.get((dominant, source_hash(dominant)))

    # end to end through the public API: every step's token in from pinned host memory,
    # its result out to pinned host memory.  Headline: the stacked graph with the copies
    # inside it (the R inputs in one copy ahead of the first layer, the R results in one
    # copy after the last), ceil(K / R) replays of R steps.  Also reported: one
    # step at a time (copy in, one layer's graph, copy out, all on one stream).
    x_host = torch.stack([synth.tokens(B, d, 5000 + i, device="cpu") for i in range(64)]).pin_memory()
    y_host = torch.empty((args.steps, B, d), dtype=torch.float16).pin_memory()
    x_pin = torch.stack([synth.tokens(B, d, 6000 + r, device="cpu") for r in range(R)]).pin_memory()
    y_pin = torch.empty((R, B, d), dtype=torch.float16).pin_memory()
    e2e_graph = capture_stack_e2e(layers, x_all, y_all, ws_list, stream, x_pin, y_pin)
    reps = -(-args.steps // R)
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // R)):
            e2e_graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            e2e_graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_secs = max_over_ranks(world, e0.elapsed_time(e1) / 1e3, dev)
    e2e_value = sum_over_ranks(world, B * k * reps * R, dev) / e2e_secs

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            xs[i % R].copy_(x_host[i % 64], non_blocking=True)
            graphs[i % R].replay()
            y_host[i % args.steps].copy_(ys[i % R], non_blocking=True)
    torch.cuda.synchronize()
    barrier(world)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            xs[i % R].copy_(x_host[i % 64], non_blocking=True)
            graphs[i % R].replay()
            y_host[i].copy_(ys[i % R], non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_step_secs = max_over_ranks(world, e0.elapsed_time(e1) / 1e3, dev)
    e2e_step_value = sum_over_ranks(world, B * k * args.steps, dev) / e2e_step_secs

    hook = prefetch_hook_times(layers, xs, ys, ws_list, stream, max(R * 50, args.steps // 4), args.warmup)

    # the further configurations, measured in this run too (one GPU, replicas only)
    further = []
    if world == 1 and not args.no_further:
        def keep(rec):
            further.append({key: rec[key] for key in ("workload", "tokens", "sparsity_pct", "path", "layer_us",
                                                      "expert_tokens_per_s", "bytes_per_step",
                                                      "frac_of_measured_hbm", "kept_fraction",
                                                      "layers_per_graph", "chained")})
        for wname, toks in FURTHER_POINTS:
            run_workload(args, world, rank, local, workload=wname, tokens=toks, emit=keep)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        xs_o, wr_o, experts_o = oracle_prepare(dev, 2, table, pct)
        n_o = 6
        osecs = time_oracle(xs_o, wr_o, experts_o, n_o, 1)
        cpu = {"value": B * k * n_o / osecs, "unit": "expert-tokens/s", "cores": oracle_threads(),
               "kind": "oracle",
               "sample": f"{n_o} single-token layer decodes (2 tokens of layer copy 0, {pct}% thresholds), "
                         "fp64 numpy oracle"}

    if rank != 0:
        return
    line = {
        "metric": METRIC.replace("70%", pct_label(pct)), "value": value, "unit": "expert-tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": config_dict(pct, R, world),
        "layer_us": ms_per_step * 1e3,
        "layer_us_one_graph_per_layer": secs_single / args.steps * 1e6,
        "layer_us_distribution": dist,
        "layer_roofline": {"bytes_per_step": mean_bytes, "hbm_gbs": mean_bytes / (ms_per_step * 1e-3) / 1e9,
                           "peak": peak, "frac": mean_bytes / (ms_per_step * 1e-3) / 1e9 / peak,
                           "peak_kind": peak_kind},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "bytes_per_launch": kernel_bytes[dominant], "peak_kind": peak_kind},
        "kernel_us": kt,
        "sweep": sweep,
        "e2e": {"value": e2e_value, "unit": "expert-tokens/s", "h2d_bytes_per_step": B * d * 2,
                "d2h_bytes_per_step": B * d * 2, "steps": reps * R,
                "how": "stacked graph of the R layer copies with each step's host copies inside it "
                       "(the R inputs in one copy ahead of the first layer, the R results in one "
                       "copy after the last)",
                "one_step_at_a_time": {"value": e2e_step_value, "unit": "expert-tokens/s",
                                       "how": "per step: copy in, one layer's graph, copy out, one stream"}},
        "prefetch_hook": hook,
        "further_configs": further,
        "gpu_launches": {"decode_fused": 1, "decode": 2}.get(path, 4) * args.steps,
        "path": path,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_workload(args, world, rank, local, workload=None, tokens=None, emit=None):
    """The further shapes: for every batch size and sparsity of the workload, the layer
    copies back to back in one CUDA graph (a stack: each copy's input is the previous
    copy's RMS-normalised output when `chained`, else its own tokens), timed on the
    device; algorithmic bytes from the realised masks.  One JSON line per point, or
    one dict per point to `emit` (the default run's further configurations)."""
    import sparse_expert_swiglu_gb300 as ses
    from sparse_expert_swiglu_gb300 import synth
    ses.build_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    name = workload or args.workload
    W = dict(WORKLOADS[name])
    d, f, E, k, ns = W["d"], W["f"], W["E"], W["k"], W["shared"]
    R = W["copies"] if (args.copies == N_LAYER_COPIES or workload) else max(1, args.copies)
    peak, peak_kind = measured_peaks()
    layers, tables = [], []
    xcal = synth.calibration_tokens(W["calib_tokens"], d, 7, device=dev)
    cws = ses.Workspace(ses.expert_workspace_bytes(W["calib_tokens"], d, f), dev)

    def packed(de, nexp):
        return ses.Experts.from_dense(de.w_up, de.gate_t, de.down,
                                      torch.zeros(nexp, dtype=torch.float32, device=dev), interleave=True)

    def thresholds(ex, nexp):
        ex.thr.fill_(float("inf"))  # nothing kept: only v is computed
        thr = {p: torch.zeros(nexp, dtype=torch.float32, device=dev) for p in W["sparsities"]}
        for e in range(nexp):
            _, dbg = ses.expert_sparse_swiglu(xcal, ex, e, ws=cws, debug=True)
            a = torch.sort(dbg["v"].abs().flatten()).values
            for p in W["sparsities"]:
                if p > 0:
                    thr[p][e] = a[(p * a.numel() + 99) // 100 - 1]
        return thr

    for r in range(R):
        ex = packed(synth.experts(E, d, f, 200 + r, device=dev, layer=r), E)
        sh = packed(synth.experts(ns, d, f, 200 + r, device=dev, layer=r, kind=1), ns) if ns else None
        torch.cuda.empty_cache()
        layers.append(ses.Layer(synth.router(d, E, 200 + r, device=dev, layer=r), ex, k, True, sh))
        tables.append((thresholds(ex, E), thresholds(sh, ns) if ns else None))
    host_rows = bool(W.get("host_rows"))
    h2d_gbs = None
    if host_rows:
        layers = [ses.Layer(l.w_router, l.routed.to_host_rows(), k, True,
                            l.shared.to_host_rows() if l.shared else None) for l in layers]
        torch.cuda.empty_cache()
        # the host link's copy-engine rate: 1 GiB from page-locked host memory, best of 3
        src = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
        dst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
        best = math.inf
        for _ in range(3):
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record()
            dst.copy_(src, non_blocking=True)
            a1.record()
            torch.cuda.synchronize()
            best = min(best, a0.elapsed_time(a1) / 1e3)
        h2d_gbs = (1 << 30) / best / 1e9
        del src, dst
        torch.cuda.empty_cache()
    decode = ses.layer_decode_host_rows if host_rows else ses.layer_decode
    ws_bytes = ses.layer_host_rows_workspace_bytes if host_rows else ses.layer_workspace_bytes
    up_bytes = ses.packed_bytes(d, f)
    weights_gb = sum(l.routed.gate_t.numel() * 4 + l.routed.up_packed.numel() +
                     (l.shared.gate_t.numel() * 4 + l.shared.up_packed.numel() if l.shared else 0)
                     for l in layers) / 1e9
    stream = torch.cuda.Stream()
    for B in (tokens if tokens else [args.tokens] if args.tokens else W["tokens"]):
        xs = [synth.tokens(B, d, 3000 + r + 100 * rank, device=dev) for r in range(R)]
        ys = [torch.empty_like(x) for x in xs]
        if W["chained"]:
            xs = [xs[0]] + ys[:-1]
        wss = [ses.Workspace(ws_bytes(layers[r], B), dev) for r in range(R)]
        path = "decode (host rows)" if host_rows else ses.layer_path(layers[0], B)
        # the tokens and workspaces are written on the current stream
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            for r in range(R):
                decode(xs[r], layers[r], rmsnorm=True, ws=wss[r], out=ys[r])
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        c_layers = [l.c_struct(host_rows=host_rows) for l in layers]
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for r in range(R):
                decode(xs[r], layers[r], rmsnorm=True, ws=wss[r], out=ys[r], c_layer=c_layers[r])
        torch.cuda.synchronize()
        for pct in W["sparsities"]:
            for r, layer in enumerate(layers):
                layer.routed.thr.copy_(tables[r][0][pct])
                if ns:
                    layer.shared.thr.copy_(tables[r][1][pct])
            # realised bytes, layer by layer along the same inputs
            total, kept, cols = 0.0, 0, 0
            for r, layer in enumerate(layers):
                _, dbg = decode(xs[r], layer, rmsnorm=True, ws=wss[r], out=ys[r], debug=True)
                idx = dbg["topk_idx"].cpu().numpy()
                words = dbg["mask"].cpu().numpy().astype(np.uint32)
                bits = ((words[..., None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(B, k + ns, -1)[..., :f]
                bits = bits.astype(bool)
                groups = [bits[np.nonzero(idx == e)[0], np.nonzero(idx == e)[1]] for e in sorted(set(idx.ravel().tolist()))]
                groups += [bits[:, k + s_] for s_ in range(ns)]
                for gb in groups:
                    u = int(np.any(gb, axis=0).sum())
                    kept += u
                    cols += f
                    total += up_bytes + 4 * d * u
                total += 2 * d * E + 4 * B * d
            torch.cuda.synchronize()
            reps = max(2, 200 // R)
            with torch.cuda.stream(stream):
                for _ in range(2):
                    g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            secs = max_over_ranks(world, e0.elapsed_time(e1) / 1e3, dev)
            steps = reps * R
            us = secs / steps * 1e6
            mean_bytes = total / R
            # per-kernel device times on copy 0, from events inside a graph (they
            # serialise the kernels but leave no host gaps)
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            for ev in evs:
                ev.record()
            torch.cuda.synchronize()
            ge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ge, stream=stream, capture_error_mode="thread_local"):
                decode(xs[0], layers[0], rmsnorm=True, ws=wss[0], out=ys[0], c_layer=c_layers[0],
                       events=evs)
            kacc = np.zeros(4)
            for it in range(12):
                with torch.cuda.stream(stream):
                    ge.replay()
                torch.cuda.synchronize()
                if it >= 2:
                    kacc += [evs[j].elapsed_time(evs[j + 1]) * 1e3 for j in range(4)]
            del ge
            names = (["event_pair_us", "decode_up_kernel", "decode_fetch_and_gather_kernels", "event_pair_us_2"]
                     if host_rows else
                     ["event_pair_us", "decode_up_kernel", "decode_gather_kernel", "event_pair_us_2"]
                     if path == "decode" else
                     ["event_pair_us", "decode_layer_kernel", "event_pair_us_2", "event_pair_us_3"]
                     if path == "decode_fused" else
                     ["event_pair_us", "first_pair", "other_pairs", "event_pair_us_2"]
                     if path == "decode_pairs" else ["route_kernel", "up_kernel", "gather_kernel", "combine_kernel"])
            kt = {nm: float(v) / 10 for nm, v in zip(names, kacc)}
            extra = {}
            if host_rows:
                link = 4 * d * kept / R  # kept rows over the host link per step
                extra = {"link_bytes_per_step": link, "link_gbs": link / (us * 1e-6) / 1e9,
                         "h2d_copy_gbs": h2d_gbs, "frac_of_h2d_copy": link / (us * 1e-6) / 1e9 / h2d_gbs,
                         "h2d_copy_how": "1 GiB page-locked host -> device copy in this run, best of 3"}
            rec = {
                    "workload": name, "tokens": B, "sparsity_pct": pct, "path": path, **extra,
                    "layer_us": us, "expert_tokens_per_s": world * B * k * steps / secs,
                    "bytes_per_step": mean_bytes, "hbm_gbs": mean_bytes / (us * 1e-6) / 1e9,
                    "frac_of_measured_hbm": mean_bytes / (us * 1e-6) / 1e9 / peak, "peak_kind": peak_kind,
                    "kept_fraction": kept / max(cols, 1), "layers_per_graph": R, "chained": W["chained"],
                    "steps": steps, "weights_gb": weights_gb, "kernel_us": kt,
                    "config": {"d": d, "f": f, "experts": E, "top_k": k, "shared": ns,
                               "calib_tokens": W["calib_tokens"]}}
            if emit is not None:
                emit(rec)
            elif rank == 0:
                print(json.dumps(rec), flush=True)
        del g, wss
        torch.cuda.empty_cache()
    del layers, tables
    torch.cuda.empty_cache()


def run_eamc(args):
    """Host timing of the EAM collection (match, PredictEAM, insert with replacement) and
    of a full expert cache's miss (prediction + eviction) through the Python binding, on
    seeded synthetic request matrices (each request skewed towards a few experts per
    layer).  The binding's own cost per call is reported beside it."""
    import sparse_expert_swiglu_gb300 as ses
    W = WORKLOADS[args.workload]
    L, E, cap = W["L"], W["E"], W["capacity"]
    rng = np.random.default_rng(11)
    groups = [rng.dirichlet(np.full(E, 0.3), size=L) for _ in range(16)]

    def request(iters):
        pref = groups[rng.integers(len(groups))]
        m = np.zeros((L, E), np.int32)
        for i in range(L):
            m[i] += np.bincount(rng.choice(E, size=2 * iters, p=pref[i]), minlength=E).astype(np.int32)
        return m

    eamc = ses.EAMC(L, E, cap)
    for _ in range(cap):
        eamc.insert(request(64))
    cur = request(16)
    n = 2000

    def per_call(fn):
        fn()
        t = time.perf_counter()
        for _ in range(n):
            fn()
        return (time.perf_counter() - t) / n * 1e6

    cache = ses.ExpertCache(L * 2, L, E)
    for i in range(L):
        for j in range(2):
            cache.lookup(eamc, cur, i, j)
    keys = [(i, j) for i in range(L) for j in range(2, E)]
    it = iter(keys * (n // len(keys) + 2))
    line = {
        "workload": args.workload, "L": L, "E": E, "capacity": cap, "stored": len(eamc),
        "match_us": per_call(lambda: eamc.match(cur, 1)),
        "predict_us": per_call(lambda: eamc.predict(cur, L // 2, 1)),
        "predict_4_matches_us": per_call(lambda: eamc.predict(cur, L // 2, 4)),
        "insert_full_us": per_call(lambda: eamc.insert(cur)),
        "cache_miss_evict_us": per_call(lambda: cache.lookup(eamc, cur, *next(it))),
        "binding_call_floor_us": per_call(lambda: ses.lib().moe_eamc_size(eamc.ptr())),
        "cores_used": 1, "cpu": platform_cpu(),
        "context": "the pages quote 21 us per query at 1K matrices on their CPU (matrix size not given)",
    }
    print(json.dumps(line), flush=True)


def platform_cpu():
    import platform
    return f"{platform.machine()} x{os.cpu_count()}"


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank, local)
        elif args.workload and WORKLOADS[args.workload].get("host_only"):
            if rank == 0:
                run_eamc(args)
        elif args.workload:
            run_workload(args, world, rank, local)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
