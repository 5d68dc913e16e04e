#!/usr/bin/env python3
"""Benchmark of the NVFP4-weight MoE layer on GB300: MoE-layer tokens/s.

One step = one complete layer call (router + plan + W13/SwiGLU + W2 + combine,
i.e. moe_nvfp4_plan + moe_nvfp4_forward) over one batch of seeded synthetic
tokens, with every input resident in HBM.  As in the pages' own protocol, the
calls are timed 16 to a CUDA graph, call i on the i-th of 16 distinct
allocations of the same weights with its own token batch (the routes change
from call to call), so that weights stream from HBM as in a layer stack; the
L2 cache is also flushed (a 2x-L2 buffer is written) before every replay,
outside its events.  Exactly --steps calls are timed (the remainder of a
16-call graph runs as a shorter graph).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workloads A,B,..]
    python bench.py --workload NAME        # one workload only
    python bench.py --impl reference ...   # the CPU oracle arm
    python bench.py --only-dense           # the dense projection records only
    python bench.py --stack 1 ...          # one weight allocation (profiler captures
                                           # that must hold little device memory)

Workloads (seeded; see nvfp4_weight_mixture_gb300/synth.py).  The default run
times all five in turn under the same protocol and prints one JSON line: the
headline decode_m1 (1 token, H 2048, 512 experts, top-10, I 512), with
decode_m16_bias, prefill_m8192, prefill_m8192_zipf_shared and tiny_m8 in its
"configs" map (each with its own value, roofline, e2e and clocks).

Under torchrun each rank runs the same workload on its own GPU (token-parallel
replicas, no collective on the data path); value = all ranks' tokens / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MoE-layer tokens/s"
# the headline (decode M = 1) first, then the other workloads the metric is
# quoted on (M = 16, M = 8192) and the remaining seeded ones
DEFAULT_WORKLOADS = ["decode_m1", "decode_m16_bias", "prefill_m8192",
                     "prefill_m8192_zipf_shared", "prefill_m784", "tiny_m8"]
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workloads", default=",".join(DEFAULT_WORKLOADS),
                   help="comma-separated workloads; the first is the headline line, the "
                        "others are timed the same way into its \"configs\" map")
    p.add_argument("--workload", default=None, help="time this one workload only")
    p.add_argument("--tokens", type=int, default=None,
                   help="override the workload's token count (same shapes and seeds)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-dense", action="store_true",
                   help="skip the dense QPN2 / QPN8 projection records")
    p.add_argument("--only-dense", action="store_true",
                   help="time the dense QPN2 / QPN8 projection records only (one JSON line of "
                        "them)")
    p.add_argument("--stack", type=int, default=16,
                   help="calls per CUDA graph, each on its own allocation of the weights (16: the "
                        "pages' protocol; fewer holds less device memory, e.g. under a profiler)")
    p.add_argument("--crossover", default=None,
                   help="comma-separated token counts: time the forward's decode and grouped "
                        "paths at each M (one JSON line each) instead of the bench")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle sample")
    return p.parse_args()


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# accounting (algorithmic bytes and FLOPs)
# ---------------------------------------------------------------------------
def max_over_ranks(value, dist, device):
    """The largest value over the ranks (the slowest rank's time); the value
    itself without a process group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world_size, tokens_per_rank_step, steps, total_ms):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world_size * tokens_per_rank_step * steps / (total_ms / 1e3)


def w13_expert_bytes(wl):
    return 2 * wl.I * wl.H // 2 + 2 * wl.I * wl.H // 16 + 4


def w2_expert_bytes(wl):
    return wl.H * wl.I // 2 + wl.H * wl.I // 16 + 4


def layer_accounting(wl, n_active, n_pairs):
    """Algorithmic bytes / FLOPs of one layer call: weights of the touched
    experts (routed + shared), router weight, x, y, bias; FLOPs of the router,
    gate and every pair's MLP.  Intermediates (h, partials) are not counted."""
    bytes_ = n_active * (w13_expert_bytes(wl) + w2_expert_bytes(wl))
    bytes_ += wl.H * wl.E * 2 + wl.M * wl.H * 2 * 2
    if wl.bias != "none":
        bytes_ += wl.E * 4
    if wl.shared:
        bytes_ += wl.H * 2
    flops = 2 * wl.M * wl.H * wl.E + n_pairs * (2 * wl.H * 2 * wl.I + 2 * wl.I * wl.H)
    if wl.shared:
        flops += 2 * wl.M * wl.H
    return bytes_, flops


def kernel_accounting(wl, step, n_active, n_pairs, decode):
    """(bound, algorithmic bytes, algorithmic FLOPs) of one launch of a traced step."""
    H, I, M = wl.H, wl.I, wl.M
    if step == "w13":
        b = n_active * w13_expert_bytes(wl) + M * H * 2 + n_pairs * I * 2
        f = n_pairs * 2 * H * 2 * I
    elif step == "w2":
        # decode: the combine runs inside the W2 kernel (writes y); prefill: FP16 partials
        out = M * H * 2 if decode else n_pairs * H * 2
        b = n_active * w2_expert_bytes(wl) + n_pairs * I * 2 + out
        f = n_pairs * 2 * I * H
    elif step == "combine":
        b = n_pairs * H * 2 + M * H * 2
        f = n_pairs * H
    else:  # plan: router weight + x + ids / weights
        b = H * wl.E * 2 + M * H * 2 + n_pairs * 8
        f = 2 * M * H * wl.E
    bound = "hbm" if (decode or step in ("combine", "plan")) else "tensor"
    return bound, b, f


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def load_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when the summary is missing or the kernel sources changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    src = os.path.join(ROOT, "nvfp4_weight_mixture_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(src)):
        with open(os.path.join(src, f), "rb") as fh:
            h.update(fh.read())
    sha = h.hexdigest()[:16]
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and parts[0] == workload and parts[1] == kernel:
                return float(parts[2]) if parts[3] == sha else None
    return None


# ---------------------------------------------------------------------------
# clocks sampler (nvidia-smi during the timed region)
# ---------------------------------------------------------------------------
class Clocks:
    """nvidia-smi samples every 50 ms, each stamped; only the samples taken
    between region_begin() and region_end() are reported (all of them, marked
    "in_region": false, if the region was too short to catch one)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # the first sample lands before the region opens
        except Exception:
            self.proc = None

    def region_begin(self):
        self.t0 = time.time()

    def region_end(self):
        self.t1 = time.time()

    @staticmethod
    def parse(out, t0=None, t1=None):
        """(samples inside [t0, t1], all samples), each (sm, max_sm, reasons)."""
        import datetime
        inside, every = [], []
        for line in out.splitlines():
            v = [x.strip() for x in line.split(",")]
            if len(v) < 9:
                continue
            try:
                s = (float(v[1]), float(v[2]),
                     {n for n, f in zip(Clocks.NAMES, v[5:9]) if f.lower() == "active"})
            except ValueError:
                continue
            every.append(s)
            try:
                ts = datetime.datetime.strptime(v[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if t0 is not None and t1 is not None and t0 <= ts <= t1:
                inside.append(s)
        return inside, every

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        inside, every = self.parse(out, self.t0, self.t1)
        use = inside or every
        if not use:
            return None
        return {"sm_mhz": statistics.median(s[0] for s in use),
                "sm_max_mhz": max(s[1] for s in use),
                "reasons": sorted(set().union(*(s[2] for s in use))),
                "samples": len(use), "in_region": bool(inside)}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(wl, seconds, max_tokens=None):
    """Times the oracle (router + plan-free forward, as it stands) on sampled
    tokens of the workload, batched so that all host cores are used.  Weights
    of the touched experts are quantised by the oracle before timing."""
    import oracle
    from nvfp4_weight_mixture_gb300 import synth
    cores = len(os.sched_getaffinity(0))
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    # token pool: decode workloads draw fresh token batches (variants)
    pool = []
    v = 0
    while sum(len(p) for p in pool) < max(4 * cores, 64):
        pool.append(synth.activations(wl, 100 + v))
        v += 1
    x = np.concatenate(pool)[: max(4 * cores, 64)]
    wr = synth.router_weight(wl)
    bias = synth.router_bias(wl)
    wg = synth.gate_weight(wl)
    E, H, I = wl.E, wl.H, wl.I

    def route(xb):
        _, ids, w = oracle.router(xb, wr, bias, wl.k)
        gm = oracle.shared_gate(xb, wg) if wl.shared else None
        return ids, w, gm

    # quantise the experts of the first batch (outside timing)
    o13 = (np.zeros((E, 2 * I, H // 2), np.uint8), np.zeros((E, 2 * I, H // 16), np.uint8),
           np.ones((E,), np.float32))
    o2 = (np.zeros((E, H, I // 2), np.uint8), np.zeros((E, H, I // 16), np.uint8),
          np.ones((E,), np.float32))
    have = set()
    shared = None
    if wl.shared:
        a = oracle.quantize(synth.shared_w13(wl)[None])
        b = oracle.quantize(synth.shared_w2(wl)[None])
        shared = ((a[0][0], a[1][0], a[2][0]), (b[0][0], b[1][0], b[2][0]))

    def ensure(ids):
        for e in set(int(e) for e in ids.ravel()) - have:
            a = oracle.quantize(synth.expert_w13(wl, e)[None])
            b = oracle.quantize(synth.expert_w2(wl, e)[None])
            for i in range(3):
                o13[i][e] = a[i][0]
                o2[i][e] = b[i][0]
            have.add(e)

    batch = cores
    done = 0
    elapsed = 0.0
    idx = 0
    while True:
        sel = np.arange(idx, idx + batch) % len(x)
        idx += batch
        xb = np.ascontiguousarray(x[sel])
        # expert weights are prepared outside the timed region
        ids_pre, _, _ = route(xb)
        ensure(ids_pre)
        t0 = time.perf_counter()
        ids, w, gm = route(xb)
        oracle.forward(xb, ids, w, o13, o2, shared=shared, gamma=gm)
        elapsed += time.perf_counter() - t0
        done += len(sel)
        if elapsed >= seconds or (max_tokens is not None and done >= max_tokens):
            break
    return done / elapsed, cores, done, elapsed


def run_reference(args, wl):
    ws, rank, _ = dist_info()
    if rank != 0:
        return 0
    steps = args.steps or 10
    warmup = args.warmup if args.warmup is not None else 1
    per_step = max(1, min(wl.M, len(os.sched_getaffinity(0))))
    budget = 150.0 / max(steps + warmup, 1)
    if warmup:
        oracle_sample(wl, 0.0, max_tokens=per_step * warmup)
    rate, cores, done, el = oracle_sample(wl, budget * steps, max_tokens=per_step * steps)
    ms = 1000.0 * wl.M / rate
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT,
        "n_gpus": args.gpus, "steps": steps, "warmup": warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(wl),
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{done} tokens of {wl.name} in {el:.1f} s (batches of "
                                   f"{cores}), C oracle as it stands"},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl):
    return {"workload": wl.name, "tokens": wl.M, "hidden": wl.H, "experts": wl.E,
            "top_k": wl.k, "intermediate": wl.I, "router_bias": wl.bias,
            "shared_expert": wl.shared,
            "weights": "NVFP4 (E2M1, E4M3 per 16 along K, FP32 per tensor) from N(0,0.02)",
            "activations": "FP16 N(0,1), 16 rotating token batches",
            "l2": f"{STACK} complete layer calls per CUDA graph, call i on the i-th of {STACK} "
                  "distinct allocations of the same weights; 2x L2 buffer written before every "
                  "replay",
            "parallelism": "token-parallel replicas, no collective"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def build_layer(wl, dev, moe, synth):
    import torch
    from concurrent.futures import ThreadPoolExecutor
    E, H, I = wl.E, wl.H, wl.I
    q13 = torch.empty((E, I * H), dtype=torch.uint8, device=dev)
    s13 = torch.empty((E, I * H // 8), dtype=torch.uint8, device=dev)
    g13 = torch.empty((E,), dtype=torch.float32, device=dev)
    q2 = torch.empty((E, H * I // 2), dtype=torch.uint8, device=dev)
    s2 = torch.empty((E, H * I // 16), dtype=torch.uint8, device=dev)
    g2 = torch.empty((E,), dtype=torch.float32, device=dev)
    chunk = 32
    with ThreadPoolExecutor(min(16, os.cpu_count() or 4)) as pool:
        for e0 in range(0, E, chunk):
            e1 = min(E, e0 + chunk)
            a = np.stack(list(pool.map(lambda e: synth.expert_w13(wl, e), range(e0, e1))))
            moe.quantize(torch.from_numpy(a).to(dev), moe.LAYOUT_FRAGMENT_W13, q=q13[e0:e1],
                         s=s13[e0:e1], g=g13[e0:e1])
            b = np.stack(list(pool.map(lambda e: synth.expert_w2(wl, e), range(e0, e1))))
            moe.quantize(torch.from_numpy(b).to(dev), moe.LAYOUT_FRAGMENT, q=q2[e0:e1],
                         s=s2[e0:e1], g=g2[e0:e1])
    sh13 = sh2 = None
    if wl.shared:
        sh13 = moe.quantize(torch.from_numpy(synth.shared_w13(wl)).to(dev), moe.LAYOUT_FRAGMENT_W13)
        sh2 = moe.quantize(torch.from_numpy(synth.shared_w2(wl)).to(dev), moe.LAYOUT_FRAGMENT)
    wr = torch.from_numpy(synth.router_weight(wl)).to(dev)
    bias = synth.router_bias(wl)
    wg = synth.gate_weight(wl)
    layer = moe.MoELayer(H, E, wl.k, I, wr, (q13, s13, g13), (q2, s2, g2), sh13, sh2,
                         None if wg is None else torch.from_numpy(wg).to(dev),
                         None if bias is None else torch.from_numpy(bias).to(dev),
                         max_tokens=wl.M, device=dev)
    return layer


# Timing protocol of the pages ("[Kernel][SM70] Improve Qwen3.8 no-MTP
# concurrency", sections "Test Result" and "Latest grouped-MoE screen"): hot
# single-call timing misleads, so the layer is timed as 16 complete calls per
# CUDA graph, call i on the i-th of 16 distinct allocations of the same
# weights (a layer-like weight working set: what one call reads is evicted
# from L2 by the 15 others before it comes round again).
STACK = 16


def clone_layer(layer, moe):
    """Another allocation of the same layer (a copy of every weight tensor),
    sharing the plan and workspace buffers of `layer`."""
    c = lambda t: None if t is None else t.clone()
    cw = lambda w: None if w is None else tuple(t.clone() for t in w)
    L = moe.MoELayer(layer.H, layer.E, layer.k, layer.I, c(layer.w_router), cw(layer.w13),
                     cw(layer.w2), cw(layer.shared13), cw(layer.shared2), c(layer.w_gate),
                     c(layer.bias), max_tokens=0, device=layer.device)
    L.plan_buf, L.ws, L.max_tokens, L.status = layer.plan_buf, layer.ws, layer.max_tokens, layer.status
    return L


def _plan_stats(layer):
    """(touched experts, valid pairs) of the plan in the layer's plan buffer."""
    import torch
    h = layer.plan_buf[:64].view(torch.int32).cpu().numpy()
    return int(h[3]), int(h[5])


def time_workload(wl, args, dist, dev, local, ws, rank):
    """Times one workload under the bench protocol on this rank; returns the
    per-workload record (rank 0 reads it; other ranks return after the
    collectives)."""
    import torch
    from nvfp4_weight_mixture_gb300 import moe, synth

    decode = wl.M <= moe.DECODE_MAX_TOKENS
    steps = args.steps or (5000 if decode else 300)
    warmup = max(3, args.warmup if args.warmup is not None else 10)

    layer = build_layer(wl, dev, moe, synth)
    n_var = max(16, STACK)  # token batches (the routes change from call to call)
    xs = [torch.from_numpy(synth.activations(wl, v)).to(dev) for v in range(n_var)]
    ys = [torch.empty((wl.M, wl.H), dtype=torch.float16, device=dev) for _ in range(n_var)]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    # warm-up (eager), the plan statistics of every token batch
    touched, pairs = [], []
    with torch.cuda.stream(stream):
        for i in range(max(warmup, n_var)):
            layer(xs[i % n_var], ys[i % n_var])
            if i < n_var:
                stream.synchronize()
                a, p_ = _plan_stats(layer)
                touched.append(a)
                pairs.append(p_)
    stream.synchronize()
    n_active, n_valid = statistics.mean(touched), statistics.mean(pairs)
    # 16 distinct allocations of the same layer (same bytes, other addresses),
    # sharing the plan and workspace buffers (the calls run in stream order)
    stack = [layer] + [clone_layer(layer, moe) for _ in range(STACK - 1)]

    def capture(n_calls):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_calls):
                stack[i](xs[i], ys[i])
        return g

    g_full = capture(STACK)
    n_full, n_rem = divmod(steps, STACK)
    g_rem = capture(n_rem) if n_rem else None
    with torch.cuda.stream(stream):
        for i in range(warmup):
            flush.zero_()
            g_full.replay()
    stream.synchronize()
    # this library's kernels per step: decode = router/plan cluster, W13, W2;
    # prefill = router (tensor-core path: W_r transpose + per 8192-token chunk
    # logits and top-k; else one mma.sync router), histogram, scan, scatter,
    # row gather, W13, W2, combine
    if decode:
        launches_per_step = 3
    else:
        tc_router = wl.E >= 256 and wl.E % 16 == 0 and wl.M >= 128
        n_chunks = -(-wl.M // 8192)
        launches_per_step = (1 + 2 * n_chunks if tc_router else 1) + 7

    # ---- timed region: exactly `steps` layer calls, as replays of the 16-call
    # graph (and one shorter graph for the remainder); L2 flushed before each
    # replay, outside its events ------------------------------------------------
    plan_ = [g_full] * n_full + ([g_rem] if g_rem is not None else [])
    calls = [STACK] * n_full + ([n_rem] if n_rem else [])
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(len(plan_))]
    clocks = Clocks(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    clocks.region_begin()
    t_wall = time.perf_counter()
    with torch.cuda.stream(stream):
        for i, g in enumerate(plan_):
            flush.zero_()
            ev[i][0].record(stream)
            g.replay()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clocks.region_end()
    ck = clocks.stop()
    times = [a.elapsed_time(b) for a, b in ev]
    per_call = [t / c for t, c in zip(times, calls)]
    total_ms = max_over_ranks(sum(times), dist, dev)
    if dist:
        dist.barrier()
    ms_per_step = total_ms / steps
    value = job_tokens_per_s(ws, wl.M, steps, total_ms)
    del g_full, g_rem, stack[1:]

    # ---- per-kernel durations inside graph-replayed steps ------------------------
    # The library records caller events around each of its kernels; captured
    # into the step's graph they become event nodes, so every kernel is timed
    # as it runs in the replayed step (same flush protocol).  The event nodes
    # order the kernels, so a traced step runs without programmatic-launch
    # overlap: its kernels add up to a little more than the untraced step.
    tr = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    moe.set_trace_events(tr)
    tgraphs = []
    for v in range(4):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            layer(xs[v], ys[v])
        tgraphs.append(g)
    kt = {s_: [] for s_ in moe.TRACE_STEPS}
    span = []
    n_tr = min(steps, 100)
    with torch.cuda.stream(stream):
        for i in range(n_tr):
            flush.zero_()
            tgraphs[i % len(tgraphs)].replay()
            stream.synchronize()
            for j, s_ in enumerate(moe.TRACE_STEPS):
                kt[s_].append(tr[2 * j].elapsed_time(tr[2 * j + 1]))
            span.append(tr[0].elapsed_time(tr[7]))
    moe.set_trace_events(None)
    del tgraphs
    kernel_ms = {s_: statistics.mean(v) for s_, v in kt.items()}
    traced_step_ms = statistics.mean(span)
    # On the decode path the combine runs inside the W2 kernel, so its record
    # pair encloses no kernel: that pair's time is the cost of one pair of
    # event nodes, taken off every traced kernel's duration.
    event_pair_ms = kernel_ms["combine"] if decode else 0.0
    kernel_ms_raw = dict(kernel_ms)
    if decode:
        kernel_ms = {s_: max(v - event_pair_ms, 0.0) for s_, v in kernel_ms.items()}
    st = int(layer.status.item())

    # ---- end to end through the public API: pinned H2D + layer + D2H ------------
    xh = [torch.from_numpy(synth.activations(wl, v)).pin_memory() for v in range(n_var)]
    yh = torch.empty((wl.M, wl.H), dtype=torch.float16).pin_memory()
    xd = torch.empty_like(xs[0])
    yd = torch.empty_like(ys[0])
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(warmup):
            xd.copy_(xh[i % n_var], non_blocking=True)
            layer(xd, yd)
            yh.copy_(yd, non_blocking=True)
    stream.synchronize()
    if dist:
        dist.barrier()
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.zero_()
            eev[i][0].record(stream)
            xd.copy_(xh[i % n_var], non_blocking=True)
            layer(xd, yd)
            yh.copy_(yd, non_blocking=True)
            eev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in eev), dist, dev)
    e2e_value = job_tokens_per_s(ws, wl.M, steps, e2e_ms)
    del layer, xs, ys, flush, xh
    torch.cuda.empty_cache()

    # ---- roofline of the dominant kernel -------------------------------------------
    hbm, tflops, peak_src = load_peaks()
    dom = max(("w13", "w2", "combine", "plan") if not decode else ("w13", "w2", "plan"),
              key=lambda s_: kernel_ms[s_])
    bound, kb, kf = kernel_accounting(wl, dom, n_active, n_valid, decode)
    dur = kernel_ms[dom] / 1e3
    if bound == "hbm":
        achieved, peak, unit = kb / dur / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit = kf / dur / 1e12, tflops, "TFLOP/s"
    traffic = load_traffic(wl.name, dom)
    lb, lf = layer_accounting(wl, n_active, n_valid)
    step_s = ms_per_step / 1e3
    layer_roof = max(lb / (hbm * 1e9), lf / (tflops * 1e12))
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": workload_config(wl),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic, "kernel": dom,
                     "peak_source": f"{peak_src} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops'}"
                                    f"{', fp16 = bf16 nominal rate' if bound == 'tensor' else ''})",
                     "kernel_timing": "event nodes captured in the replayed step graph",
                     "algorithmic": {"bytes": kb, "flops": kf, "kernel_ms": kernel_ms[dom]}},
        "layer": {"algorithmic_bytes": lb, "flops": lf, "touched_experts": n_active,
                  "pairs": n_valid, "roofline_us": layer_roof * 1e6,
                  "frac_of_roofline": layer_roof / step_s,
                  "hbm_gbs_achieved": lb / step_s / 1e9,
                  "tensor_tflops_achieved": lf / step_s / 1e12,
                  "step_ms_p10_p50_p90": [float(np.percentile(per_call, q)) for q in (10, 50, 90)],
                  "kernel_ms_in_graph": kernel_ms, "kernel_ms_in_graph_raw": kernel_ms_raw,
                  "event_pair_ms": event_pair_ms, "traced_step_ms": traced_step_ms,
                  "status": st},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": wl.M * wl.H * 2,
                "d2h_bytes_per_step": wl.M * wl.H * 2},
        "gpu_launches": launches_per_step * steps,
        "clocks": ck,
        "wall_s_timed_region": wall,
    }


def run_crossover(args):
    """The M crossover of the forward's two paths (the pages' M-bucketed
    dispatch): per-call time of the layer in the 16-call stack for M tokens of
    the prefill_m8192 layer (uniform routing) through the weight-streaming
    decode kernels (M <= 16) and through the grouped tensor-core GEMMs (any
    M).  Prints one JSON line per (M, path)."""
    import torch
    from nvfp4_weight_mixture_gb300 import moe, synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    moe.load_library()
    base = synth.WORKLOADS["prefill_m8192"]
    Ms = [int(v) for v in args.crossover.split(",")]
    layer = build_layer(synth.with_tokens(base, max(Ms)), dev, moe, synth)
    stack = [layer] + [clone_layer(layer, moe) for _ in range(STACK - 1)]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    reps = args.steps or 20
    for M in Ms:
        wl = synth.with_tokens(base, M)
        xs = [torch.from_numpy(synth.activations(wl, v)).to(dev) for v in range(STACK)]
        ys = [torch.empty((M, wl.H), dtype=torch.float16, device=dev) for _ in range(STACK)]
        for path, bucket in (("decode_gemv", 16), ("grouped_tcgen05", 0)):
            if path == "decode_gemv" and M > moe.DECODE_MAX_TOKENS:
                continue
            moe.set_decode_max_tokens(bucket)
            try:
                with torch.cuda.stream(stream):
                    for i in range(STACK):
                        stack[i](xs[i], ys[i])
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(STACK):
                        stack[i](xs[i], ys[i])
                ts = []
                with torch.cuda.stream(stream):
                    for r in range(reps + 3):
                        flush.zero_()
                        a = torch.cuda.Event(enable_timing=True)
                        b = torch.cuda.Event(enable_timing=True)
                        a.record(stream)
                        g.replay()
                        b.record(stream)
                        stream.synchronize()
                        if r >= 3:
                            ts.append(a.elapsed_time(b) / STACK)
                del g
            finally:
                moe.set_decode_max_tokens(16)
            us = statistics.median(ts) * 1e3
            print(json.dumps({"crossover": True, "M": M, "path": path, "us_per_call": us,
                              "tokens_per_s": M / (us * 1e-6),
                              "status": int(layer.status.item())}), flush=True)
    return 0


def time_dense(wl, fmt, args, dev):
    """The dense few-row projection (QPN2 NVFP4 or QPN8 channel-FP8) of a
    dense workload under the same protocol as the layer: 16 calls per CUDA
    graph over 16 distinct allocations of the same weights, a 2x-L2 buffer
    written before every replay.  Returns the record for the configs map."""
    import torch
    from nvfp4_weight_mixture_gb300 import moe, synth
    w = torch.from_numpy(synth.dense_weight(wl)).to(dev)
    if fmt == "fp8":
        q, cs = moe.fp8_quantize(w, moe.LAYOUT_FP8_FRAGMENT)
        mats = [(q.clone(), cs.clone()) for _ in range(STACK)]
        wbytes = wl.N * wl.K + 4 * wl.N
    else:
        q, sc, g = moe.quantize(w[None], moe.LAYOUT_FRAGMENT)
        mats = [(q.reshape(-1).clone(), sc.reshape(-1).clone(), g.clone()) for _ in range(STACK)]
        wbytes = wl.N * wl.K // 2 + wl.N * wl.K // 16 + 4
    del w
    xs = [torch.from_numpy(synth.dense_activations(wl, v)).to(dev) for v in range(STACK)]
    ys = [torch.empty((wl.M, wl.N), dtype=torch.float16, device=dev) for _ in range(STACK)]
    ws = torch.zeros(max(moe.dense_query(wl.M, wl.N, wl.K), 16), dtype=torch.uint8, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def call(i):
        if fmt == "fp8":
            moe.fp8_dense(xs[i], mats[i][0], mats[i][1], y=ys[i], ws=ws)
        else:
            moe.dense(xs[i], mats[i], wl.N, y=ys[i], ws=ws)
    with torch.cuda.stream(stream):
        for i in range(STACK):
            call(i)
    stream.synchronize()
    g_ = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_, stream=stream):
        for i in range(STACK):
            call(i)
    reps = max(3, (args.steps or 320) // STACK)
    ts = []
    with torch.cuda.stream(stream):
        for r in range(reps + 3):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g_.replay()
            b.record(stream)
            stream.synchronize()
            if r >= 3:
                ts.append(a.elapsed_time(b) / STACK)
    us = statistics.median(ts) * 1e3
    hbm, _, peak_src = load_peaks()
    byts = wbytes + wl.M * wl.K * 2 + wl.M * wl.N * 2
    achieved = byts / (us * 1e-6) / 1e9
    del g_, mats, xs, ys, flush
    torch.cuda.empty_cache()
    return {"value": wl.M / (us * 1e-6), "unit": "tokens/s", "us_per_call": us,
            "calls": reps * STACK,
            "config": {"workload": wl.name, "format": "NVFP4 (QPN2)" if fmt == "nvfp4"
                       else "channel-FP8 (QPN8)", "M": wl.M, "N": wl.N, "K": wl.K},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_source": f"{peak_src} (hbm_gbs)",
                         "algorithmic": {"bytes": byts}}}


def run_dense_only(args):
    """The dense projection records alone, one JSON line {"dense": {...}}."""
    import torch
    from nvfp4_weight_mixture_gb300 import moe, synth
    dev = torch.device("cuda", 0)
    moe.load_library()
    out = {}
    for dn in ("dense_gate_up_m16", "dense_down_m16"):
        for fmt in ("nvfp4", "fp8"):
            out[f"{dn}_{fmt}"] = time_dense(synth.DENSE_WORKLOADS[dn], fmt, args, dev)
    print(json.dumps({"dense": out}), flush=True)
    return 0


def run_gpu(args, workloads):
    """Times every workload (the first is the headline line; the others go
    into its "configs" map, each measured under the same protocol)."""
    import torch
    from nvfp4_weight_mixture_gb300 import moe

    ws, rank, local = dist_info()
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe.load_library()
    recs = [time_workload(wl, args, dist, dev, local, ws, rank) for wl in workloads]
    dense = {}
    if args.workload is None and not args.no_dense:
        from nvfp4_weight_mixture_gb300 import synth
        for dn in ("dense_gate_up_m16", "dense_down_m16"):
            for fmt in ("nvfp4", "fp8"):
                dense[f"{dn}_{fmt}"] = time_dense(synth.DENSE_WORKLOADS[dn], fmt, args, dev)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    line = recs[0]
    if len(recs) > 1:
        line["configs"] = {}
        for wl, r in zip(workloads[1:], recs[1:]):
            line["configs"][wl.name] = {k_: r[k_] for k_ in (
                "value", "unit", "ms_per_step", "steps", "warmup", "config", "roofline", "layer",
                "e2e", "gpu_launches", "clocks", "wall_s_timed_region")}
    if dense:
        line.setdefault("configs", {}).update(dense)
    wl = workloads[0]
    if ws == 1 and not args.no_cpu_baseline:
        rate, cores, done, el = oracle_sample(wl, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{done} tokens of {wl.name} in {el:.1f} s (batches of"
                                          f" {cores} tokens; router + forward), C oracle as it "
                                          f"stands"}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    global STACK
    args = parse_args()
    if args.stack < 1:
        raise SystemExit("--stack must be at least 1")
    STACK = args.stack
    from nvfp4_weight_mixture_gb300 import synth
    names = [args.workload] if args.workload else args.workloads.split(",")
    for n in names:
        if n not in synth.WORKLOADS:
            raise SystemExit(f"unknown workload {n}; one of {list(synth.WORKLOADS)}")
    wls = [synth.WORKLOADS[n] for n in names]
    if args.tokens is not None:
        wls = [synth.with_tokens(w, args.tokens) for w in wls]
    if args.impl == "reference":
        return run_reference(args, wls[0])
    if args.crossover:
        return run_crossover(args)
    if args.only_dense:
        return run_dense_only(args)
    return run_gpu(args, wls)


if __name__ == "__main__":
    sys.exit(main())
