"""Benchmark of the routed-expert VQ2 MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole layer (router logits, top-k, permutation,
expert FFN, combine) over one batch of synthetic tokens, for each layer of
the workload.  Default workload: decode batch 1 (hidden 4096, intermediate
2048, 256 experts, top-8, all experts resident, 4 independent layers).  The
value is MoE-layer tokens per second (tokens x layers / time).  Inputs
already sit in HBM when the timed region starts; the e2e figure adds the
pinned-host -> device copy of each step's tokens and the device -> host copy
of the layer outputs.  The roofline entry covers the expert-FFN call
(moe_vq2_expert_ffn: its schedule, FC1 and FC2 kernels), with the code +
scale bytes of each distinct expert touched as algorithmic bytes.
--impl reference times the CPU oracle on the same workload and metric.

Under torchrun (N > 1) every rank runs its own replica of the workload on its
own GPU (the layer has no exchange step); the slowest rank's time counts.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth as ms  # noqa: E402

METRIC = "MoE-layer tokens/s and achieved HBM GB/s of VQ2 code reads vs ~8 TB/s (1 GB300)"
UNIT = "layer-tokens/s"
VQ2_EXPERT_BYTES = 6_684_672     # codes + scales, gate + up + down, H=4096 I=2048
FP4_EXPERT_BYTES = 13_369_344
VQ2_EXPERT_CODE_BYTES = 6_291_456  # codes only
FP4_EXPERT_CODE_BYTES = 12_582_912
FFN_FLOP_PER_PAIR = 2 * 3 * 4096 * 2048  # gate, up and down matvecs of one (token, expert) pair
L2_BYTES = 129 * 2 ** 20

# DRAM bytes (read + write) of one expert-FFN call, from one ncu capture of its
# kernels (the two single-token table kernels, ffn_lut_kernel<1,1,0> and
# ffn_lut_kernel<0,1,0>, of `python bench.py --layers 1 --steps 3 --warmup 3
# --no-cpu` under ncu: FC1 35,727,104 + 3,840, FC2 18,553,600 at decode batch 1).
# Reported only while the kernel sources hash to the ones the counters were
# taken on.
TRAFFIC = {"decode_b1": {"bytes": 54_284_544,
                         "profile": "ncu capture of ffn_lut_kernel<1,1,0> and ffn_lut_kernel<0,1,0>, decode batch 1",
                         "sources": ["ffn_lut.cu", "lut_core.cuh", "ffn_common.cuh", "common.cuh"],
                         "sha256": "2b0d38e17623b08719a47955646d2b6e7ffa9c2e9bc753a007b5f37e221598d8"}}


# Workloads whose bench figure averages many token batches (different expert
# sets): an ncu capture of one batch's call gives its ratio, not a per-launch
# figure of the average.
TRAFFIC_ONE_BATCH = {
    "decode_b32_zipf": ("ncu capture of the call on one token batch (pool slot 0, 55 experts): 403.4 MB of DRAM "
                        "reads and writes against 367.7 MB algorithmic (1.10); the bench averages 64 batches"),
}


def measured_traffic(name):
    t = TRAFFIC.get(name)
    if t is None:
        return None, TRAFFIC_ONE_BATCH.get(name, "no ncu capture of this workload's kernels")
    import hashlib
    h = hashlib.sha256()
    for f in t["sources"]:
        with open(os.path.join(ROOT, "bit_vq_routed_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != t["sha256"]:
        return None, "kernel sources changed since the ncu capture"
    return t["bytes"], t["profile"]

WORKLOADS = {
    "decode_b1": dict(T=1, layers=4, zipf=None, fp4_top=0, pool=64,
                      desc="decode batch 1: H4096 I2048 E256 top-8 softmax, all 256 experts resident, "
                           "4 layers with independent seeded weights"),
    "decode_b32_zipf": dict(T=32, layers=1, zipf=1.1, fp4_top=0, pool=8,
                            desc="decode batch 32, Zipf(1.1) router bias, H4096 I2048 E256 top-8"),
    "mixed_fp4_b8": dict(T=8, layers=1, zipf=1.1, fp4_top=52, pool=8,
                         desc="decode batch 8, 52 most routed experts FP4 (MXFP4), 204 VQ2, Zipf(1.1)"),
    "mixed_fp4_b1": dict(T=1, layers=4, zipf=1.1, fp4_top=52, pool=64,
                         desc="decode batch 1, 52 most routed experts FP4 (MXFP4), 204 VQ2, Zipf(1.1), 4 layers "
                              "with independent seeded weights"),
    "prefill_4096": dict(T=4096, layers=1, zipf=1.1, fp4_top=0, pool=1,
                         desc="prefill chunk 4096 tokens, Zipf(1.1), H4096 I2048 E256 top-8"),
    "tandem_mixed_b8": dict(T=8, layers=1, zipf=1.1, fp4_top=52, pool=8, gpu_resident=96,
                            desc="decode batch 8, 52 most routed experts FP4, 204 VQ2, Zipf(1.1); only the 96 most "
                                 "routed experts in the GPU slot table, the pairs of the other 160 computed on "
                                 "the host's cores at the same time (GPU partial + CPU remainder)"),
    "decode_b1_fetch": dict(T=1, layers=1, zipf=1.1, fp4_top=0, pool=256, slots=64,
                            desc="decode batch 1, Zipf(1.1) router bias, H4096 I2048 E256 top-8, the 256 "
                                 "experts in page-locked host memory, a GPU expert cache of 64 slots "
                                 "(eviction by routing counts); a miss is fetched and the step's graph "
                                 "replayed"),
}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return f"{platform.machine()} ({os.cpu_count()} cores)"


def max_over_ranks(v: float, device="cuda") -> float:
    """The slowest rank's figure (the job's time); v itself without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / (ms / 1000.0)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def make_layers(wl):
    return [ms.Layer(ms.spec_decode(L, zipf_s=wl["zipf"], fp4_top=wl["fp4_top"])) for L in range(wl["layers"])]


def token_pool(wl, L):
    return ms.tokens(wl["T"] * wl["pool"], 4096, seed=1000 + L).reshape(wl["pool"], wl["T"], 4096)


# --------------------------------------------------------------- CPU oracle arm

def oracle_time(wl, layers, budget_s: float, max_steps: int, threads: int = 0):
    """Times the CPU oracle over whole steps (every layer, one batch each)
    until the budget is spent, on `threads` host threads (0 = every core).
    Weights are drawn before the clock starts."""
    import oracle
    O = oracle.default
    cores = O.set_threads(threads or os.cpu_count() or 1)
    pools = [token_pool(wl, L) for L in range(len(layers))]
    T = wl["T"]
    if T > 64:  # prefill: a bounded token sample of the chunk
        sample = np.arange(0, T, T // 16)[:16]
    else:
        sample = None
    # draw the experts each step needs before timing
    for s in range(max_steps):
        for L, layer in enumerate(layers):
            x = pools[L][s % wl["pool"]]
            lg = O.router_logits(x, layer.w_router, layer.bias)
            ids, _ = O.route_topk(lg, layer.spec.k, 1)
            sel = ids if sample is None else ids[sample]
            for e in np.unique(sel):
                layer.expert(int(e))
    done, t0, tok = 0, time.perf_counter(), 0
    while done < max_steps:
        for L, layer in enumerate(layers):
            x = pools[L][done % wl["pool"]]
            r = O.moe_layer(layer, x, tokens=sample)
            tok += len(r["tokens"])
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    what = f"{done} step(s) x {len(layers)} layer(s) x {T if sample is None else len(sample)} token(s)"
    if sample is not None:
        what += f" (token sample of the {T}-token chunk; routing of all {T} tokens included)"
    return tok / el, cores, what, done, el


# --------------------------------------------------------------- GPU arm

def run_gpu(args, wl, world, rank, local):
    import torch
    import bit_vq_routed_gb300 as bv

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    layers = make_layers(wl)
    T, nL = wl["T"], len(layers)
    devs, keeps = [], []
    for layer in layers:
        s = layer.spec
        dev, keep = bv.upload_layer(s.H, s.I, s.E, s.k, T, layer.codebook, layer.w_router, layer.bias,
                                    lambda e, L=layer: (lambda ex: (ex.fmt, ex.codes, ex.scales))(
                                        L.expert(e, cache=False)))
        devs.append(dev)
        keeps.append(keep)
    pools = [torch.from_numpy(token_pool(wl, L)).view(torch.bfloat16).cuda() for L in range(nL)]
    torch.cuda.synchronize()
    G = wl["pool"]

    def step(s, evs=None):
        for L, dev in enumerate(devs):
            x = pools[L][s % G]
            dev.route(x)
            if evs is not None:
                evs[L][0].record()
            dev.experts(x, bv.MOE_PER_PAIR)
            if evs is not None:
                evs[L][1].record()
            bv.moe_combine(dev.ypair[:T * dev.k], dev.pair_to_sorted[:T * dev.k], dev.weights[:T],
                           dev.pair_status[:T * dev.k], dev.k, dev.out[:T])

    def new_events():
        return [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(nL)]

    step(0)  # first eager step: the library sets its kernel attributes outside any capture
    torch.cuda.synchronize()
    def piece(fn):
        g = torch.cuda.CUDAGraph()
        n0 = bv.moe_launch_count()
        with torch.cuda.graph(g):
            fn()
        g.kernels = bv.moe_launch_count() - n0  # library kernel nodes in this graph
        return g

    if args.graph:
        # Per token batch s of the pool: one CUDA graph of the whole step (every
        # layer's route, expert FFN and combine, back to back with programmatic
        # dependent launch), and one of the step's expert-FFN calls alone.
        step_graphs = [piece(lambda s=s: step(s)) for s in range(G)]
        ffn_graphs = [piece(lambda s=s: [devs[L].experts(pools[L][s], bv.MOE_PER_PAIR) for L in range(nL)])
                      for s in range(G)]

        def run(s, evs=None):
            g = step_graphs[s % G]
            g.replay()
            return g.kernels
    else:
        def run(s, evs=None):
            n0 = bv.moe_launch_count()
            step(s, evs)
            return bv.moe_launch_count() - n0
    stream = torch.cuda.current_stream()
    if args.graph:
        # every graph launched once, untimed: a graph's first launch uploads
        # it (one-time setup, not work of a step)
        for s in range(G):
            step_graphs[s].replay()
            ffn_graphs[s].replay()
        torch.cuda.synchronize()
    for s in range(args.warmup):
        run(s)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    step_ev = [new_events() for _ in range(args.steps)] if not args.graph else None
    clocks = ClockSampler(local)
    clocks.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    launches = 0
    start.record(stream)
    for s in range(args.steps):
        launches += run(args.warmup + s, None if step_ev is None else step_ev[s])
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = start.elapsed_time(end)
    timed_slots = [(args.warmup + s) % G for s in range(args.steps)]
    if args.graph:
        # The expert-FFN call alone: per pool batch, the step graph (untimed)
        # leaves every layer routed, then the graph of the step's nL FFN calls
        # runs between two events; a call's time is that span / nL.
        ffn_slots = timed_slots[:min(len(timed_slots), 64)]
        ffn_ms = []
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in ffn_slots]
        for (a, b), sl in zip(ev, ffn_slots):
            step_graphs[sl].replay()
            a.record(stream)
            ffn_graphs[sl].replay()
            b.record(stream)
        torch.cuda.synchronize()
        for (a, b), sl in zip(ev, ffn_slots):
            ffn_ms += [a.elapsed_time(b) / nL] * nL
    else:
        ffn_slots = timed_slots
        ffn_ms = [step_ev[s][L][0].elapsed_time(step_ev[s][L][1]) for s in range(args.steps) for L in range(nL)]
    # distinct experts touched per FFN launch (read back after timing)
    per_slot = {}
    for sl in sorted(set(ffn_slots)):
        for L, dev in enumerate(devs):
            dev.route(pools[L][sl])
            ids = np.unique(dev.ids[:T].cpu().numpy())
            fmts = layers[L].formats[ids]
            nv, nf = int((fmts == ms.FMT_VQ2).sum()), int((fmts == ms.FMT_FP4).sum())
            per_slot[(sl, L)] = (nv * VQ2_EXPERT_BYTES + nf * FP4_EXPERT_BYTES,
                                 nv * VQ2_EXPERT_CODE_BYTES + nf * FP4_EXPERT_CODE_BYTES)
    code_bytes = [per_slot[(sl, L)][0] for sl in ffn_slots for L in range(nL)]
    codes_only = [per_slot[(sl, L)][1] for sl in ffn_slots for L in range(nL)]
    ms_total = max_over_ranks(ms_total)

    # end to end through the public API: pinned host tokens in, outputs out.
    # Graphed: PipelinedSteps (the layers of a step as one CUDA graph over
    # double-buffered device tokens and outputs; each step's tokens are
    # copied in on one stream and its outputs out on another, overlapping the
    # neighbouring steps' layers; every copy is inside the timed region).
    host_in = torch.from_numpy(np.stack([token_pool(wl, L) for L in range(nL)], axis=1)).view(
        torch.bfloat16).pin_memory()  # [G, layers, T, H]
    host_out = torch.empty(nL, T, 4096, dtype=torch.float32).pin_memory()
    if args.graph:
        pipe = bv.PipelinedSteps(devs, T)
        for s in range(3):  # warm-up
            pipe.step(host_in[s % G], host_out)
        pipe.join()
    e2e_steps = args.steps
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(e2e_steps):
        if args.graph:
            pipe.step(host_in[s % G], host_out)
            continue
        for L, dev in enumerate(devs):
            xin = host_in[s % G][L].cuda(non_blocking=True)
            out = dev.forward(xin)
            host_out[L].copy_(out, non_blocking=True)
    if args.graph:
        pipe.join()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms)
    if world > 1:
        torch.distributed.destroy_process_group()
    return dict(ms_total=ms_total, ffn_ms=ffn_ms, code_bytes=code_bytes, codes_only=codes_only, clocks=clk,
                e2e_ms=e2e_ms,
                e2e_steps=e2e_steps, launches=launches)


def run_fetch(args, wl, world, rank, local):
    """The decode step over a GPU expert cache: every expert in page-locked
    host memory, the layer's slot table filled by an ExpertCache of
    wl["slots"] slots; each step replays the routing graph, reads the routed
    ids back, names them to the cache (misses are copied in) and replays the
    expert graph (MissFetchForward)."""
    import torch
    import bit_vq_routed_gb300 as bv

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    layer = make_layers(wl)[0]
    s = layer.spec
    T, G = wl["T"], wl["pool"]
    dev = bv.MoELayer(s.H, s.I, s.E, s.k, T, layer.codebook, layer.w_router, layer.bias, s.renormalize)
    slot_bytes = bv.moe_expert_cache_slot_bytes(s.H, s.I, bv.MOE_FMT_VQ2)
    pool = torch.empty(wl["slots"] * slot_bytes, dtype=torch.uint8, device="cuda")
    cache = bv.ExpertCache(dev.table, pool, slot_bytes)
    for e in range(s.E):  # each expert one page-locked block in the slot's layout
        ex = layer.expert(e, cache=False)
        cache.set_host_image(e, ex.fmt, bv.host_expert_image(ex.fmt, ex.codes, ex.scales))
    toks = torch.from_numpy(token_pool(wl, 0)).view(torch.bfloat16).cuda()
    n0 = bv.moe_launch_count()
    mf = bv.MissFetchForward(dev, cache, T)
    graph_kernels = (bv.moe_launch_count() - n0) // 2  # one eager forward, then its two graphs
    stream = torch.cuda.current_stream()

    # the denominator: a plain page-locked host -> device copy, 256 MiB, best of 5
    src = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
    dst = torch.empty(src.numel(), dtype=torch.uint8, device="cuda")
    best = float("inf")
    for i in range(6):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        if i:
            best = min(best, a.elapsed_time(b))
    h2d_peak = src.numel() / (best / 1000.0) / 1e9
    del src, dst

    for w in range(args.warmup):
        mf.step(toks[w % G])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    st0, rep0, l0 = cache.stats(), mf.steps, bv.moe_launch_count()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    fetched = []
    clocks = ClockSampler(local)
    clocks.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        mf.step(toks[(args.warmup + i) % G], evs[i])
        fetched.append(mf.last["n_fetched"])
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = max_over_ranks(start.elapsed_time(end))
    st1, rep1 = cache.stats(), mf.steps
    launches = (rep1 - rep0) * graph_kernels + (bv.moe_launch_count() - l0)
    step_fetch_ms = sum(a.elapsed_time(b) for (a, b), n in zip(evs, fetched) if n > 0)

    # The fetch alone (the roofline entry): 32 fetches of two experts that are
    # not resident, each enqueued while the stream is held busy (a sleep
    # kernel), so that the span between the events is the copies and the
    # table write, not the host's enqueue.
    fb0, fetch_ms = cache.stats()["bytes_fetched"], 0.0
    for i in range(32):
        cold = [e for e in range(s.E) if cache.slot_of(e) < 0][:2]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(200_000)
        a.record(stream)
        cache.fetch(cold)
        b.record(stream)
        torch.cuda.synchronize()
        fetch_ms += a.elapsed_time(b)
    fetch_bytes = cache.stats()["bytes_fetched"] - fb0

    # end to end: tokens from page-locked host memory, outputs back to it
    host_in = toks.cpu().pin_memory()
    host_out = torch.empty(args.steps, T, s.H, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        out = mf.step(host_in[(args.warmup + args.steps + i) % G])
        host_out[i].copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1))
    if world > 1:
        torch.distributed.destroy_process_group()
    named = st1["hits"] - st0["hits"] + st1["misses"] - st0["misses"] + st1["unplaced"] - st0["unplaced"]
    return dict(ms_total=ms_total, e2e_ms=e2e_ms, clocks=clk, launches=launches, h2d_peak=h2d_peak,
                fetch_ms=fetch_ms, fetch_bytes=fetch_bytes, step_fetch_ms=step_fetch_ms,
                step_fetch_bytes=st1["bytes_fetched"] - st0["bytes_fetched"], graph_kernels=graph_kernels,
                cache={"slots": wl["slots"], "hits": st1["hits"] - st0["hits"],
                       "misses": st1["misses"] - st0["misses"], "unplaced": st1["unplaced"] - st0["unplaced"],
                       "miss_rate": (st1["misses"] - st0["misses"]) / max(named, 1),
                       "steps_with_a_miss": sum(1 for n in fetched if n > 0)})


def run_tandem(args, wl, world, rank, local):
    """The decode step with the GPU holding only the wl["gpu_resident"] most
    routed experts and the host's cores computing the pairs of the others,
    overlapped with the GPU's call (TandemForward)."""
    import torch
    import bit_vq_routed_gb300 as bv

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    layer = make_layers(wl)[0]
    s = layer.spec
    T, G = wl["T"], wl["pool"]
    res = np.zeros(s.E, bool)
    res[ms.most_popular(layer, wl["gpu_resident"])] = True
    dev, keep = bv.upload_layer(s.H, s.I, s.E, s.k, T, layer.codebook, layer.w_router, layer.bias,
                                lambda e: (lambda ex: (ex.fmt, ex.codes, ex.scales))(layer.expert(e, cache=False)),
                                s.renormalize, np.nonzero(res)[0])
    hx = bv.HostExperts(s.E)
    host_bytes = 0
    for e in np.nonzero(~res)[0]:
        ex = layer.expert(int(e), cache=False)
        fmt, pc, ps = bv.host_pack_expert(ex.fmt, ex.codes, ex.scales)
        hx.set(int(e), fmt, pc, ps)
        host_bytes += sum(a.nbytes for a in pc) + sum(a.nbytes for a in ps)
    # one host core left to the CUDA driver's threads and this thread's other
    # work (16 Grace cores: 15 threads measured 16.7 K layer-tokens/s, 16
    # threads 15.1-15.6 K, 12 threads 14.8 K)
    pool = bv.CpuPool(max(1, (os.cpu_count() or 2) - 1))
    step = bv.TandemForward(dev, pool, hx, T)
    toks = torch.from_numpy(token_pool(wl, 0).view(np.int16)).view(torch.bfloat16).pin_memory()  # [G, T, H]
    stream = torch.cuda.current_stream()
    for w in range(args.warmup):
        step.step(toks[w % G])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    cpu_s, cpu_pairs, cpu_bytes = [], [], []
    clocks = ClockSampler(local)
    clocks.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        sl = (args.warmup + i) % G
        step.step(toks[sl], evs[i])
        cpu_s.append(step.last["cpu_s"])
        cpu_pairs.append(step.last["cpu_pairs"])
        ids = step.ids_host.numpy()
        miss = np.unique(ids[~res[ids]])
        cpu_bytes.append(sum(VQ2_EXPERT_BYTES if layer.formats[e] == ms.FMT_VQ2 else FP4_EXPERT_BYTES for e in miss))
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = max_over_ranks(start.elapsed_time(end))
    gpu_ms = [a.elapsed_time(b) for a, b in evs]
    # the same steps' GPU expert bytes (resident experts touched)
    gpu_bytes = []
    for i in range(args.steps):
        dev.route(toks[(args.warmup + i) % G].cuda())
        ids = dev.ids[:T].cpu().numpy()
        hit = np.unique(ids[res[ids]])
        gpu_bytes.append(sum(VQ2_EXPERT_BYTES if layer.formats[e] == ms.FMT_VQ2 else FP4_EXPERT_BYTES for e in hit))
    pool_threads = pool.threads
    launches = args.steps * step.kernels_per_step
    pool.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return dict(ms_total=ms_total, gpu_ms=gpu_ms, cpu_s=cpu_s, cpu_pairs=cpu_pairs, cpu_bytes=cpu_bytes,
                gpu_bytes=gpu_bytes, clocks=clk, threads=pool_threads, host_bytes=host_bytes, launches=launches)


def tandem_line(args, wl, r, world, config):
    T = wl["T"]
    ms_step = r["ms_total"] / args.steps
    hbm, _, peak_src = measured_peaks()
    gpu_ms = float(np.mean(r["gpu_ms"]))
    achieved = float(np.mean(r["gpu_bytes"])) / (gpu_ms / 1000.0) / 1e9
    cpu_ms = 1000.0 * float(np.mean(r["cpu_s"]))
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)",
            "kernel": "the GPU's expert graph (moe_vq2_expert_ffn over the 96 resident experts + moe_combine), "
                      "timed with events around its replay while the host computes the remainder",
            "algorithmic_bytes_per_launch": float(np.mean(r["gpu_bytes"])), "avg_launch_ms": gpu_ms,
            "traffic": None, "traffic_source": "no ncu capture of this workload"}
    if args.no_cpu:
        tps, cores, what = None, None, "skipped (--no-cpu)"
    else:
        tps, cores, what, _, _ = oracle_time(wl, make_layers(wl), budget_s=args.cpu_budget, max_steps=4)
    return {
        "metric": METRIC, "value": job_rate(T, world, ms_step), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16*f16->f32 (bf16 activations); host fp32",
        "data": "synthetic (seeded; random weights, no trained checkpoint)", "config": config,
        "roofline": roof,
        "host_experts": {"threads": r["threads"], "cpu_ms_per_step": cpu_ms,
                         "pairs_per_step": float(np.mean(r["cpu_pairs"])),
                         "code_bytes_per_step": float(np.mean(r["cpu_bytes"])),
                         "gbs": float(np.mean(r["cpu_bytes"])) / (cpu_ms / 1000.0) / 1e9 if cpu_ms > 0 else None,
                         "host_base_bytes": r["host_bytes"],
                         "overlap": "the GPU's expert graph is enqueued before the host computes; the step waits "
                                    "for both, then adds the remainder on the device"},
        "cpu_baseline": {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": what,
                         "cpu": cpu_model()},
        "e2e": {"value": job_rate(T, world, ms_step), "unit": UNIT, "h2d_bytes_per_step": T * 4096 * 2 + T * 4096 * 4,
                "d2h_bytes_per_step": T * 8 * 8,
                "how": "every step copies its tokens from page-locked host memory and reads the routed ids and "
                       "weights back, inside the timed region (the step's output stays on the device)"},
        "gpu_launches": r["launches"],
        "launch": "routing graph, read-back of ids/weights, expert graph (GPU) and moe_cpu_expert_ffn (host) "
                  "at the same time, then the remainder's copy and moe_accumulate",
        "clocks": r["clocks"],
    }


def fetch_line(args, wl, r, world, config):
    T = wl["T"]
    ms_step = r["ms_total"] / args.steps
    achieved = r["fetch_bytes"] / (r["fetch_ms"] / 1000.0) / 1e9 if r["fetch_ms"] > 0 else None
    roof = {"bound": "h2d", "achieved": achieved, "peak": r["h2d_peak"], "unit": "GB/s",
            "frac": None if achieved is None else achieved / r["h2d_peak"],
            "peak_source": "plain page-locked host -> device copy of 256 MiB, measured in the same run (best of 5)",
            "traffic": None, "traffic_source": "no ncu capture (host -> device copies)",
            "kernel": "moe_expert_cache_fetch: one cudaMemcpyAsync per expert (a host block in the slot's layout) "
                      "and one slot-table write kernel per fetch; 32 fetches of two experts, each timed on the "
                      "stream while a sleep kernel holds it during the host's enqueue",
            "algorithmic_bytes": r["fetch_bytes"], "fetch_ms": r["fetch_ms"],
            "in_step": {"fetch_ms": r["step_fetch_ms"], "bytes": r["step_fetch_bytes"],
                        "gbs_with_host_enqueue": (r["step_fetch_bytes"] / (r["step_fetch_ms"] / 1000.0) / 1e9
                                                  if r["step_fetch_ms"] > 0 else None)}}
    if args.no_cpu:
        tps, cores, what = None, None, "skipped (--no-cpu)"
    else:
        tps, cores, what, _, _ = oracle_time(wl, make_layers(wl), budget_s=args.cpu_budget, max_steps=4)
    return {
        "metric": METRIC, "value": job_rate(T, world, ms_step), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16*f16->f32 (bf16 activations)",
        "data": "synthetic (seeded; random weights, no trained checkpoint)", "config": config,
        "roofline": roof, "cache": r["cache"],
        "cpu_baseline": {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": what,
                         "cpu": cpu_model()},
        "e2e": {"value": job_rate(T, world, r["e2e_ms"] / args.steps), "unit": UNIT,
                "h2d_bytes_per_step": T * 4096 * 2, "d2h_bytes_per_step": T * 4096 * 4},
        "gpu_launches": r["launches"],
        "launch": ("two CUDA graphs per step: the routing, then (after the routed ids are read back and the "
                   "misses fetched) the expert FFN and combine"),
        "clocks": r["clocks"],
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode_b1", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count (profiling)")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's tokens per step (profiling)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--eager", dest="graph", action="store_false",
                    help="launch every call from Python instead of replaying one CUDA graph per step")
    args = ap.parse_args()
    world, rank, local = dist_env()
    wl = dict(WORKLOADS[args.workload])
    if args.layers:
        wl["layers"] = args.layers
    if args.tokens:
        wl["T"] = args.tokens
    config = {"workload": wl["desc"], "name": args.workload, "tokens_per_step": wl["T"],
              "layers_per_step": wl["layers"],
              "l2": f"inputs larger than L2: each step touches its layers' routed experts "
                    f"(>= {wl['layers'] * 8 * VQ2_EXPERT_BYTES / 1e6:.0f} MB vs 129 MB L2), tokens rotate "
                    f"over a pool of {wl['pool']} batches per layer"}
    T, nL = wl["T"], wl["layers"]

    if args.impl == "reference":
        if rank != 0:
            return
        layers = make_layers(wl)
        max_steps = args.warmup + args.steps
        tps, cores, what, done, el = oracle_time(wl, layers, budget_s=max(5.0, args.cpu_budget), max_steps=max_steps)
        line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": UNIT, "n_gpus": args.gpus,
                "steps": done, "warmup": 0, "ms_per_step": 1000 * el / max(done, 1),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded; random weights, no trained checkpoint)", "config": config,
                "cpu_baseline": {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": what,
                                 "cpu": cpu_model()},
                "e2e": {"value": tps, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if "gpu_resident" in wl:
        r = run_tandem(args, wl, world, rank, local)
        if rank == 0:
            config["l2"] = f"tokens rotate over a pool of {wl['pool']} batches; the host computes from its own memory"
            print(json.dumps(tandem_line(args, wl, r, world, config)))
        return
    if "slots" in wl:
        r = run_fetch(args, wl, world, rank, local)
        if rank == 0:
            config["l2"] = "every step's experts come from the cache's slots or host memory; tokens rotate over " \
                           f"a pool of {wl['pool']}"
            print(json.dumps(fetch_line(args, wl, r, world, config)))
        return
    r = run_gpu(args, wl, world, rank, local)
    if rank != 0:
        return
    hbm, bf16, peak_src = measured_peaks()
    traffic, traffic_src = measured_traffic(args.workload)  # (per expert-FFN call, like achieved)
    kernels = ("the two self-scheduling table kernels (FC1, FC2)" if T == 1 else
               "schedule, gather, table, mma.sync and tcgen05 kernels for FC1 and FC2")
    ms_step = r["ms_total"] / args.steps
    value = job_rate(T * nL, world, ms_step)
    ffn_avg_ms = float(np.mean(r["ffn_ms"]))
    bytes_avg = float(np.mean(r["code_bytes"]))
    achieved = bytes_avg / (ffn_avg_ms / 1000.0) / 1e9
    codes_gbs = float(np.mean(r["codes_only"])) / (ffn_avg_ms / 1000.0) / 1e9
    # the prefill chunk is a dense contraction: its roofline is the tensor pipe
    # (fp16 operands; the measured bf16 GEMM rate, fp16 being the same nominal
    # dense rate on this part)
    flop = T * 8 * FFN_FLOP_PER_PAIR
    tensor = T > 64
    if tensor:
        hbm_line = {"achieved_gbs": achieved, "peak_gbs": hbm, "algorithmic_bytes_per_launch": bytes_avg}
        roof = {"bound": "tensor", "achieved": flop / (ffn_avg_ms / 1000.0) / 1e12, "peak": bf16,
                "unit": "TFLOP/s", "frac": flop / (ffn_avg_ms / 1000.0) / 1e12 / bf16,
                "peak_source": f"{peak_src} bf16_tflops (cuBLAS bf16 GEMM, burst: the call is timed alone; "
                               "fp16 has the same nominal dense rate)",
                "algorithmic_flop_per_launch": flop, "hbm": hbm_line}
    else:
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy, burst: the call is timed alone)",
                "algorithmic_bytes_per_launch": bytes_avg}
    roof.update({"kernel": f"moe_vq2_expert_ffn: {kernels}", "traffic": traffic, "traffic_source": traffic_src,
                 "avg_launch_ms": ffn_avg_ms, "codes_only_gbs": codes_gbs})
    e2e_value = job_rate(T * nL, world, r["e2e_ms"] / r["e2e_steps"])
    if args.no_cpu:
        tps, cores, what = None, None, "skipped (--no-cpu)"
    else:
        layers = make_layers(wl)
        tps, cores, what, done, el = oracle_time(wl, layers, budget_s=args.cpu_budget, max_steps=4)
    single = None
    if not args.no_cpu and T == 1:  # the oracle on one core too, one step
        s_tps, s_cores, s_what, _, _ = oracle_time(wl, layers[:1], budget_s=1.0, max_steps=1, threads=1)
        single = {"value": s_tps, "unit": UNIT, "cores": s_cores, "sample": s_what}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16*f16->f32 (bf16 activations)",
        "data": "synthetic (seeded; random weights, no trained checkpoint)", "config": config,
        "roofline": roof,
        "other_bytes_per_layer": {"router_weights": 256 * 4096 * 2, "activations": T * 4096 * 2,
                                  "per_pair_outputs": T * 8 * 4096 * 4 * 2, "outputs": T * 4096 * 4},
        "cpu_baseline": {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": what,
                         "cpu": cpu_model(), "single_core": single},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": T * 4096 * 2 * nL,
                "d2h_bytes_per_step": T * 4096 * 4 * nL,
                "how": ("PipelinedSteps: the layers of a step as one CUDA graph over double-buffered device "
                        "tokens and outputs; each step's page-locked host -> device copy of every layer's tokens "
                        "and device -> host copy of their outputs run on two copy streams, overlapping the "
                        "neighbouring steps' layers")
                if args.graph else "eager calls with a copy in and out per layer"},
        "gpu_launches": r["launches"],
        "launch": ("one CUDA graph per step (every layer's route, expert FFN and combine; programmatic "
                   "dependent launch between kernels); the expert-FFN time is a graph of the step's FFN calls "
                   "back to back, divided by the calls") if args.graph else "eager",
        "clocks": r["clocks"],
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
