r"""One routed-expert MoE layer on the device: the buffers it needs and the
sequence of library calls of one forward pass.

    logits = router(x)                  moe_router_logits  \
    ids, w = top-k softmax(logits)      moe_route_topk      > moe_route (one kernel
    permutation by expert               moe_permute        /  for small batches)
    y per (token, expert) pair          moe_vq2_expert_ffn (per-pair mode)  \ (or both in one call:
    out = sum_j w * y                   moe_combine                         /  moe_vq2_expert_ffn_combine)

All five run as library kernels on one stream, with no host synchronisation,
so a forward pass can be captured in a CUDA graph.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

from . import (MOE_FMT_FP4, MOE_FMT_VQ2, MOE_FUSED_SCATTER, MOE_PER_PAIR, SlotTable, moe_combine,
               moe_fp4_pack, moe_permute, moe_route, moe_route_topk, moe_route_workspace_size, moe_router_logits,
               moe_vq2_expert_ffn, moe_vq2_expert_ffn_combine, moe_vq2_expert_ffn_workspace_size)


def _dev(a, dtype=None, device="cuda"):
    if isinstance(a, torch.Tensor):
        return a.to(device=device)
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device=device)


def upload_expert(fmt: int, codes: Sequence, scales: Sequence, stream=None, device="cuda"):
    """Copies one expert's logical (row-major) codes and scales to the device
    and packs them (moe_vq2_pack / moe_fp4_pack).  Returns (packed codes,
    packed scales), three tensors each: gate, up, down."""
    from . import moe_vq2_pack
    pc, ps = [], []
    for m in range(3):
        c = _dev(codes[m], torch.uint8, device)
        if fmt == MOE_FMT_VQ2:
            s = _dev(scales[m], torch.float16, device)
            c2, s2 = torch.empty_like(c), torch.empty_like(s)
            moe_vq2_pack(c, s, c2, s2, stream)
        else:
            s = _dev(scales[m], torch.uint8, device)
            c2, s2 = torch.empty_like(c), torch.empty_like(s)
            moe_fp4_pack(c, s, c2, s2, stream)
        pc.append(c2)
        ps.append(s2)
    return pc, ps


class MoELayer:
    """Device buffers and the call sequence of one layer.  table_experts: the
    slot table's entries (E when None; 2E for the confidence gate, whose
    entries E..2E-1 hold FP4 weights)."""

    def __init__(self, H: int, I: int, E: int, k: int, T_max: int, codebook, w_router, bias=None,
                 renormalize: int = 1, device="cuda", table_experts: Optional[int] = None):
        self.H, self.I, self.E, self.k, self.T_max = H, I, E, k, T_max
        self.table_experts = E if table_experts is None else table_experts
        self.renormalize = renormalize
        self.codebook = _dev(codebook, torch.float16, device).contiguous()
        self.w_router = _dev(w_router, torch.bfloat16, device).contiguous()
        self.bias = None if bias is None else _dev(bias, torch.float32, device).contiguous()
        self.table = SlotTable(self.table_experts, H, I, self.codebook)
        P = T_max * k
        f32, i32 = torch.float32, torch.int32
        self.logits = torch.empty(T_max, E, dtype=f32, device=device)
        self.ids = torch.empty(T_max, k, dtype=i32, device=device)
        self.weights = torch.empty(T_max, k, dtype=f32, device=device)
        self.offsets = torch.empty(self.table_experts + 1, dtype=i32, device=device)
        self.sorted_pair = torch.empty(P, dtype=i32, device=device)
        self.pair_to_sorted = torch.empty(P, dtype=i32, device=device)
        self.pair_status = torch.empty(P, dtype=torch.uint8, device=device)
        self.ypair = torch.empty(P, H, dtype=f32, device=device)
        self.out = torch.empty(T_max, H, dtype=f32, device=device)
        self.ws = torch.empty(moe_vq2_expert_ffn_workspace_size(T_max, k, self.table_experts, H, I), dtype=torch.uint8,
                              device=device)
        # (zero-filled once; moe_route leaves its counter at zero)
        self.route_ws = torch.zeros(moe_route_workspace_size(T_max, k, E), dtype=torch.uint8, device=device)

    def set_expert(self, e: int, fmt: int, packed_codes, packed_scales, stream=None):
        self.table.set(e, fmt, packed_codes, packed_scales, stream)

    def evict(self, e: int, stream=None):
        self.table.evict(e, stream)

    def route(self, x, stream=None):
        T = x.shape[0]
        moe_route(x, self.w_router, self.bias, self.k, self.renormalize, self.logits[:T], self.ids[:T],
                  self.weights[:T], self.offsets, self.sorted_pair[:T * self.k], self.pair_to_sorted[:T * self.k],
                  self.route_ws, stream)

    def route_stepwise(self, x, stream=None):
        """The same routing as route() through the three separate calls."""
        T = x.shape[0]
        moe_router_logits(x, self.w_router, self.bias, self.logits[:T], stream)
        moe_route_topk(self.logits[:T], self.k, self.renormalize, self.ids[:T], self.weights[:T], stream)
        moe_permute(self.ids[:T], self.E, self.offsets, self.sorted_pair[:T * self.k],
                    self.pair_to_sorted[:T * self.k], None, stream)

    def experts(self, x, mode=MOE_PER_PAIR, out=None, stream=None):
        T = x.shape[0]
        P = T * self.k
        dst = self.ypair[:P] if mode == MOE_PER_PAIR else out
        moe_vq2_expert_ffn(self.table, x, self.offsets, self.sorted_pair[:P], self.weights[:T], self.k, mode,
                           dst, self.pair_status[:P], self.ws, stream)

    def experts_combine(self, x, out, out_bf16=None, stream=None):
        """experts() in per-pair mode and the combine into out (fp32 [T, H])
        and/or out_bf16, in one call (moe_vq2_expert_ffn_combine)."""
        T = x.shape[0]
        P = T * self.k
        moe_vq2_expert_ffn_combine(self.table, x, self.offsets, self.sorted_pair[:P], self.pair_to_sorted[:P],
                                   self.weights[:T], self.k, self.ypair[:P], self.pair_status[:P], out, out_bf16,
                                   self.ws, stream)

    def forward(self, x, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """x: bf16 [T, H] on the device -> fp32 [T, H] (a view of self.out
        unless out is given)."""
        T = x.shape[0]
        if T > self.T_max:
            raise ValueError(f"T={T} above T_max={self.T_max}")
        o = self.out[:T] if out is None else out
        self.route(x, stream)
        self.experts(x, MOE_PER_PAIR, None, stream)
        moe_combine(self.ypair[:T * self.k], self.pair_to_sorted[:T * self.k], self.weights[:T],
                    self.pair_status[:T * self.k], self.k, o, None, stream)
        return o


class GraphedForward:
    """MoELayer.forward for a fixed batch of T tokens captured in a CUDA graph
    (all of its kernels, no host work per step): write the tokens into
    ``self.x``, call ``replay()``, read ``self.out``."""

    def __init__(self, layer: MoELayer, T: int, device="cuda"):
        self.layer = layer
        self.x = torch.zeros(T, layer.H, dtype=torch.bfloat16, device=device)
        layer.forward(self.x)  # first eager call: kernel attributes are set outside capture
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.out = layer.forward(self.x)

    def replay(self):
        self.graph.replay()
        return self.out


class GraphedStep:
    """One step over several layers as one CUDA graph, inputs and outputs
    included: the graph copies the step's tokens from page-locked host memory
    (``host_in``: bf16 [L, T, H], one copy), runs every layer's forward on its
    own slice, and copies the fp32 outputs back (``host_out``: [L, T, H], one
    copy).  Write the next tokens into ``host_in`` (or capture one
    GraphedStep per input buffer), call ``replay()``, and read ``host_out``
    after synchronising the stream."""

    def __init__(self, layers: Sequence[MoELayer], host_in: torch.Tensor, host_out: torch.Tensor, device="cuda"):
        if not (host_in.is_pinned() and host_out.is_pinned()):
            raise ValueError("host_in and host_out must be page-locked")
        L, T, H = host_in.shape
        if L != len(layers) or tuple(host_out.shape) != (L, T, H):
            raise ValueError("host_in / host_out must be [layers, T, H]")
        self.layers, self.host_in, self.host_out = list(layers), host_in, host_out
        self.x = torch.empty(L, T, H, dtype=torch.bfloat16, device=device)
        self.out = torch.empty(L, T, H, dtype=torch.float32, device=device)
        self._run()  # first eager call: kernel attributes are set outside capture
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._run()

    def _run(self):
        self.x.copy_(self.host_in, non_blocking=True)
        for i, layer in enumerate(self.layers):
            layer.forward(self.x[i], out=self.out[i])
        self.host_out.copy_(self.out, non_blocking=True)

    def replay(self):
        self.graph.replay()


class PipelinedSteps:
    """Steps over several layers with the host copies overlapping the layers
    of the neighbouring steps: the layers run as one CUDA graph per device
    buffer pair (tokens bf16 [L, T, H], outputs fp32 [L, T, H], two pairs),
    a step's tokens are copied in from page-locked host memory on one stream
    and its outputs copied out on another, ordered by events.

    ``step(host_in, host_out)`` enqueues one step: the copy of ``host_in``
    (pinned bf16 [L, T, H]) into the free buffer, the layers on the current
    stream once that copy is done, and the copy of the outputs into
    ``host_out`` (pinned fp32 [L, T, H]) once they are done.  The copy of
    step s + 1 in runs while step s computes, and the copy of step s out
    while step s + 1 computes.  ``join()`` makes the current stream wait for
    every enqueued copy; synchronise it before reading ``host_out``.  The
    host buffers of a step must stay unchanged until its copies are done."""

    def __init__(self, layers: Sequence[MoELayer], T: int, device="cuda"):
        self.layers = list(layers)
        L, H = len(self.layers), self.layers[0].H
        self.x = [torch.zeros(L, T, H, dtype=torch.bfloat16, device=device) for _ in range(2)]
        self.out = [torch.empty(L, T, H, dtype=torch.float32, device=device) for _ in range(2)]
        self.copy_in = torch.cuda.Stream(device=device)
        self.copy_out = torch.cuda.Stream(device=device)
        # per buffer: tokens copied in, layers done, outputs copied out
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_done = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]
        self.n = 0
        self._run(0)  # first eager call: kernel attributes are set outside capture
        torch.cuda.synchronize()
        self.graphs = []
        for b in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._run(b)
            self.graphs.append(g)

    def _run(self, b: int):
        for i, layer in enumerate(self.layers):
            layer.forward(self.x[b][i], out=self.out[b][i])

    def step(self, host_in: torch.Tensor, host_out: torch.Tensor):
        b = self.n & 1
        cur = torch.cuda.current_stream()
        if self.n == 0:  # the copies start after the work enqueued before the first step
            self.ev_first = torch.cuda.Event()
            self.ev_first.record(cur)
        self.n += 1
        if self.used[b]:  # the buffer's previous step is done with its tokens
            self.copy_in.wait_event(self.ev_done[b])
        else:
            self.copy_in.wait_event(self.ev_first)
        with torch.cuda.stream(self.copy_in):
            self.x[b].copy_(host_in, non_blocking=True)
            self.ev_in[b].record(self.copy_in)
        cur.wait_event(self.ev_in[b])
        if self.used[b]:  # and the outputs of its previous step are copied out
            cur.wait_event(self.ev_out[b])
        self.graphs[b].replay()
        self.ev_done[b].record(cur)
        self.copy_out.wait_event(self.ev_done[b])
        with torch.cuda.stream(self.copy_out):
            host_out.copy_(self.out[b], non_blocking=True)
            self.ev_out[b].record(self.copy_out)
        self.used[b] = True

    def join(self):
        cur = torch.cuda.current_stream()
        cur.wait_stream(self.copy_in)
        cur.wait_stream(self.copy_out)


def host_expert(fmt: int, codes: Sequence, scales: Sequence, stream=None, device="cuda"):
    """Packs one expert on the device (upload_expert) and returns page-locked
    host copies of the packed buffers (codes[3], scales[3]): the host-resident
    base that an ExpertCache fetches from."""
    pc, ps = upload_expert(fmt, codes, scales, stream, device)
    torch.cuda.synchronize()
    return [c.cpu().pin_memory() for c in pc], [s.cpu().pin_memory() for s in ps]


def slot_layout(H: int, I: int, fmt: int):
    """(offset, bytes) of the six packed buffers of an expert in a cache slot
    or host image: codes of gate, up, down, then their scales, each offset
    rounded up to 256 bytes (the layout moe_expert_cache_set_host_image
    reads)."""
    out, off = [], 0
    for b in range(6):
        rows, K = (H, I) if b % 3 == 2 else (I, H)
        n = (rows * K // 4 if b < 3 else rows * K // 128 * 2) if fmt == MOE_FMT_VQ2 else \
            (rows * K // 2 if b < 3 else rows * K // 32)
        out.append((off, n))
        off += (n + 255) // 256 * 256
    return out, off


def host_expert_image(fmt: int, codes: Sequence, scales: Sequence, stream=None, device="cuda"):
    """Packs one expert on the device straight into a block in the slot's
    layout and returns a page-locked host copy of it (one uint8 tensor): the
    host-resident base that an ExpertCache fetches with one copy."""
    from . import moe_vq2_pack
    I, H4 = np.asarray(codes[0]).shape
    H = H4 * (4 if fmt == MOE_FMT_VQ2 else 2)
    lay, total = slot_layout(H, I, fmt)
    img = torch.zeros(total, dtype=torch.uint8, device=device)
    for m in range(3):
        (oc, nc), (osc, ns) = lay[m], lay[3 + m]
        c = _dev(codes[m], torch.uint8, device)
        pc = img[oc:oc + nc].view(c.shape)
        if fmt == MOE_FMT_VQ2:
            s = _dev(scales[m], torch.float16, device)
            moe_vq2_pack(c, s, pc, img[osc:osc + ns].view(torch.float16).view(s.shape), stream)
        else:
            s = _dev(scales[m], torch.uint8, device)
            moe_fp4_pack(c, s, pc, img[osc:osc + ns].view(s.shape), stream)
    torch.cuda.synchronize()
    return img.cpu().pin_memory()


class MissFetchForward:
    """The forward of a layer whose experts live in host memory, with the GPU
    as an expert cache (vLLM-Moet page, "2-bit experts on vLLM v0.24.0",
    "Experts beyond VRAM": a miss is fetched and the step's graph replayed).

    The step's work is captured as two CUDA graphs, split at the routing:
    each step replays the routing graph, reads the routed ids back (one
    device-to-host copy and one wait), names them to the cache (routing
    counts; misses are copied in) and then replays the expert graph (expert
    FFN and combine) once, over experts that are all resident when they fit
    in the cache's slots.  Its output is then bit-identical to a forward with
    every expert resident.  The expert graph is captured again when a fetch
    changes whether the table holds FP4 experts (the expert-FFN call picks
    its kernels by that on the host)."""

    def __init__(self, layer: MoELayer, cache, T: int, device="cuda"):
        self.layer, self.cache, self.T = layer, cache, T
        self.x = torch.zeros(T, layer.H, dtype=torch.bfloat16, device=device)
        self.out = layer.out[:T]
        self.ids_host = torch.empty(T, layer.k, dtype=torch.int32).pin_memory()
        layer.forward(self.x)  # first eager call: kernel attributes are set outside capture
        torch.cuda.synchronize()
        self.g_route = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_route):
            layer.route(self.x)
        self._capture_experts()
        self.steps = 0
        self.fetch_steps = 0
        self.captures = 1
        self.last = None

    def _capture_experts(self):
        T, k = self.T, self.layer.k
        self.g_ffn = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_ffn):
            self.layer.experts(self.x, MOE_PER_PAIR)
            moe_combine(self.layer.ypair[:T * k], self.layer.pair_to_sorted[:T * k], self.layer.weights[:T],
                        self.layer.pair_status[:T * k], k, self.out)

    def step(self, x=None, fetch_events=None) -> torch.Tensor:
        """x: bf16 [T, H] (copied into the graphs' input), or None when
        self.x already holds the tokens.  Returns the fp32 [T, H] output.
        fetch_events: optional pair of CUDA events recorded on the stream
        around the fetch; self.last holds the fetch's result."""
        if x is not None:
            self.x.copy_(x, non_blocking=True)
        self.g_route.replay()
        self.ids_host.copy_(self.layer.ids[:self.T], non_blocking=True)
        torch.cuda.current_stream().synchronize()
        if fetch_events is not None:
            fetch_events[0].record()
        r = self.cache.fetch(self.ids_host.numpy())
        if fetch_events is not None:
            fetch_events[1].record()
        self.last = r
        if r["recapture"]:
            self._capture_experts()
            self.captures += 1
        self.g_ffn.replay()
        self.steps += 1
        self.fetch_steps += 1 if r["n_fetched"] else 0
        return self.out


class TandemForward:
    """The forward of a layer whose GPU slot table holds only some experts,
    with the host's cores computing the pairs of the others at the same time
    (Tandem-vLLM page, "How it works": experts that miss the GPU cache are
    computed by the CPU in parallel with the GPU, nothing skipped or
    substituted).

    Each step: the tokens are copied in and the routing graph replays; the
    routed ids and weights are read back (one device-to-host copy and one
    wait); the expert graph (the GPU's expert FFN over its resident experts,
    then the combine of their pairs: the partial output) is enqueued; while
    it runs, moe_cpu_expert_ffn computes the remainder over the pairs of the
    other experts on the host, from host copies of their packed weights
    (host_experts); the remainder is copied in and added (moe_accumulate).
    The GPU reports the pairs it skipped in pair_status; the host decides the
    same set beforehand from the table's host mirror (moe_slot_table_resident).
    """

    def __init__(self, layer: MoELayer, pool, host_experts, T: int, device="cuda"):
        from . import moe_slot_table_resident
        self.layer, self.pool, self.host_experts, self.T = layer, pool, host_experts, T
        H, k = layer.H, layer.k
        self.x = torch.zeros(T, H, dtype=torch.bfloat16, device=device)
        self.out = layer.out[:T]
        self.ids_host = torch.empty(T, k, dtype=torch.int32).pin_memory()
        self.w_host = torch.empty(T, k, dtype=torch.float32).pin_memory()
        self.rem_host = torch.empty(T, H, dtype=torch.float32).pin_memory()
        self.rem_dev = torch.empty(T, H, dtype=torch.float32, device=device)
        self.codebook_host = layer.codebook.cpu().view(torch.int16).numpy().view(np.uint16)
        self.resident = np.array([moe_slot_table_resident(layer.table, e) for e in range(layer.E)], dtype=bool)
        from . import moe_launch_count
        layer.forward(self.x)  # first eager call: kernel attributes are set outside capture
        torch.cuda.synchronize()
        n0 = moe_launch_count()
        self.g_route = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_route):
            layer.route(self.x)
        self.g_ffn = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_ffn):
            layer.experts(self.x, MOE_PER_PAIR)
            moe_combine(layer.ypair[:T * k], layer.pair_to_sorted[:T * k], layer.weights[:T],
                        layer.pair_status[:T * k], k, self.out)
        # library kernels per step: the two graphs' nodes and moe_accumulate
        self.kernels_per_step = moe_launch_count() - n0 + 1
        self.last = {}

    def step(self, x_host: torch.Tensor, events=None) -> torch.Tensor:
        """x_host: bf16 [T, H] in page-locked host memory.  Returns the fp32
        [T, H] output on the device (enqueued: synchronise before reading).
        events: optional (gpu_start, gpu_end) CUDA events recorded around the
        expert graph; self.last holds the pairs and the host seconds of the
        CPU part."""
        import time
        from . import moe_accumulate, moe_cpu_expert_ffn
        L, T, k = self.layer, self.T, self.layer.k
        self.x.copy_(x_host, non_blocking=True)
        self.g_route.replay()
        self.ids_host.copy_(L.ids[:T], non_blocking=True)
        self.w_host.copy_(L.weights[:T], non_blocking=True)
        torch.cuda.current_stream().synchronize()
        ids = self.ids_host.numpy()
        status = self.resident[ids].astype(np.uint8).ravel()
        if events is not None:
            events[0].record()
        self.g_ffn.replay()  # the GPU's partial output, running while the host computes
        if events is not None:
            events[1].record()
        t0 = time.perf_counter()
        moe_cpu_expert_ffn(self.pool, L.H, L.I, self.codebook_host, self.host_experts,
                           x_host.view(torch.int16).numpy().view(np.uint16), ids, self.w_host.numpy(), status, k,
                           self.rem_host.numpy())
        cpu_s = time.perf_counter() - t0
        self.rem_dev.copy_(self.rem_host, non_blocking=True)
        moe_accumulate(self.out, self.rem_dev)
        self.last = dict(cpu_pairs=int((status == 0).sum()), cpu_s=cpu_s)
        return self.out


class GatedForward:
    """The forward with the confidence gate over an FP4 delta cache (the
    vLLM-Moet page, "2-bit experts on vLLM v0.24.0": a delta cache and a
    confidence gate bring FP4 back where it matters; its bench table: "FP4
    delta (auto) + confidence gate tau=0.60").  The layer's slot table has
    2E entries: the 2-bit base of expert e at e, its FP4 weights at E + e
    while held.  A step: the routing; moe_confidence_gate (pairs with router
    weight >= tau whose FP4 entry is set go to entry E + e); the permutation
    over 2E entries; the expert FFN; the combine.

    With cache (an ExpertCache over the same table whose host images are the
    experts' FP4 weights, named E + e), the step is split at the routing:
    the routed ids and weights are read back, the cache fetches the FP4
    entries of the pairs the gate wants (routing counts decide the
    evictions), then the rest runs.  Without it, the FP4 entries set on the
    table are used as they are and the whole step is one CUDA graph."""

    def __init__(self, layer: MoELayer, T: int, tau: float = 0.6, cache=None, device="cuda"):
        from . import moe_confidence_gate, moe_permute_workspace_size
        if layer.table_experts < 2 * layer.E:
            raise ValueError("the layer's table needs 2E entries")
        self.layer, self.T, self.tau, self.cache = layer, T, tau, cache
        E, k = layer.E, layer.k
        P = T * k
        i32 = torch.int32
        self.x = torch.zeros(T, layer.H, dtype=torch.bfloat16, device=device)
        self.out = layer.out[:T]
        self.gated = torch.empty(T, k, dtype=i32, device=device)
        self.offsets2 = torch.empty(2 * E + 1, dtype=i32, device=device)
        self.sorted2 = torch.empty(P, dtype=i32, device=device)
        self.p2s2 = torch.empty(P, dtype=i32, device=device)
        self.perm_ws = torch.empty(max(moe_permute_workspace_size(T, k, 2 * E), 16), dtype=torch.uint8,
                                   device=device)
        self.ids_host = torch.empty(T, k, dtype=i32).pin_memory()
        self.w_host = torch.empty(T, k, dtype=torch.float32).pin_memory()
        self._gate = moe_confidence_gate
        if cache is not None:
            layer.route(self.x)  # (the rest reads the routing)
        self._rest()  # first eager call: kernel attributes are set outside capture
        torch.cuda.synchronize()
        self.g_route = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_route):
            layer.route(self.x)
        self._capture_rest()
        self.last = {}

    def _rest(self):
        L, T, k, E = self.layer, self.T, self.layer.k, self.layer.E
        P = T * k
        if self.cache is None:
            L.route(self.x)
        self._gate(L.table, L.ids[:T], L.weights[:T], E, self.tau, self.gated)
        moe_permute(self.gated, 2 * E, self.offsets2, self.sorted2, self.p2s2, self.perm_ws)
        moe_vq2_expert_ffn(L.table, self.x, self.offsets2, self.sorted2, L.weights[:T], k, MOE_PER_PAIR,
                           L.ypair[:P], L.pair_status[:P], L.ws)
        moe_combine(L.ypair[:P], self.p2s2, L.weights[:T], L.pair_status[:P], k, self.out)

    def _capture_rest(self):
        self.g_rest = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_rest):
            self._rest()

    def step(self, x=None) -> torch.Tensor:
        """x: bf16 [T, H] on the device (or None when self.x holds the
        tokens).  Returns the fp32 [T, H] output (enqueued)."""
        if x is not None:
            self.x.copy_(x, non_blocking=True)
        if self.cache is None:
            self.g_rest.replay()  # (the routing is inside)
            return self.out
        L, T, E = self.layer, self.T, self.layer.E
        self.g_route.replay()
        self.ids_host.copy_(L.ids[:T], non_blocking=True)
        self.w_host.copy_(L.weights[:T], non_blocking=True)
        torch.cuda.current_stream().synchronize()
        ids, w = self.ids_host.numpy(), self.w_host.numpy()
        want = np.unique(ids[w >= self.tau]) + E
        r = self.cache.fetch(want) if want.size else dict(n_fetched=0, n_unplaced=0, recapture=False)
        if r["recapture"]:
            self._capture_rest()
        self.last = dict(wanted=int(want.size), **r)
        self.g_rest.replay()
        return self.out


def upload_layer(H, I, E, k, T_max, codebook, w_router, bias, experts, renormalize=1, resident=None,
                 stream=None, device="cuda"):
    """Builds a MoELayer and makes resident the experts in ``resident`` (all
    when None).  ``experts(e)`` returns (fmt, codes[3], scales[3]) in the
    logical layout.  Returns (layer, packed buffers by expert id)."""
    layer = MoELayer(H, I, E, k, T_max, codebook, w_router, bias, renormalize, device)
    keep = {}
    ids = range(E) if resident is None else resident
    for e in ids:
        fmt, codes, scales = experts(int(e))
        pc, ps = upload_expert(fmt, codes, scales, stream, device)
        layer.set_expert(int(e), fmt, pc, ps, stream)
        keep[int(e)] = (pc, ps)
    return layer, keep
