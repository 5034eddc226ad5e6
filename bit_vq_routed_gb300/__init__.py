"""Python binding of libmoe_vq2.so, the GB300 (sm_103a) routed-expert VQ2 MoE
layer library.  Argument marshalling only: every step of the layer runs in
the library's CUDA kernels; PyTorch provides device memory and streams.

The functions carry the names of the C ABI in ``include/moe_vq2.h`` and take
CUDA tensors (any dtype of the right element size: bf16 activations as
``torch.bfloat16``, fp16 codebook/scales as ``torch.float16``, codes and
ue8m0 scales as ``torch.uint8``).  A non-zero status raises ``MoeError``
with the library's message.  There is no CPU or PyTorch fallback: if the
shared library cannot be built or loaded, the import of the functions fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_NO_MEM = -4
MOE_ERR_WORKSPACE = -5
MOE_ERR_TIMEOUT = -6
MOE_ERR_MISMATCH = -7

MOE_FMT_VQ2 = 0
MOE_FMT_FP4 = 1
MOE_FUSED_SCATTER = 0
MOE_PER_PAIR = 1

LIB_PATH = _build.LIB


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"status {status}: {msg}")
        self.status = status


class _ExpertDesc(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int), ("codes", ctypes.c_void_p * 3), ("scales", ctypes.c_void_p * 3)]


_lib = None

EXPORTED = [
    "moe_version", "moe_last_error", "moe_vq2_pack", "moe_fp4_pack", "moe_slot_table_create",
    "moe_slot_table_set", "moe_slot_table_evict", "moe_slot_table_destroy", "moe_router_logits",
    "moe_route_topk", "moe_permute_workspace_size", "moe_permute",
    "moe_vq2_expert_ffn_workspace_size", "moe_vq2_expert_ffn", "moe_vq2_expert_ffn_noalloc", "moe_combine",
    "moe_launch_count", "moe_route_workspace_size", "moe_route", "moe_vq2_expert_ffn_combine",
    "moe_selftest", "moe_selftest_wait_timeout", "moe_expert_cache_slot_bytes", "moe_expert_cache_create", "moe_expert_cache_set_host",
    "moe_expert_cache_fetch", "moe_expert_cache_slot_of", "moe_expert_cache_stats", "moe_expert_cache_plan",
    "moe_expert_cache_destroy", "moe_expert_cache_set_host_image", "moe_cpu_pool_create", "moe_cpu_pool_threads",
    "moe_cpu_pool_destroy", "moe_cpu_expert_ffn", "moe_accumulate", "moe_slot_table_resident", "moe_vq2_pack_host",
    "moe_fp4_pack_host", "moe_confidence_gate", "moe_vq2_encoder_workspace_size", "moe_vq2_train_codebook", "moe_vq2_encode",
]


def load(path: Optional[str] = None, build_if_stale: bool = True):
    """Loads (building it first if it is missing or older than its sources)
    the shared library and declares the C signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if path is None and build_if_stale and not _build.up_to_date():
        _build.build()
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with bit_vq_routed_gb300.build.build()")
    lib = ctypes.CDLL(p)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "moe_version": ([], I),
        "moe_last_error": ([], ctypes.c_char_p),
        "moe_vq2_pack": ([P, P, I, I, P, P, P], I),
        "moe_fp4_pack": ([P, P, I, I, P, P, P], I),
        "moe_slot_table_create": ([I, I, I, P, ctypes.POINTER(P)], I),
        "moe_slot_table_set": ([P, I, ctypes.POINTER(_ExpertDesc), P], I),
        "moe_slot_table_evict": ([P, I, P], I),
        "moe_slot_table_destroy": ([P], I),
        "moe_router_logits": ([P, P, P, P, I, I, I, P], I),
        "moe_route_topk": ([P, I, I, I, I, P, P, P], I),
        "moe_permute_workspace_size": ([I, I, I], Z),
        "moe_permute": ([P, I, I, I, P, P, P, P, Z, P], I),
        "moe_vq2_expert_ffn_workspace_size": ([I, I, I, I, I], Z),
        "moe_vq2_expert_ffn": ([P, P, P, P, P, I, I, I, P, P, P, Z, P], I),
        "moe_vq2_expert_ffn_noalloc": ([P, P, P, P, P, I, I, I, P, P, P], I),
        "moe_combine": ([P, P, P, P, I, I, I, P, P, P], I),
        "moe_launch_count": ([], ctypes.c_uint64),
        "moe_route_workspace_size": ([I, I, I], Z),
        "moe_route": ([P, P, P, I, I, I, I, I, P, P, P, P, P, P, P, Z, P], I),
        "moe_vq2_expert_ffn_combine": ([P, P, P, P, P, P, I, I, P, P, P, P, P, Z, P], I),
        "moe_selftest": ([P], I),
        "moe_selftest_wait_timeout": ([P, P], I),
        "moe_expert_cache_slot_bytes": ([I, I, I], Z),
        "moe_expert_cache_create": ([P, P, Z, Z, ctypes.POINTER(P)], I),
        "moe_expert_cache_set_host": ([P, I, ctypes.POINTER(_ExpertDesc)], I),
        "moe_expert_cache_fetch": ([P, P, I, P, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I)], I),
        "moe_expert_cache_slot_of": ([P, I], I),
        "moe_expert_cache_stats": ([P] + [ctypes.POINTER(ctypes.c_uint64)] * 4, I),
        "moe_expert_cache_plan": ([I, I, P, P, P, ctypes.c_uint64, P, I, P, P, ctypes.POINTER(I)], I),
        "moe_expert_cache_destroy": ([P, P], I),
        "moe_expert_cache_set_host_image": ([P, I, I, P], I),
        "moe_cpu_pool_create": ([I, ctypes.POINTER(P)], I),
        "moe_cpu_pool_threads": ([P], I),
        "moe_cpu_pool_destroy": ([P], I),
        "moe_cpu_expert_ffn": ([P, I, I, P, ctypes.POINTER(_ExpertDesc), I, P, P, P, P, I, I, P], I),
        "moe_accumulate": ([P, P, Z, P], I),
        "moe_slot_table_resident": ([P, I], I),
        "moe_vq2_pack_host": ([P, P, I, I, P, P], I),
        "moe_fp4_pack_host": ([P, P, I, I, P, P], I),
        "moe_confidence_gate": ([P, P, P, I, I, I, ctypes.c_float, P, P], I),
        "moe_vq2_encoder_workspace_size": ([I, I], Z),
        "moe_vq2_train_codebook": ([P, I, I, P, I, P, P, P, Z, P], I),
        "moe_vq2_encode": ([P, I, I, P, I, P, P, P, Z, P], I),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    if path is None:
        _lib = lib
    return lib


def _check(status: int):
    if status != MOE_OK:
        raise MoeError(status, load().moe_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ formats

def moe_vq2_pack(codes, scales, packed_codes, packed_scales, stream=None):
    rows, G = codes.shape
    _check(load().moe_vq2_pack(_ptr(codes), _ptr(scales), rows, 4 * G, _ptr(packed_codes),
                               _ptr(packed_scales), _stream(stream)))


def moe_fp4_pack(codes, scales, packed_codes, packed_scales, stream=None):
    rows, nb = codes.shape
    _check(load().moe_fp4_pack(_ptr(codes), _ptr(scales), rows, 2 * nb, _ptr(packed_codes),
                               _ptr(packed_scales), _stream(stream)))


class SlotTable:
    """moe_slot_table_create / _set / _evict / _destroy.  Keeps references to
    the tensors of every set entry so they outlive the table's use of them."""

    def __init__(self, num_experts: int, H: int, I: int, codebook: torch.Tensor):
        self.lib = load()
        self.codebook = codebook
        self.E, self.H, self.I = num_experts, H, I
        h = ctypes.c_void_p()
        _check(self.lib.moe_slot_table_create(num_experts, H, I, _ptr(codebook), ctypes.byref(h)))
        self.handle = h
        self._keep = {}

    def set(self, expert_id: int, fmt: int, codes: Sequence[torch.Tensor], scales: Sequence[torch.Tensor],
            stream=None):
        d = _ExpertDesc()
        d.format = fmt
        for m in range(3):
            d.codes[m] = _ptr(codes[m])
            d.scales[m] = _ptr(scales[m])
        _check(self.lib.moe_slot_table_set(self.handle, expert_id, ctypes.byref(d), _stream(stream)))
        self._keep[expert_id] = (list(codes), list(scales))

    def evict(self, expert_id: int, stream=None):
        _check(self.lib.moe_slot_table_evict(self.handle, expert_id, _stream(stream)))

    def destroy(self):
        if self.handle is not None:
            _check(self.lib.moe_slot_table_destroy(self.handle))
            self.handle = None
            self._keep.clear()

    def __del__(self):
        try:
            if self.handle is not None and torch.cuda.is_initialized():
                torch.cuda.synchronize()
                self.destroy()
        except Exception:
            pass


# ------------------------------------------------------------------ hot path

def moe_router_logits(x, w_router, bias, logits, stream=None):
    T, H = x.shape
    E = w_router.shape[0]
    _check(load().moe_router_logits(_ptr(x), _ptr(w_router), _ptr(bias), _ptr(logits), T, H, E,
                                    _stream(stream)))


def moe_route_topk(logits, k: int, renormalize: int, ids, weights, stream=None):
    T, E = logits.shape
    _check(load().moe_route_topk(_ptr(logits), T, E, k, renormalize, _ptr(ids), _ptr(weights),
                                 _stream(stream)))


def moe_permute_workspace_size(T: int, k: int, E: int) -> int:
    return load().moe_permute_workspace_size(T, k, E)


def moe_permute(ids, E: int, expert_offsets, sorted_pair, pair_to_sorted, ws=None, stream=None):
    T, k = ids.shape
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().moe_permute(_ptr(ids), T, k, E, _ptr(expert_offsets), _ptr(sorted_pair),
                              _ptr(pair_to_sorted), _ptr(ws), nbytes, _stream(stream)))


def moe_vq2_expert_ffn_workspace_size(T: int, k: int, E: int, H: int, I: int) -> int:
    return load().moe_vq2_expert_ffn_workspace_size(T, k, E, H, I)


def moe_vq2_expert_ffn(table: SlotTable, x, expert_offsets, sorted_pair, weights, k: int, mode: int,
                       out, pair_status, ws, stream=None):
    T = x.shape[0]
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().moe_vq2_expert_ffn(table.handle, _ptr(x), _ptr(expert_offsets), _ptr(sorted_pair),
                                     _ptr(weights), T, k, mode, _ptr(out), _ptr(pair_status), _ptr(ws),
                                     nbytes, _stream(stream)))


MOE_NOALLOC_SCRATCH_BYTES = 64 << 20


def moe_vq2_expert_ffn_noalloc(table: SlotTable, x, expert_offsets, sorted_pair, weights, k: int, mode: int,
                               out, pair_status, stream=None):
    """moe_vq2_expert_ffn without a workspace argument, for callers that cannot
    allocate device memory: the library's fixed MOE_NOALLOC_SCRATCH_BYTES
    device array serves as scratch (shared by every call on a device, so
    calls must not overlap on the GPU)."""
    T = x.shape[0]
    _check(load().moe_vq2_expert_ffn_noalloc(table.handle, _ptr(x), _ptr(expert_offsets), _ptr(sorted_pair),
                                             _ptr(weights), T, k, mode, _ptr(out), _ptr(pair_status),
                                             _stream(stream)))


def moe_combine(ypair, pair_to_sorted, weights, pair_status, k: int, out_f32=None, out_bf16=None,
                stream=None):
    T = weights.shape[0]
    H = ypair.shape[1]
    _check(load().moe_combine(_ptr(ypair), _ptr(pair_to_sorted), _ptr(weights), _ptr(pair_status), T, k,
                              H, _ptr(out_f32), _ptr(out_bf16), _stream(stream)))




def moe_launch_count() -> int:
    """Kernel launches the library has issued since it was loaded (a launch
    inside a stream capture counts once)."""
    return int(load().moe_launch_count())


def moe_selftest(stream=None) -> None:
    """Boot self-check of the library on the current device: runs a tiny
    layer through every kernel family and compares with stored CPU-reference
    results.  Synchronises the stream; raises MoeError (status
    MOE_ERR_MISMATCH for a wrong result) on failure."""
    _check(load().moe_selftest(_stream(stream)))


def moe_selftest_wait_timeout(stream=None) -> dict:
    """Self-check of the kernels' bounded-wait pattern: two waits on mbarriers
    that nothing completes give up, record their codes and return.  Raises
    MoeError if they do not; returns the codes and each wait's microseconds."""
    codes = (ctypes.c_int * 6)()
    _check(load().moe_selftest_wait_timeout(codes, _stream(stream)))
    return dict(codes=(codes[0], codes[1]), gave_up=(codes[2] == 0, codes[3] == 0), us=(codes[4], codes[5]))


def moe_route_workspace_size(T: int, k: int, E: int) -> int:
    return int(load().moe_route_workspace_size(T, k, E))


def moe_route(x, w_router, bias, k: int, renormalize: int, logits, ids, weights, expert_offsets, sorted_pair,
              pair_to_sorted, ws, stream=None):
    """Router logits, top-k softmax and permutation in one call (one kernel
    for small batches).  ws: a zero-filled device buffer of at least
    moe_route_workspace_size bytes, left zeroed by the call."""
    T, H = x.shape
    E = w_router.shape[0]
    _check(load().moe_route(_ptr(x), _ptr(w_router), _ptr(bias), T, H, E, k, renormalize, _ptr(logits), _ptr(ids),
                            _ptr(weights), _ptr(expert_offsets), _ptr(sorted_pair), _ptr(pair_to_sorted), _ptr(ws),
                            ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream)))


def moe_vq2_expert_ffn_combine(table: "SlotTable", x, expert_offsets, sorted_pair, pair_to_sorted, weights, k: int,
                               ypair, pair_status, out_f32=None, out_bf16=None, ws=None, stream=None):
    """moe_vq2_expert_ffn (per-pair mode) and then moe_combine in one call
    (for single-token calls the combine runs inside the expert kernels)."""
    T = x.shape[0]
    _check(load().moe_vq2_expert_ffn_combine(table.handle, _ptr(x), _ptr(expert_offsets), _ptr(sorted_pair),
                                             _ptr(pair_to_sorted), _ptr(weights), T, k, _ptr(ypair),
                                             _ptr(pair_status), _ptr(out_f32), _ptr(out_bf16), _ptr(ws),
                                             ws.numel() * ws.element_size() if ws is not None else 0,
                                             _stream(stream)))


# ------------------------------------------------------------------ expert cache

def moe_expert_cache_slot_bytes(H: int, I: int, fmt: int) -> int:
    """Bytes of one cache slot for an expert of format fmt."""
    return int(load().moe_expert_cache_slot_bytes(H, I, fmt))


def moe_expert_cache_plan(num_experts: int, slot_expert, counts, last_step, step: int, request):
    """Host-only planning step of the expert cache.  slot_expert (int32),
    counts and last_step (uint64) are numpy arrays updated in place; returns
    (fill_slot, evicted, n_unplaced) for the requests."""
    import numpy as np
    for a, dt in ((slot_expert, np.int32), (counts, np.uint64), (last_step, np.uint64)):
        if not (isinstance(a, np.ndarray) and a.dtype == dt and a.flags.c_contiguous):
            raise ValueError(f"expected a contiguous numpy {dt.__name__} array")
    req = np.ascontiguousarray(request, dtype=np.int32)
    fill = np.empty(req.size, np.int32)
    ev = np.empty(req.size, np.int32)
    left = ctypes.c_int(0)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    _check(load().moe_expert_cache_plan(num_experts, slot_expert.size, vp(slot_expert), vp(counts), vp(last_step),
                                        step, vp(req), req.size, vp(fill), vp(ev), ctypes.byref(left)))
    return fill, ev, left.value


def _host_ptr(t: torch.Tensor) -> int:
    if t.is_cuda or not t.is_pinned():
        raise ValueError("expected a page-locked (pinned) host tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


class ExpertCache:
    """moe_expert_cache_*: slot-table entries filled on a miss from pinned
    host copies of the experts' packed buffers, into slots of a device pool
    (a uint8 CUDA tensor this object keeps).  Keeps references to the host
    tensors it was given."""

    def __init__(self, table: SlotTable, pool: torch.Tensor, slot_bytes: int):
        self.lib = load()
        self.table, self.pool, self.slot_bytes = table, pool, slot_bytes
        h = ctypes.c_void_p()
        _check(self.lib.moe_expert_cache_create(table.handle, _ptr(pool), pool.numel() * pool.element_size(),
                                                slot_bytes, ctypes.byref(h)))
        self.handle = h
        self.num_slots = pool.numel() * pool.element_size() // slot_bytes
        self._host = {}

    def set_host(self, expert_id: int, fmt: int, codes: Sequence[torch.Tensor], scales: Sequence[torch.Tensor]):
        H, I = self.table.H, self.table.I
        for m in range(3):  # the packed sizes the fetch copies (the C side trusts them)
            rows, K = (H, I) if m == 2 else (I, H)
            want = (rows * K // 4, rows * K // 128 * 2) if fmt == MOE_FMT_VQ2 else (rows * K // 2, rows * K // 32)
            got = (codes[m].numel() * codes[m].element_size(), scales[m].numel() * scales[m].element_size())
            if got != want:
                raise ValueError(f"expert {expert_id} matrix {m}: {got} bytes of codes/scales, expected {want}")
        d = _ExpertDesc()
        d.format = fmt
        for m in range(3):
            d.codes[m] = _host_ptr(codes[m])
            d.scales[m] = _host_ptr(scales[m])
        _check(self.lib.moe_expert_cache_set_host(self.handle, expert_id, ctypes.byref(d)))
        self._host[expert_id] = (list(codes), list(scales))

    def set_host_image(self, expert_id: int, fmt: int, image: torch.Tensor):
        """One pinned uint8 block in the slot's layout (host_expert_image):
        fetched with one copy."""
        want = moe_expert_cache_slot_bytes(self.table.H, self.table.I, fmt)
        if image.numel() * image.element_size() != want:
            raise ValueError(f"expert {expert_id}: image of {image.numel() * image.element_size()} bytes, "
                             f"expected {want}")
        _check(self.lib.moe_expert_cache_set_host_image(self.handle, expert_id, fmt, _host_ptr(image)))
        self._host[expert_id] = image

    def fetch(self, experts, stream=None) -> dict:
        """One step: makes the named experts resident (see the C header for
        the eviction rule).  Returns n_fetched, n_unplaced and recapture."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(experts).ravel(), dtype=np.int32)
        nf, nu, rc = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
        _check(self.lib.moe_expert_cache_fetch(self.handle, ids.ctypes.data_as(ctypes.c_void_p), ids.size,
                                               _stream(stream), ctypes.byref(nf), ctypes.byref(nu),
                                               ctypes.byref(rc)))
        return dict(n_fetched=nf.value, n_unplaced=nu.value, recapture=bool(rc.value))

    def slot_of(self, expert_id: int) -> int:
        return int(self.lib.moe_expert_cache_slot_of(self.handle, expert_id))

    def stats(self) -> dict:
        v = [ctypes.c_uint64(0) for _ in range(4)]
        _check(self.lib.moe_expert_cache_stats(self.handle, *[ctypes.byref(x) for x in v]))
        return dict(hits=v[0].value, misses=v[1].value, unplaced=v[2].value, bytes_fetched=v[3].value)

    def destroy(self, stream=None):
        if self.handle is not None:
            h, self.handle = self.handle, None
            if self.table.handle is not None:  # (the table's entries die with the table)
                _check(self.lib.moe_expert_cache_destroy(h, _stream(stream)))

    def __del__(self):
        try:
            if self.handle is not None and torch.cuda.is_initialized():
                self.destroy()
                torch.cuda.synchronize()
        except Exception:
            pass


# ------------------------------------------------------------------ host CPU path

def _np_ptr(a, dtype=None):
    """(pointer, keep-alive) of a contiguous host array: a numpy array or a
    CPU torch tensor."""
    import numpy as np
    if isinstance(a, torch.Tensor):
        if a.is_cuda:
            raise ValueError("expected a host array")
        a = a.contiguous()
        return a.data_ptr(), a
    arr = np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))
    return arr.ctypes.data, arr


def moe_vq2_pack_host(codes, scales):
    """Packs a logical VQ2 matrix on the host (uint8 [rows, K/4], fp16 bits
    [rows, K/4/32]) into the slot layout; returns (packed codes, packed
    scales) as numpy arrays of the same shapes and types."""
    import numpy as np
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.uint16)
    rows, G = c.shape
    pc, ps = np.empty_like(c), np.empty_like(sc)
    _check(load().moe_vq2_pack_host(c.ctypes.data, sc.ctypes.data, rows, 4 * G, pc.ctypes.data, ps.ctypes.data))
    return pc, ps


def moe_fp4_pack_host(codes, scales):
    """The same for a logical FP4 matrix (uint8 [rows, K/2], uint8 [rows, K/32])."""
    import numpy as np
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, nb = c.shape
    pc, ps = np.empty_like(c), np.empty_like(sc)
    _check(load().moe_fp4_pack_host(c.ctypes.data, sc.ctypes.data, rows, 2 * nb, pc.ctypes.data, ps.ctypes.data))
    return pc, ps


def host_pack_expert(fmt: int, codes: Sequence, scales: Sequence):
    """One expert's three matrices packed on the host: (fmt, [codes x3], [scales x3])."""
    pack = moe_vq2_pack_host if fmt == MOE_FMT_VQ2 else moe_fp4_pack_host
    pcs, pss = [], []
    for m in range(3):
        pc, ps = pack(codes[m], scales[m])
        pcs.append(pc)
        pss.append(ps)
    return fmt, pcs, pss


class CpuPool:
    """moe_cpu_pool: host threads for moe_cpu_expert_ffn (threads <= 0: all)."""

    def __init__(self, threads: int = 0):
        self.lib = load()
        h = ctypes.c_void_p()
        _check(self.lib.moe_cpu_pool_create(threads, ctypes.byref(h)))
        self.handle = h

    @property
    def threads(self) -> int:
        return int(self.lib.moe_cpu_pool_threads(self.handle))

    def close(self):
        if self.handle is not None:
            h, self.handle = self.handle, None
            _check(self.lib.moe_cpu_pool_destroy(h))

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HostExperts:
    """The moe_expert_desc array of host-resident packed experts that
    moe_cpu_expert_ffn reads: entry e is (fmt, [codes x3], [scales x3]) host
    arrays (host_pack_expert) or None.  Keeps the arrays alive."""

    def __init__(self, E: int):
        self.E = E
        self.descs = (_ExpertDesc * E)()
        self._keep = {}

    def set(self, e: int, fmt: int, codes: Sequence, scales: Sequence):
        d = self.descs[e]
        d.format = fmt
        keep = []
        for m in range(3):
            pc, kc = _np_ptr(codes[m])
            ps, ks = _np_ptr(scales[m])
            d.codes[m] = pc
            d.scales[m] = ps
            keep += [kc, ks]
        self._keep[e] = keep


def moe_cpu_expert_ffn(pool: CpuPool, H: int, I: int, codebook, experts: HostExperts, x, ids, weights,
                       gpu_status, k: int, out=None):
    """The remainder of the combine over the pairs with gpu_status 0,
    computed on the host (see the C header).  x: host bf16 bits [T, H];
    ids int32 / weights fp32 [T, k]; gpu_status uint8 [T*k]; out: host fp32
    [T, H] (allocated when None).  Returns out."""
    import numpy as np
    xp, xk = _np_ptr(x, np.uint16)
    ip, ik = _np_ptr(ids, np.int32)
    wp, wk = _np_ptr(weights, np.float32)
    sp, sk = _np_ptr(gpu_status, np.uint8)
    cp, ck = _np_ptr(codebook, np.uint16)
    T = int(np.prod(xk.shape)) // H
    if out is None:
        out = np.empty((T, H), np.float32)
    op, ok = _np_ptr(out)
    _check(load().moe_cpu_expert_ffn(pool.handle, H, I, cp, experts.descs, experts.E, xp, ip, wp, sp, T, k, op))
    return out


def moe_accumulate(dst, src, stream=None):
    """dst += src on the device (fp32 CUDA tensors of equal size)."""
    if dst.numel() != src.numel():
        raise ValueError("moe_accumulate: sizes differ")
    _check(load().moe_accumulate(_ptr(dst), _ptr(src), dst.numel(), _stream(stream)))


def moe_slot_table_resident(table: "SlotTable", expert_id: int) -> bool:
    r = int(load().moe_slot_table_resident(table.handle, expert_id))
    if r < 0:
        _check(r)
    return r == 1


def moe_confidence_gate(table: "SlotTable", ids, weights, E: int, tau: float, gated_ids, stream=None):
    """gated_ids = ids + E where weights >= tau and the table holds entry
    E + id (the expert's FP4 weights), ids elsewhere (see the C header)."""
    T, k = ids.shape
    _check(load().moe_confidence_gate(table.handle, _ptr(ids), _ptr(weights), T, k, E, tau, _ptr(gated_ids),
                                      _stream(stream)))


# ------------------------------------------------------------------ encoder

def moe_vq2_train_codebook(W: torch.Tensor, init_idx, iters: int, stream=None):
    """The layer codebook from dense fp32 weights W [rows, K] (CUDA): k-means
    from the normalised group vectors at init_idx (128 indices).  Returns
    (codebook fp16 [128, 4], centroids fp32 [128, 4]) on the device."""
    import numpy as np
    rows, K = W.shape
    idx = np.ascontiguousarray(np.asarray(init_idx, dtype=np.int64).ravel())
    if idx.size != 128:
        raise ValueError("init_idx needs 128 indices")
    ws = torch.empty(load().moe_vq2_encoder_workspace_size(rows, K), dtype=torch.uint8, device=W.device)
    cb = torch.empty(128, 4, dtype=torch.float16, device=W.device)
    C = torch.empty(128, 4, dtype=torch.float32, device=W.device)
    _check(load().moe_vq2_train_codebook(_ptr(W), rows, K, idx.ctypes.data, iters, _ptr(cb), _ptr(C), _ptr(ws),
                                         ws.numel(), _stream(stream)))
    return cb, C


def moe_vq2_encode(W: torch.Tensor, codebook: torch.Tensor, iters: int = 3, stream=None):
    """Codes uint8 [rows, K/4] and scales fp16 [rows, K/128] (logical layout)
    of dense fp32 weights W [rows, K] (CUDA) with a fp16 codebook [128, 4]."""
    rows, K = W.shape
    ws = torch.empty(load().moe_vq2_encoder_workspace_size(rows, K), dtype=torch.uint8, device=W.device)
    codes = torch.empty(rows, K // 4, dtype=torch.uint8, device=W.device)
    scales = torch.empty(rows, K // 128, dtype=torch.float16, device=W.device)
    _check(load().moe_vq2_encode(_ptr(W), rows, K, _ptr(codebook), iters, _ptr(codes), _ptr(scales), _ptr(ws),
                                 ws.numel(), _stream(stream)))
    return codes, scales


from .layer import (GatedForward, GraphedForward, GraphedStep, MissFetchForward, MoELayer, PipelinedSteps,  # noqa: E402,F401
                    TandemForward, host_expert, host_expert_image, upload_layer, upload_expert)
