"""Seeded synthetic inputs for the routed-expert VQ2 MoE layer.

This module only draws random numbers and lays them out in the storage
formats; it holds none of the layer's arithmetic (no decoding, routing,
matmul or combine).  Both the CPU oracle (``oracle/``) and the CUDA
library's tests and benchmark take their inputs from here, so that the two
sides are fed identical bytes.

Formats (the VQ2 expert code of the Tandem-vLLM page, "How it works":
2-bit vector codes at about 2.1 bits/weight; sign-symmetric codebook of the
vLLM-Moet page, "2-bit experts on vLLM v0.24.0"):

* VQ2 matrix [rows, K]: ``codes`` uint8 [rows, K/4] (bit 7 = sign, bits 0-6 =
  index into a 128-entry codebook of 4-vectors, one code per 4 consecutive
  inputs of a row), ``scales`` fp16 bits (uint16) [rows, K/128].
* FP4 matrix [rows, K] (MXFP4: e2m1 elements, one ue8m0 exponent per 32):
  ``codes`` uint8 [rows, K/2] (low nibble = even element), ``scales`` uint8
  [rows, K/32].
* codebook fp16 bits [128, 4]; router weight bf16 bits [E, H]; tokens bf16
  bits [T, H]; router bias fp32 [E] or None.

Every array comes from its own ``numpy.random.default_rng`` stream keyed by
(seed, layer, expert, tensor), so experts can be drawn lazily and in any
order.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

FMT_VQ2 = 0
FMT_FP4 = 1

# stream tags
_TAG_TOKENS, _TAG_WR, _TAG_CB, _TAG_RANK = 1, 2, 3, 4
_TAG_CODES, _TAG_SCALES = 10, 20


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); return the
    16-bit patterns as uint16."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def fp16_bits(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng([int(k) for k in key])


def _uniform_bytes(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return np.frombuffer(rng.bytes(n), dtype=np.uint8).reshape(shape).copy()


@dataclasses.dataclass
class ExpertWeights:
    """One routed expert: gate [I,H], up [I,H], down [H,I] in one format."""
    fmt: int
    codes: List[np.ndarray]    # gate, up, down
    scales: List[np.ndarray]   # gate, up, down

    @property
    def nbytes(self) -> int:
        return sum(c.nbytes for c in self.codes) + sum(s.nbytes for s in self.scales)


@dataclasses.dataclass
class LayerSpec:
    H: int
    I: int
    E: int
    k: int
    seed: int
    layer: int = 0
    zipf_s: Optional[float] = None          # router bias gives Zipf(s) popularity
    fp4_top: int = 0                        # this many most popular experts stored FP4
    renormalize: int = 1

    def key(self, *tags: int):
        return (self.seed, self.layer) + tags


class Layer:
    """Lazily drawn weights of one synthetic MoE layer."""

    def __init__(self, spec: LayerSpec):
        if spec.H % 256 or spec.I % 128:
            raise ValueError("H must be a multiple of 256 and I of 128")
        self.spec = spec
        H, E = spec.H, spec.E
        r = _rng(*spec.key(_TAG_WR))
        self.w_router = bf16_bits(r.normal(0.0, 0.02, size=(E, H)).astype(np.float32))
        r = _rng(*spec.key(_TAG_CB))
        self.codebook = fp16_bits(r.normal(0.0, 1.0, size=(128, 4)))
        # popularity rank of each expert (1 = most routed), a seeded permutation
        r = _rng(*spec.key(_TAG_RANK))
        self.rank = (r.permutation(E) + 1).astype(np.int64)
        if spec.zipf_s is not None:
            # log-probability of a Zipf(s) law over the ranks, added to the router
            # logits; top-k of (Gaussian router noise + log p) then routes like
            # Plackett-Luce sampling from Zipf(s) (the Gaussian noise std,
            # 0.02*sqrt(H) = 1.28 at H=4096, matches the Gumbel std pi/sqrt(6)).
            self.bias = (-spec.zipf_s * np.log(self.rank.astype(np.float64))).astype(np.float32)
        else:
            self.bias = None
        self.formats = np.full(E, FMT_VQ2, dtype=np.int32)
        if spec.fp4_top:
            self.formats[self.rank <= spec.fp4_top] = FMT_FP4
        self._cache: Dict[int, ExpertWeights] = {}

    def expert(self, e: int, cache: bool = True) -> ExpertWeights:
        if e in self._cache:
            return self._cache[e]
        s = self.spec
        H, I = s.H, s.I
        shapes = [(I, H), (I, H), (H, I)]
        fmt = int(self.formats[e])
        codes, scales = [], []
        for m, (rows, K) in enumerate(shapes):
            rc = _rng(*s.key(_TAG_CODES + m, e))
            rs = _rng(*s.key(_TAG_SCALES + m, e))
            if fmt == FMT_VQ2:
                codes.append(_uniform_bytes(rc, (rows, K // 4)))
                scales.append(fp16_bits(rs.uniform(0.005, 0.02, size=(rows, K // 128))))
            else:
                codes.append(_uniform_bytes(rc, (rows, K // 2)))
                # ue8m0 exponents 118..120 (2^-9..2^-7): weight spread close to VQ2's
                scales.append(rs.integers(118, 121, size=(rows, K // 32)).astype(np.uint8))
        w = ExpertWeights(fmt, codes, scales)
        if cache:
            self._cache[e] = w
        return w

    def drop_cache(self):
        self._cache.clear()


def tokens(T: int, H: int, seed: int, layer: int = 0, stream: int = 0) -> np.ndarray:
    """bf16 bits [T, H] of N(0,1) activations."""
    r = _rng(seed, layer, _TAG_TOKENS, stream)
    return bf16_bits(r.normal(0.0, 1.0, size=(T, H)).astype(np.float32))


# The five workloads of the benchmark and parity suite.
def spec_tiny(seed: int = 0) -> LayerSpec:
    """hidden 256, intermediate 128, 8 experts, top-2, 4 tokens."""
    return LayerSpec(H=256, I=128, E=8, k=2, seed=seed)


def spec_decode(layer: int, seed: int = 0, zipf_s=None, fp4_top: int = 0) -> LayerSpec:
    """hidden 4096, intermediate 2048, 256 experts, top-8."""
    return LayerSpec(H=4096, I=2048, E=256, k=8, seed=seed + layer, layer=layer,
                     zipf_s=zipf_s, fp4_top=fp4_top)


WORKLOADS = {
    "tiny": dict(T=4, layers=1),
    "decode_b1": dict(T=1, layers=4),
    "decode_b32_zipf": dict(T=32, layers=1, zipf_s=1.1),
    "mixed_fp4_b8": dict(T=8, layers=1, zipf_s=1.1, fp4_top=52, resident_subset=96),
    "prefill_4096": dict(T=4096, layers=1, zipf_s=1.1),
}


def most_popular(layer: Layer, n: int) -> np.ndarray:
    """Ids of the n experts with the lowest popularity rank."""
    return np.nonzero(layer.rank <= n)[0].astype(np.int32)
