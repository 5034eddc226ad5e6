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
_TAG_DENSE = 30


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


def tokens_outliers(T: int, H: int, seed: int, n_channels: int = 4, lo: float = 1e3, hi: float = 1e5,
                    stream: int = 0) -> np.ndarray:
    """bf16 bits [T, H]: N(0,1) activations with n_channels outlier channels
    (the same channels for every token, as activation outliers of language
    models are), each value of magnitude log-uniform in [lo, hi] with a
    random sign; the first outlier of token 0 has magnitude hi."""
    r = _rng(seed, 0, _TAG_TOKENS, 1000 + stream)
    x = r.normal(0.0, 1.0, size=(T, H))
    ch = r.choice(H, size=n_channels, replace=False)
    mag = np.exp(r.uniform(np.log(lo), np.log(hi), size=(T, n_channels)))
    mag[0, 0] = hi
    x[:, ch] = mag * r.choice([-1.0, 1.0], size=(T, n_channels))
    return bf16_bits(x.astype(np.float32))


def dense_weights(rows: int, K: int, seed: int, std: float = 0.013, stream: int = 0) -> np.ndarray:
    """fp32 [rows, K] of N(0, std^2) weights (dense input of the encoder)."""
    r = _rng(seed, 0, _TAG_DENSE, stream)
    return r.normal(0.0, std, size=(rows, K)).astype(np.float32)


def encoder_init_indices(n_groups: int, seed: int, n: int = 128) -> np.ndarray:
    """n distinct indices in [0, n_groups) (int64): where the codebook's
    k-means starts."""
    return _rng(seed, 0, _TAG_DENSE, 999).choice(n_groups, size=n, replace=False).astype(np.int64)


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
    "mixed_fp4_b1": dict(T=1, layers=4, zipf_s=1.1, fp4_top=52),
    "prefill_4096": dict(T=4096, layers=1, zipf_s=1.1),
}


def most_popular(layer: Layer, n: int) -> np.ndarray:
    """Ids of the n experts with the lowest popularity rank."""
    return np.nonzero(layer.rank <= n)[0].astype(np.int32)


# ---------------------------------------------------------------------------
# Counter-based inputs of the library's boot self-check.
#
# The self-check (Tandem-vLLM page, "New in 0.2.0": each kernel is checked
# against a reference at boot) draws its inputs on the GPU, so they cannot be
# handed over from here; the CUDA library draws the same numbers from the
# same published generator, implemented separately there.
#
# Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
# number generators", OOPSLA 2014): the first output of the generator whose
# state is s, i.e. z = s + 0x9E3779B97F4A7C15, z = (z ^ z>>30) *
# 0xBF58476D1CE4E5B9, z = (z ^ z>>27) * 0x94D049BB133111EB, z ^ z>>31, all
# mod 2^64.  Draw i of stream `tag` is the output for s = tag * 2^32 + i.
#
# Values (each exactly representable, so that rounding cannot differ):
#   g(v)   = sum of the 6-bit fields v>>0, v>>8, v>>16, v>>24 (& 63) - 126,
#            an integer in [-126, 126] with a bell-shaped law, std 36.9;
#   tokens     bf16  g / 32            (std 1.15; the N(0,1) activations)
#   router     bf16  g / 2048          (std 0.018; the N(0,0.02) router)
#   codebook   fp16  g / 32            (std 1.15; the N(0,1) codebook)
#   VQ2 codes  uint8 v & 255           (uniform codes)
#   VQ2 scales fp16  (40 + v mod 124) / 8192   (0.0049 .. 0.0199)
#   FP4 codes  uint8 v & 255           (two uniform e2m1 nibbles)
#   FP4 scales uint8 118 + v mod 3     (2^-9 .. 2^-7)
# Arrays are drawn in row-major order of their logical layout; token row t
# uses draws of row t mod 4, so larger batches repeat the four tokens.
# ---------------------------------------------------------------------------
SELFTEST_H, SELFTEST_I, SELFTEST_E, SELFTEST_K, SELFTEST_T = 256, 128, 8, 2, 4
ST_TAG_TOKENS, ST_TAG_ROUTER, ST_TAG_CODEBOOK = 1, 2, 3
ST_TAG_VQ2_CODES, ST_TAG_VQ2_SCALES = 16, 48      # + 4*expert + matrix
ST_TAG_FP4_CODES, ST_TAG_FP4_SCALES = 80, 112     # + 4*expert + matrix
SELFTEST_FP4_EXPERTS = (1, 3, 5, 7)               # FP4 in the mixed-format layer

_SM_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_SM_M1 = np.uint64(0xBF58476D1CE4E5B9)
_SM_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(state: np.ndarray) -> np.ndarray:
    """First SplitMix64 output for each uint64 state (wrapping arithmetic)."""
    z = np.asarray(state, dtype=np.uint64) + _SM_GAMMA
    z = (z ^ (z >> np.uint64(30))) * _SM_M1
    z = (z ^ (z >> np.uint64(27))) * _SM_M2
    return z ^ (z >> np.uint64(31))


def st_draw(tag: int, n: int, period: Optional[int] = None) -> np.ndarray:
    i = np.arange(n, dtype=np.uint64)
    if period is not None:
        i = i % np.uint64(period)
    return splitmix64((np.uint64(tag) << np.uint64(32)) | i)


def st_bell(v: np.ndarray) -> np.ndarray:
    f = np.zeros(v.shape, dtype=np.int64)
    for sh in (0, 8, 16, 24):
        f += ((v >> np.uint64(sh)) & np.uint64(63)).astype(np.int64)
    return f - 126


class SelftestLayer:
    """The self-check's layer (hidden 256, intermediate 128, 8 experts,
    top-2, no router bias), VQ2 everywhere or, with ``mixed``, FP4 for the
    experts in SELFTEST_FP4_EXPERTS; same interface as :class:`Layer`."""

    def __init__(self, mixed: bool = False):
        H, I, E, k = SELFTEST_H, SELFTEST_I, SELFTEST_E, SELFTEST_K
        self.spec = LayerSpec(H=H, I=I, E=E, k=k, seed=0)
        self.w_router = bf16_bits((st_bell(st_draw(ST_TAG_ROUTER, E * H)) / 2048.0)
                                  .astype(np.float32)).reshape(E, H)
        self.codebook = fp16_bits(st_bell(st_draw(ST_TAG_CODEBOOK, 512)) / 32.0).reshape(128, 4)
        self.bias = None
        self.formats = np.full(E, FMT_VQ2, dtype=np.int32)
        if mixed:
            self.formats[list(SELFTEST_FP4_EXPERTS)] = FMT_FP4

    def expert(self, e: int, cache: bool = True) -> ExpertWeights:
        H, I = SELFTEST_H, SELFTEST_I
        fmt = int(self.formats[e])
        codes, scales = [], []
        for m, (rows, K) in enumerate([(I, H), (I, H), (H, I)]):
            if fmt == FMT_VQ2:
                c = st_draw(ST_TAG_VQ2_CODES + 4 * e + m, rows * K // 4)
                s = st_draw(ST_TAG_VQ2_SCALES + 4 * e + m, rows * K // 128)
                codes.append((c & np.uint64(255)).astype(np.uint8).reshape(rows, K // 4))
                scales.append(fp16_bits((40 + (s % np.uint64(124)).astype(np.int64)) / 8192.0)
                              .reshape(rows, K // 128))
            else:
                c = st_draw(ST_TAG_FP4_CODES + 4 * e + m, rows * K // 2)
                s = st_draw(ST_TAG_FP4_SCALES + 4 * e + m, rows * K // 32)
                codes.append((c & np.uint64(255)).astype(np.uint8).reshape(rows, K // 2))
                scales.append((118 + (s % np.uint64(3)).astype(np.int64)).astype(np.uint8)
                              .reshape(rows, K // 32))
        return ExpertWeights(fmt, codes, scales)

    def drop_cache(self):
        pass


def selftest_tokens(T: int = SELFTEST_T) -> np.ndarray:
    """bf16 bits [T, 256]: row t is the self-check's token t mod 4."""
    H = SELFTEST_H
    v = st_draw(ST_TAG_TOKENS, T * H, period=SELFTEST_T * H)
    return bf16_bits((st_bell(v) / 32.0).astype(np.float32)).reshape(T, H)
