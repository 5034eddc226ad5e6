"""CPU oracle of the routed-expert VQ2 MoE layer (plain C, fp64) + a thin
ctypes wrapper.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
cpu_baseline / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never imports it, and it imports nothing from the
CUDA library; the only module both sides share is the seeded input generator
``moe_synth``.

Every function follows the definition in ``moe_oracle.c`` (see the citations
there): decode the codes to dense fp64 weights and run naive matmuls.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libmoe_oracle.so")

_lib = None


def build(out: str = _LIB, src: str = _SRC) -> str:
    """Compile the oracle with gcc (OpenMP, -O2, no fast-math, no FMA
    contraction)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_router_logits_f32.argtypes = [P, P, P, i, i, i, P]
    lib.oracle_router_logits_f64.argtypes = [P, P, P, i, i, i, P]
    lib.oracle_route_topk.argtypes = [P, i, i, i, i, P, P]
    lib.oracle_permute.argtypes = [P, i, i, P, P, P]
    lib.oracle_decode_vq2.argtypes = [P, P, P, i, i, P]
    lib.oracle_decode_fp4.argtypes = [P, P, i, i, P]
    lib.oracle_expert_ffn.argtypes = [i, P, P, P, P, P, P, P, i, i, i, P, P]
    lib.oracle_combine.argtypes = [i, i, i, P, P, P, P]
    lib.oracle_set_threads.argtypes = [i]
    lib.oracle_fp16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_fp16_value.restype = ctypes.c_double
    lib.oracle_e2m1_value.argtypes = [ctypes.c_uint]
    lib.oracle_e2m1_value.restype = ctypes.c_double
    return lib


def lib():
    """The oracle library; MOE_ORACLE_LIB names another build of the same
    source (used only by the planted-mistake test)."""
    global _lib
    if _lib is None:
        alt = os.environ.get("MOE_ORACLE_LIB")
        if alt:
            _lib = _bind(alt)
            return _lib
        if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            build()
        _lib = _bind(_LIB)
    return _lib


def load_variant(path: str) -> "Oracle":
    """An Oracle bound to another build of moe_oracle.c (planted-mistake tests)."""
    return Oracle(_bind(path))


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with status {rc}")


class Oracle:
    def __init__(self, handle=None):
        self._h = handle

    @property
    def h(self):
        return self._h if self._h is not None else lib()

    def set_threads(self, n: int = 0) -> int:
        return self.h.oracle_set_threads(int(n))

    # -- scalar formats -------------------------------------------------
    def fp16_value(self, bits: int) -> float:
        return self.h.oracle_fp16_value(int(bits))

    def e2m1_value(self, nib: int) -> float:
        return self.h.oracle_e2m1_value(int(nib))

    # -- router ---------------------------------------------------------
    def router_logits(self, x_bits, w_bits, bias=None) -> np.ndarray:
        x = np.ascontiguousarray(x_bits, np.uint16)
        w = np.ascontiguousarray(w_bits, np.uint16)
        b = None if bias is None else np.ascontiguousarray(bias, np.float32)
        T, H = x.shape
        E = w.shape[0]
        out = np.empty((T, E), np.float32)
        _check(self.h.oracle_router_logits_f32(_p(x), _p(w), _p(b), T, H, E, _p(out)), "router")
        return out

    def router_logits_f64(self, x_bits, w_bits, bias=None) -> np.ndarray:
        x = np.ascontiguousarray(x_bits, np.uint16)
        w = np.ascontiguousarray(w_bits, np.uint16)
        b = None if bias is None else np.ascontiguousarray(bias, np.float32)
        T, H = x.shape
        E = w.shape[0]
        out = np.empty((T, E), np.float64)
        _check(self.h.oracle_router_logits_f64(_p(x), _p(w), _p(b), T, H, E, _p(out)), "router64")
        return out

    def route_topk(self, logits, k: int, renormalize: int = 1):
        l = np.ascontiguousarray(logits, np.float32)
        T, E = l.shape
        ids = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float64)
        _check(self.h.oracle_route_topk(_p(l), T, E, k, renormalize, _p(ids), _p(w)), "topk")
        return ids, w

    def permute(self, ids, E: int):
        i = np.ascontiguousarray(ids, np.int32).ravel()
        P = i.size
        off = np.empty(E + 1, np.int32)
        sp = np.empty(P, np.int32)
        p2s = np.empty(P, np.int32)
        _check(self.h.oracle_permute(_p(i), P, E, _p(off), _p(sp), _p(p2s)), "permute")
        return off, sp, p2s

    # -- experts --------------------------------------------------------
    def decode_vq2(self, codes, scales, cb) -> np.ndarray:
        c = np.ascontiguousarray(codes, np.uint8)
        s = np.ascontiguousarray(scales, np.uint16)
        b = np.ascontiguousarray(cb, np.uint16)
        rows, G = c.shape
        W = np.empty((rows, 4 * G), np.float64)
        _check(self.h.oracle_decode_vq2(_p(c), _p(s), _p(b), rows, 4 * G, _p(W)), "decode_vq2")
        return W

    def decode_fp4(self, codes, scales) -> np.ndarray:
        c = np.ascontiguousarray(codes, np.uint8)
        s = np.ascontiguousarray(scales, np.uint8)
        rows, nb = c.shape
        W = np.empty((rows, 2 * nb), np.float64)
        _check(self.h.oracle_decode_fp4(_p(c), _p(s), rows, 2 * nb, _p(W)), "decode_fp4")
        return W

    def expert_ffn(self, expert, cb, X) -> np.ndarray:
        """expert: moe_synth.ExpertWeights; X: fp64 [n, H] -> Y fp64 [n, H]."""
        X = np.ascontiguousarray(X, np.float64)
        n, H = X.shape
        I = expert.codes[0].shape[0]
        c = [np.ascontiguousarray(a) for a in expert.codes]
        s = [np.ascontiguousarray(a) for a in expert.scales]
        cbb = np.ascontiguousarray(cb, np.uint16)
        Y = np.empty((n, H), np.float64)
        _check(self.h.oracle_expert_ffn(int(expert.fmt), _p(c[0]), _p(s[0]), _p(c[1]), _p(s[1]),
                                        _p(c[2]), _p(s[2]), _p(cbb), H, I, n, _p(X), _p(Y)),
               "expert_ffn")
        return Y

    def combine(self, weights, ypair, include=None) -> np.ndarray:
        w = np.ascontiguousarray(weights, np.float64)
        T, k = w.shape
        y = np.ascontiguousarray(ypair, np.float64)
        H = y.shape[1]
        inc = None if include is None else np.ascontiguousarray(include, np.uint8).ravel()
        out = np.empty((T, H), np.float64)
        _check(self.h.oracle_combine(T, k, H, _p(w), _p(y), _p(inc), _p(out)), "combine")
        return out

    # -- the whole layer ------------------------------------------------
    def moe_layer(self, layer, x_bits, resident: Optional[np.ndarray] = None,
                  tokens: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
        """Route every token; run the expert FFNs for the pairs of ``tokens``
        (all tokens when None); combine.  ``resident``: bool [E] mask of the
        experts held on the GPU (None = all).  Returns ids, weights (fp64),
        logits (fp32), the permutation, ypair (fp64 [P, H], pair order; NaN
        rows for pairs not computed), out (all pairs), partial (resident
        experts only) and remainder (the others), each [T', H] for the
        selected tokens."""
        spec = layer.spec
        x = np.ascontiguousarray(x_bits, np.uint16)
        T = x.shape[0]
        logits = self.router_logits(x, layer.w_router, layer.bias)
        ids, w = self.route_topk(logits, spec.k, spec.renormalize)
        off, sp, p2s = self.permute(ids, spec.E)
        sel = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
        k = spec.k
        ypair = np.full((T * k, spec.H), np.nan)
        xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        want = np.zeros(T, bool)
        want[sel] = True
        for e in np.unique(ids[sel]):
            pairs = [p for p in range(off[e], off[e + 1]) if want[sp[p] // k]]
            pairs = [int(sp[s]) for s in pairs]
            if not pairs:
                continue
            X = xf[[p // k for p in pairs]]
            Y = self.expert_ffn(layer.expert(int(e)), layer.codebook, X)
            ypair[pairs] = Y
        res = np.ones(spec.E, bool) if resident is None else np.asarray(resident, bool)
        inc_res = res[ids].astype(np.uint8)
        ysel = ypair.reshape(T, k, spec.H)[sel].reshape(-1, spec.H)
        wsel = w[sel]
        out = self.combine(wsel, ysel)
        partial = self.combine(wsel, ysel, inc_res[sel])
        remainder = self.combine(wsel, ysel, 1 - inc_res[sel])
        return dict(logits=logits, ids=ids, weights=w, offsets=off, sorted_pair=sp,
                    pair_to_sorted=p2s, ypair=ypair, out=out, partial=partial,
                    remainder=remainder, tokens=sel)


default = Oracle()
