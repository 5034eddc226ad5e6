"""Pins of the VQ2 encoder oracle (oracle/vq2_encoder.py) against facts that
do not come from the oracle itself: exact recovery of a planted codebook
assignment and its power-of-two scales, exact symmetry under negation,
brute-force fp64 nearest codewords, the k-means objective never rising,
recovery of planted clusters, the block scale against fp64, and the decode
round trip through the layer oracle's decoder."""
import numpy as np
import pytest

import oracle
from oracle import vq2_encoder as enc

F32 = np.float32


def _unit_codebook(seed, min_gap=0.02):
    """128 fp16 4-vectors of norm ~1 whose pairs {+c, -c} are apart: every
    |cos| between two of them below 1 - min_gap (drawn one at a time)."""
    r = np.random.default_rng(seed)
    out = []
    while len(out) < 128:
        v = r.normal(size=4)
        v = (v / np.linalg.norm(v)).astype(np.float16).astype(np.float64)
        if all(abs(v @ w) / (np.linalg.norm(v) * np.linalg.norm(w)) < 1 - min_gap for w in out):
            out.append(v)
    return np.array(out).astype(np.float16)


def _planted(seed, rows=32, K=512):
    r = np.random.default_rng(seed)
    C16 = _unit_codebook(seed)
    idx = r.integers(0, 128, size=(rows, K // 4))
    neg = r.integers(0, 2, size=(rows, K // 4)).astype(bool)
    e = r.integers(-8, -3, size=(rows, K // 128))
    s = np.ldexp(1.0, e).astype(F32)
    q = C16.astype(F32)[idx] * np.where(neg, -1.0, 1.0)[..., None].astype(F32)
    W = (q * np.repeat(s, 32, axis=1)[..., None]).reshape(rows, K).astype(F32)
    codes = (idx | (neg.astype(np.int64) << 7)).astype(np.uint8)
    return W, C16, codes, s


def test_planted_codebook_recovered_exactly():
    W, C16, codes, s = _planted(1)
    got_c, got_s = enc.encode(W, C16.view(np.uint16), iters=2)
    assert np.array_equal(got_c, codes)
    assert np.array_equal(got_s.view(np.float16).astype(F32), s)


def test_negation_flips_every_sign_bit_and_keeps_scales():
    r = np.random.default_rng(2)
    W = r.normal(0, 0.02, size=(48, 1024)).astype(F32)
    C16 = r.normal(size=(128, 4)).astype(np.float16)
    c1, s1 = enc.encode(W, C16.view(np.uint16), iters=3)
    c2, s2 = enc.encode(-W, C16.view(np.uint16), iters=3)
    assert np.array_equal(c2, c1 ^ 0x80)
    assert np.array_equal(s1, s2)


def test_assignment_is_the_nearest_signed_codeword():
    r = np.random.default_rng(3)
    U = r.normal(size=(4000, 4)).astype(F32)
    C = r.normal(size=(128, 4)).astype(F32)
    idx, neg = enc.assign(U, C)
    u, c = U.astype(np.float64), C.astype(np.float64)
    dp = ((u[:, None, :] - c[None]) ** 2).sum(-1)
    dn = ((u[:, None, :] + c[None]) ** 2).sum(-1)
    d = np.minimum(dp, dn)
    best = d.argmin(1)
    srt = np.sort(d, axis=1)
    clear = (srt[:, 1] - srt[:, 0]) > 1e-4 * (1 + srt[:, 0])
    assert clear.mean() > 0.99
    assert np.array_equal(idx[clear], best[clear])
    want_neg = dn[np.arange(len(U)), best] < dp[np.arange(len(U)), best]
    assert np.array_equal(neg[clear], want_neg[clear])


def test_kmeans_objective_never_rises():
    r = np.random.default_rng(4)
    U = r.normal(size=(20000, 4)).astype(F32)
    C = U[r.choice(len(U), 128, replace=False)]
    prev = enc.objective(U, C)
    for _ in range(6):
        C = enc.kmeans(U, C, 1)
        cur = enc.objective(U, C)
        assert cur <= prev * (1 + 1e-9)
        prev = cur


def test_kmeans_recovers_planted_clusters():
    r = np.random.default_rng(5)
    centers = _unit_codebook(5).astype(F32) * F32(3.0)
    lab = r.integers(0, 128, size=20000)
    sg = np.where(r.integers(0, 2, size=20000) == 1, -1.0, 1.0).astype(F32)
    U = (centers[lab] * sg[:, None] + r.normal(0, 0.01, size=(20000, 4))).astype(F32)
    init = np.array([np.nonzero(lab == i)[0][0] for i in range(128)])  # one member of each cluster
    C = enc.kmeans(U, U[init], 5)
    # each centroid is its cluster's center up to sign, within the noise
    dist = np.minimum(np.abs(C - centers).max(1), np.abs(C + centers).max(1))
    assert dist.max() < 0.01


def test_block_rms_matches_fp64():
    r = np.random.default_rng(6)
    W = (r.normal(size=(16, 512)) * r.uniform(0.001, 100, size=(16, 1))).astype(F32)
    got = enc.block_rms(W).astype(np.float64)
    want = np.sqrt((W.astype(np.float64).reshape(16, 4, 128) ** 2).mean(-1))
    assert np.allclose(got, want, rtol=2e-6, atol=0)
    W[3, 128:256] = 0
    assert enc.block_rms(W)[3, 1] == 0
    assert not enc.group_vectors(W, enc.block_rms(W))[3, 32:64].any()


def test_encode_decode_round_trip_error():
    r = np.random.default_rng(7)
    W = r.normal(0, 0.013, size=(64, 2048)).astype(F32)
    init = r.choice(64 * 512, 128, replace=False)
    C, C16 = enc.train_codebook(W, init, iters=8)
    codes, scales = enc.encode(W, C16, iters=3)
    D = oracle.default.decode_vq2(codes, scales, C16)
    rel = np.sqrt(((D - W) ** 2).mean() / (W.astype(np.float64) ** 2).mean())
    # 2 bits per weight with a learned 4-D codebook: about a third of the signal
    assert rel < 0.45, rel
    # the least-squares scale never does worse than the starting scale
    s0 = enc.block_rms(W).astype(np.float16).view(np.uint16)
    c0, _ = enc.encode(W, C16, iters=0)
    D0 = oracle.default.decode_vq2(c0, s0, C16)
    assert ((D - W) ** 2).sum() <= ((D0 - W) ** 2).sum()
