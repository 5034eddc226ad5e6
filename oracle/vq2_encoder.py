"""CPU oracle of the VQ2 encoder: dense weights -> a sign-symmetric codebook
of 128 4-vectors, 8-bit codes and fp16 scales per row per 128 inputs.

TEST INFRASTRUCTURE.  Only ``tests/`` (and the bench's CPU legs) may import
this module; the CUDA library never imports it, and it imports nothing from
the CUDA library.

What the pages fix: the experts are stored as 2-bit vector codes with a
sign-symmetric codebook (vLLM-Moet page, "2-bit experts on vLLM v0.24.0":
naive 2-bit fails through sign asymmetry, not error size), and the repository
quantises weights at start-up (the German vLLM-Moet page: IQ2 at boot).  The
code format (1 sign bit + 7-bit index, fp16 scale per row per 128 inputs) is
the workloads' definition.  The pages give no encoding algorithm; this is the
build's reading, step by step:

  1. block scale: sigma[r, b] = sqrt(sum of W[r, i]^2 over the 128 inputs of
     block b / 128); the normalised group vectors are u = W[r, 4g..4g+3] /
     sigma (u = 0 where sigma = 0);
  2. codebook: k-means over the normalised vectors with the codebook read as
     128 pairs {+c_i, -c_i}: a vector u goes to the pair i maximising
     2 |u . c_i| - |c_i|^2 (the same as minimising |u - s c_i|^2 over i and
     s = +-1), with s = sign(u . c_i); c_i becomes the mean of s u over its
     members (unchanged when it has none).  It starts from the normalised
     vectors at 128 given indices and runs a given number of iterations; the
     codebook is the result rounded to fp16;
  3. encoding with a codebook: the scale starts at sigma; each iteration
     assigns every group of the block (u = W / scale, as in 2) and sets the
     scale to the least-squares fit sum_g W_g . q_g / sum_g q_g . q_g of the
     chosen codewords q_g = s c_i (kept where the denominator is 0); then
     the scale is rounded to fp16 and the groups assigned once more against
     the rounded scale, giving the codes (bit 7 = 1 for s = -1).

Decisions that pick an integer (the pair index and the sign) are made in
fp32 with the operation order written here: a dot product is
((a0 b0 + a1 b1) + a2 b2) + a3 b3 and sums over groups run in increasing
order, every product and sum rounded to fp32 (no fused multiply-add).  The
centroid sums are exact integers: each component of s u is rounded to a
multiple of 2^-20 and summed in int64, so the training does not depend on
the order of the members; the mean is (sum * 2^-20) / count in fp64, then
rounded to fp32.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
FIX_BITS = 20          # fixed point of the centroid sums
CHUNK = 1 << 15        # group vectors scored at a time


def _dot4(a, b):
    """((a0 b0 + a1 b1) + a2 b2) + a3 b3 in fp32; a, b broadcast over [..., 4]."""
    t = F32(a[..., 0] * b[..., 0]) + F32(a[..., 1] * b[..., 1])
    t = F32(t + F32(a[..., 2] * b[..., 2]))
    return F32(t + F32(a[..., 3] * b[..., 3]))


def block_rms(W: np.ndarray) -> np.ndarray:
    """sigma [rows, K/128] of fp32 W [rows, K] (step 1), squares summed in
    increasing input order."""
    W = np.asarray(W, F32)
    rows, K = W.shape
    W3 = W.reshape(rows, K // 128, 128)
    s = np.zeros((rows, K // 128), F32)
    for i in range(128):
        s = F32(s + F32(W3[:, :, i] * W3[:, :, i]))
    return np.sqrt(F32(s / F32(128.0))).astype(F32)


def group_vectors(W: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """u [rows, K/4, 4] = W / scale of the group's block (0 where scale is 0)."""
    W = np.asarray(W, F32)
    rows, K = W.shape
    s = np.repeat(np.asarray(scale, F32), 32, axis=1)[:, :, None]  # [rows, K/4, 1]
    W4 = W.reshape(rows, K // 4, 4)
    with np.errstate(divide="ignore", invalid="ignore"):
        u = np.where(s != 0, F32(W4 / np.where(s != 0, s, F32(1.0))), F32(0.0))
    return u.astype(F32)


def assign(U: np.ndarray, C: np.ndarray):
    """Best pair and sign of each vector (step 2's rule): U fp32 [n, 4],
    C fp32 [m, 4] -> (index int64 [n], negative bool [n]).  Ties go to the
    lower index; a zero dot product takes the + sign."""
    U = np.asarray(U, F32).reshape(-1, 4)
    C = np.asarray(C, F32)
    norms = _dot4(C, C)
    idx = np.empty(U.shape[0], np.int64)
    neg = np.empty(U.shape[0], bool)
    for a in range(0, U.shape[0], CHUNK):
        u = U[a:a + CHUNK]
        d = _dot4(u[:, None, :], C[None, :, :])                  # [c, m]
        score = F32(F32(2.0) * np.abs(d)) - norms[None, :]
        best = np.argmax(score, axis=1)                           # first maximum
        idx[a:a + CHUNK] = best
        neg[a:a + CHUNK] = d[np.arange(u.shape[0]), best] < 0
    return idx, neg


def kmeans(U: np.ndarray, C0: np.ndarray, iters: int) -> np.ndarray:
    """Step 2's iterations from the fp32 centroids C0 [m, 4]; returns fp32 [m, 4]."""
    U = np.asarray(U, F32).reshape(-1, 4)
    C = np.array(C0, F32, copy=True)
    m = C.shape[0]
    for _ in range(iters):
        idx, neg = assign(U, C)
        su = np.where(neg[:, None], -U, U).astype(F32)
        fx = np.rint(F32(su * F32(2.0 ** FIX_BITS))).astype(np.int64)
        sums = np.zeros((m, 4), np.int64)
        np.add.at(sums, idx, fx)
        cnt = np.bincount(idx, minlength=m).astype(np.int64)
        has = cnt > 0
        mean = (sums.astype(np.float64) * 2.0 ** -FIX_BITS) / np.maximum(cnt, 1)[:, None].astype(np.float64)
        C = np.where(has[:, None], mean.astype(F32), C).astype(F32)
    return C


def train_codebook(W: np.ndarray, init_idx, iters: int):
    """Steps 1-2 on one matrix: the normalised group vectors at init_idx
    (indices into the rows*K/4 groups, row-major) start the k-means.
    Returns (fp32 centroids [128, 4], fp16 bits of the codebook [128, 4])."""
    u = group_vectors(W, block_rms(W)).reshape(-1, 4)
    C = kmeans(u, u[np.asarray(init_idx, np.int64)], iters)
    return C, C.astype(np.float16).view(np.uint16)


def _block_sum(a: np.ndarray) -> np.ndarray:
    """Sum over the 32 groups of each block ([rows, KB, 32] -> [rows, KB]) in increasing order."""
    s = np.zeros(a.shape[:2], F32)
    for g in range(32):
        s = F32(s + a[:, :, g])
    return s


def encode(W: np.ndarray, codebook_bits: np.ndarray, iters: int):
    """Step 3: fp32 W [rows, K] with a fp16 codebook [128, 4] -> (codes
    uint8 [rows, K/4], fp16 bits of the scales [rows, K/128])."""
    W = np.asarray(W, F32)
    rows, K = W.shape
    KB = K // 128
    C = np.asarray(codebook_bits, np.uint16).view(np.float16).astype(F32).reshape(128, 4)
    W4 = W.reshape(rows, KB, 32, 4)
    s = block_rms(W)
    for _ in range(iters):
        idx, neg = assign(group_vectors(W, s), C)
        q = C[idx].reshape(rows, KB, 32, 4)
        q = np.where(neg.reshape(rows, KB, 32, 1), -q, q).astype(F32)
        num = _block_sum(_dot4(W4, q))
        den = _block_sum(_dot4(q, q))
        with np.errstate(divide="ignore", invalid="ignore"):
            s = np.where(den > 0, F32(num / np.where(den > 0, den, F32(1.0))), s).astype(F32)
    s16 = s.astype(np.float16)
    idx, neg = assign(group_vectors(W, s16.astype(F32)), C)
    codes = (idx | (neg.astype(np.int64) << 7)).astype(np.uint8).reshape(rows, K // 4)
    return codes, s16.view(np.uint16)


def objective(U: np.ndarray, C: np.ndarray) -> float:
    """Sum over vectors of min over pairs and signs of |u - s c|^2 (fp64)."""
    U = np.asarray(U, np.float64).reshape(-1, 4)
    C = np.asarray(C, np.float64)
    tot = 0.0
    for a in range(0, U.shape[0], CHUNK):
        u = U[a:a + CHUNK]
        d2 = np.minimum(((u[:, None, :] - C[None]) ** 2).sum(-1), ((u[:, None, :] + C[None]) ** 2).sum(-1))
        tot += float(d2.min(axis=1).sum())
    return tot
