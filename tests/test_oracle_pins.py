"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value
worked by hand from the format definition (tests/golden/), an invariant the
pages state (sign symmetry; nothing skipped or substituted), a closed form, a
library routine (numpy float16, argsort, softmax), or brute force on tiny
inputs with a separately written NumPy decode and dense matmul.
"""
import math

import numpy as np
import pytest

import moe_synth as ms
import oracle
from golden_io import keyed, lines

O = oracle.default


# ---------------------------------------------------------------- formats

def test_fp16_decoder_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([O.fp16_value(int(b)) for b in bits[::7]])
    r = ref[::7]
    ok = np.isnan(r) & np.isnan(got) | (got == r)
    assert ok.all()


def test_e2m1_and_e8m0_table():
    g = keyed("e2m1_table.txt")
    for row in lines("e2m1_table.txt"):
        if row[0] == "scale":
            continue
        nib, val = int(row[0]), float(row[1])
        got = O.e2m1_value(nib)
        assert got == val and math.copysign(1, got) == math.copysign(1, val)
    # ue8m0 through the FP4 decoder: a row of nibble 2 (= 1.0) times 2^(E-127)
    for E, val in ((int(a), float(b)) for a, b in g["scale"]):
        codes = np.full((1, 16), 0x22, np.uint8)
        W = O.decode_fp4(codes, np.array([[E]], np.uint8))
        assert (W == val).all()


def test_fp4_rejects_nan_scale():
    with pytest.raises(RuntimeError):
        O.decode_fp4(np.zeros((1, 16), np.uint8), np.array([[255]], np.uint8))


def _worked_vq2():
    g = keyed("vq2_decode_worked.txt")
    rows, K = int(g["rows"][0][0]), int(g["K"][0][0])
    cb = np.zeros((128, 4), np.float16)
    for row in g["cb"]:
        cb[int(row[0])] = [float(v) for v in row[1:]]
    scales = np.zeros((rows, K // 128), np.float16)
    for r, b, v in g["scale"]:
        scales[int(r), int(b)] = float(v)
    codes = np.full((rows, K // 4), 0x02, np.uint8)
    for r, q, c in g["code"]:
        codes[int(r), int(q)] = int(c, 16)
    expect = np.zeros((rows, K))
    for row in g["expect"]:
        r, c0 = int(row[0]), int(row[1])
        expect[r, c0:c0 + 4] = [float(v) for v in row[2:]]
    return codes, scales.view(np.uint16), cb.view(np.uint16), expect


def test_vq2_decode_worked_example():
    codes, scales, cb, expect = _worked_vq2()
    W = O.decode_vq2(codes, scales, cb)
    assert np.array_equal(W, expect)
    assert np.array_equal(np.signbit(W[0, 4:8]), np.signbit(expect[0, 4:8]))


def test_vq2_sign_flip_negates_exactly():
    # sign-symmetric codebook: the sign bit negates the decoded 4-vector
    layer = ms.Layer(ms.spec_tiny())
    ex = layer.expert(3)
    W = O.decode_vq2(ex.codes[0], ex.scales[0], layer.codebook)
    Wf = O.decode_vq2(ex.codes[0] ^ 0x80, ex.scales[0], layer.codebook)
    assert np.array_equal(Wf, -W)


def _np_decode_vq2(codes, scales, cb):
    """Separately written vectorised decode (brute-force reference)."""
    cbf = cb.view(np.float16).astype(np.float64)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    vec = cbf[codes & 0x7F] * sign[..., None]                 # [rows, G, 4]
    rows, G = codes.shape
    W = vec.reshape(rows, 4 * G)
    s = scales.view(np.float16).astype(np.float64)
    return W * np.repeat(s, 128, axis=1)


def _np_decode_fp4(codes, scales):
    table = np.array([float(r[1]) for r in lines("e2m1_table.txt") if r[0] != "scale"])
    lo, hi = table[codes & 15], table[codes >> 4]
    rows, nb = codes.shape
    W = np.stack([lo, hi], axis=-1).reshape(rows, 2 * nb)
    return W * np.repeat(np.exp2(scales.astype(np.float64) - 127), 32, axis=1)


def test_vq2_decode_bruteforce_numpy():
    layer = ms.Layer(ms.spec_tiny(seed=5))
    for e in range(3):
        ex = layer.expert(e)
        for m in range(3):
            W = O.decode_vq2(ex.codes[m], ex.scales[m], layer.codebook)
            assert np.array_equal(W, _np_decode_vq2(ex.codes[m], ex.scales[m], layer.codebook))


def test_fp4_decode_bruteforce_numpy():
    spec = ms.spec_tiny(seed=2)
    spec.fp4_top = 8
    layer = ms.Layer(spec)
    ex = layer.expert(1)
    assert ex.fmt == ms.FMT_FP4
    for m in range(3):
        W = O.decode_fp4(ex.codes[m], ex.scales[m])
        assert np.array_equal(W, _np_decode_fp4(ex.codes[m], ex.scales[m]))


# ---------------------------------------------------------------- router

def test_router_canonical_order_worked_example():
    g = keyed("router_canonical_order.txt")
    H = int(g["H"][0][0])
    x = np.full((1, H), float(g["rest"][0][0]), np.float32)
    w = np.full((1, H), float(g["rest"][0][0]), np.float32)
    x[0, 0] = float(g["x0"][0][0])
    w[0, 0] = float(g["w0"][0][0])
    x[0, 1:8] = float(g["x1_7"][0][0])
    l = O.router_logits(ms.bf16_bits(x), ms.bf16_bits(w))
    assert l[0, 0] == np.float32(g["expect_canonical"][0][0])
    # the other orders named in the fixture really give other numbers
    assert len({float(g[k][0][0]) for k in ("expect_canonical", "expect_lane_h_mod_32",
                                             "expect_sequential", "expect_exact_fp32")}) == 4
    seq = np.float32(0)
    for h in range(H):
        seq = np.float32(seq + np.float32(x[0, h] * w[0, h]))
    assert seq == np.float32(g["expect_sequential"][0][0])
    assert np.float32(float((x.astype(np.float64) * w).sum())) == np.float32(g["expect_exact_fp32"][0][0])


def test_router_butterfly_order_worked_example():
    g = keyed("router_butterfly_order.txt")
    H = int(g["H"][0][0])
    x = np.zeros((1, H), np.float32)
    w = np.zeros((1, H), np.float32)
    x[0, 0] = float(g["x0"][0][0])
    w[0, 0] = float(g["w0"][0][0])
    for h in g["h_ones"][0]:
        x[0, int(h)] = w[0, int(h)] = 1.0
    l = O.router_logits(ms.bf16_bits(x), ms.bf16_bits(w))
    assert l[0, 0] == np.float32(g["expect_canonical"][0][0])
    assert np.float32(g["expect_canonical"][0][0]) != np.float32(g["expect_xor1_first"][0][0])
    seq = np.float32(0)
    for h in range(H):
        seq = np.float32(seq + np.float32(x[0, h] * w[0, h]))
    assert seq == np.float32(g["expect_sequential"][0][0])


def test_router_logits_vs_fp64_matmul():
    layer = ms.Layer(ms.LayerSpec(H=1024, I=128, E=16, k=4, seed=9, zipf_s=1.1))
    x = ms.tokens(6, 1024, seed=9)
    l32 = O.router_logits(x, layer.w_router, layer.bias)
    xf = ms.bf16_to_f32(x).astype(np.float64)
    wf = ms.bf16_to_f32(layer.w_router).astype(np.float64)
    l64 = xf @ wf.T + layer.bias.astype(np.float64)
    assert np.allclose(O.router_logits_f64(x, layer.w_router, layer.bias), l64, rtol=0, atol=1e-12)
    # fp32 summation error bound: ~ (H/32 + 5 + 1) * 2^-24 * sum|products|
    bound = (1024 / 32 + 6) * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf).T + np.abs(layer.bias))
    assert (np.abs(l32 - l64) <= bound).all()


def test_topk_softmax_worked_example():
    g = keyed("topk_softmax_worked.txt")
    logits = np.array([[float(v) for v in g["logits"][0]]], np.float32)
    k = int(g["k"][0][0])
    ids, w = O.route_topk(logits, k, 1)
    assert ids.tolist()[0] == [int(v) for v in g["ids"][0]]
    assert np.allclose(w[0], [float(v) for v in g["weights_renorm"][0]], rtol=1e-15)
    ids0, w0 = O.route_topk(logits, k, 0)
    assert np.allclose(w0[0], [float(v) for v in g["weights_full"][0]], rtol=1e-15)


def test_topk_vs_stable_argsort_with_ties():
    rng = np.random.default_rng(4)
    # few distinct values -> many ties
    logits = rng.integers(-3, 4, size=(64, 40)).astype(np.float32)
    ids, w = O.route_topk(logits, 7, 1)
    ref = np.argsort(-logits, axis=1, kind="stable")[:, :7]
    assert np.array_equal(ids, ref)
    logits = rng.normal(size=(64, 256)).astype(np.float32)
    ids, w = O.route_topk(logits, 8, 1)
    assert np.array_equal(ids, np.argsort(-logits, axis=1, kind="stable")[:, :8])
    sel = np.take_along_axis(logits, ids, 1).astype(np.float64)
    from scipy.special import softmax
    assert np.allclose(w, softmax(sel, axis=1), rtol=1e-13, atol=0)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)
    ids0, w0 = O.route_topk(logits, 8, 0)
    full = softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(w0, np.take_along_axis(full, ids0, 1), rtol=1e-13, atol=0)


def test_permute_vs_stable_argsort():
    rng = np.random.default_rng(1)
    for (T, k, E) in [(4, 2, 8), (32, 8, 256), (100, 3, 5), (1, 1, 1)]:
        ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
        off, sp, p2s = O.permute(ids, E)
        flat = ids.ravel()
        assert np.array_equal(sp, np.argsort(flat, kind="stable"))
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
        assert np.array_equal(p2s[sp], np.arange(T * k))


# ---------------------------------------------------------------- FFN

def _onehot_expert():
    g = keyed("ffn_onehot_worked.txt")
    H, I = int(g["H"][0][0]), int(g["I"][0][0])
    cb = np.zeros((128, 4), np.float16)
    cb[1] = [2, 0, 0, 0]
    cb[2] = [0.5, 0, 0, 0]
    cb[3] = [1, 1, 1, 1]
    gate = np.zeros((I, H // 4), np.uint8)
    gate[:, 0] = 0x01
    up = np.zeros((I, H // 4), np.uint8)
    up[:, 0] = 0x02
    down = np.full((H, I // 4), 0x03, np.uint8)
    down[1::2] = 0x83
    one = np.float16(1.0).view(np.uint16)
    q = np.float16(0.25).view(np.uint16)
    sc = [np.full((I, H // 128), one, np.uint16), np.full((I, H // 128), one, np.uint16),
          np.full((H, I // 128), q, np.uint16)]
    ex = ms.ExpertWeights(ms.FMT_VQ2, [gate, up, down], sc)
    return ex, cb.view(np.uint16), g, H


def test_ffn_onehot_closed_form():
    ex, cb, g, H = _onehot_expert()
    x = np.zeros((1, H))
    x[0, 0] = 1.0
    y = O.expert_ffn(ex, cb, x)[0]
    assert np.allclose(y[0::2], float(g["y_even"][0][0]), rtol=1e-14)
    assert np.allclose(y[1::2], float(g["y_odd"][0][0]), rtol=1e-14)
    a = float(g["a"][0][0])
    assert abs(a - 2.0 / (1.0 + math.exp(-2.0)) * 0.5) < 1e-16


def _np_ffn(ex, cb, X):
    if ex.fmt == ms.FMT_VQ2:
        Wg, Wu, Wd = (_np_decode_vq2(c, s, cb) for c, s in zip(ex.codes, ex.scales))
    else:
        Wg, Wu, Wd = (_np_decode_fp4(c, s) for c, s in zip(ex.codes, ex.scales))
    G = X @ Wg.T
    U = X @ Wu.T
    A = G * (1.0 / (1.0 + np.exp(-G))) * U
    return A @ Wd.T


@pytest.mark.parametrize("fp4", [False, True])
def test_layer_bruteforce_tiny(fp4):
    spec = ms.spec_tiny(seed=0)
    if fp4:
        spec.fp4_top = 3
    layer = ms.Layer(spec)
    x = ms.tokens(4, spec.H, seed=0)
    r = O.moe_layer(layer, x)
    # independent brute force: numpy argsort routing + numpy decode + dense matmul
    xf = ms.bf16_to_f32(x).astype(np.float64)
    ref = np.zeros((4, spec.H))
    ids = np.argsort(-r["logits"], axis=1, kind="stable")[:, :spec.k]
    assert np.array_equal(ids, r["ids"])
    from scipy.special import softmax
    w = softmax(np.take_along_axis(r["logits"], ids, 1).astype(np.float64), axis=1)
    for t in range(4):
        for j in range(spec.k):
            y = _np_ffn(layer.expert(int(ids[t, j])), layer.codebook, xf[t:t + 1])[0]
            ref[t] += w[t, j] * y
    assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_single_expert_top1_is_plain_swiglu_mlp():
    spec = ms.LayerSpec(H=256, I=256, E=1, k=1, seed=3)
    layer = ms.Layer(spec)
    x = ms.tokens(5, 256, seed=3)
    r = O.moe_layer(layer, x)
    assert (r["ids"] == 0).all() and (r["weights"] == 1.0).all()
    xf = ms.bf16_to_f32(x).astype(np.float64)
    ex = layer.expert(0)
    Wg, Wu, Wd = (_np_decode_vq2(c, s, layer.codebook) for c, s in zip(ex.codes, ex.scales))
    # textbook SwiGLU MLP: W2 (silu(W1 x) * (W3 x))
    silu = lambda z: z / (1 + np.exp(-z))
    ref = (silu(xf @ Wg.T) * (xf @ Wu.T)) @ Wd.T
    assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-12)


def test_token_sample_is_a_restriction_of_the_full_layer():
    # the prefill parity test asks the oracle for a sample of the tokens only:
    # the sampled run must equal the full run's rows for those tokens, exactly
    spec = ms.LayerSpec(H=256, I=128, E=8, k=2, seed=12, zipf_s=1.1)
    layer = ms.Layer(spec)
    x = ms.tokens(9, 256, seed=12)
    full = O.moe_layer(layer, x)
    sel = np.array([7, 0, 4])
    sub = O.moe_layer(layer, x, tokens=sel)
    assert np.array_equal(sub["tokens"], sel)
    assert np.array_equal(sub["out"], full["out"][sel])
    assert np.array_equal(sub["ids"], full["ids"]) and np.array_equal(sub["weights"], full["weights"])


def test_residency_partial_plus_remainder_is_full():
    # nothing is skipped or substituted: resident part + remainder = whole layer
    spec = ms.LayerSpec(H=256, I=128, E=16, k=4, seed=11, zipf_s=1.1, fp4_top=4)
    layer = ms.Layer(spec)
    x = ms.tokens(8, 256, seed=11)
    res = np.zeros(16, bool)
    res[ms.most_popular(layer, 6)] = True
    r = O.moe_layer(layer, x, resident=res)
    assert np.allclose(r["partial"] + r["remainder"], r["out"], rtol=1e-13, atol=1e-13)
    r_all = O.moe_layer(layer, x)
    assert np.array_equal(r_all["out"], r["out"])


def test_down_scale_doubling_doubles_y_exactly():
    layer = ms.Layer(ms.spec_tiny(seed=1))
    ex = layer.expert(2)
    X = ms.bf16_to_f32(ms.tokens(2, 256, seed=1)).astype(np.float64)
    y = O.expert_ffn(ex, layer.codebook, X)
    s2 = (ex.scales[2].view(np.float16) * np.float16(2)).view(np.uint16)
    ex2 = ms.ExpertWeights(ex.fmt, ex.codes, [ex.scales[0], ex.scales[1], s2])
    assert np.array_equal(O.expert_ffn(ex2, layer.codebook, X), 2 * y)


@pytest.mark.parametrize("m", [1, 2])
def test_up_or_down_sign_flip_negates_y_exactly(m):
    layer = ms.Layer(ms.spec_tiny(seed=1))
    ex = layer.expert(5)
    X = ms.bf16_to_f32(ms.tokens(3, 256, seed=2)).astype(np.float64)
    y = O.expert_ffn(ex, layer.codebook, X)
    codes = list(ex.codes)
    codes[m] = codes[m] ^ 0x80
    yf = O.expert_ffn(ms.ExpertWeights(ex.fmt, codes, ex.scales), layer.codebook, X)
    assert np.array_equal(yf, -y)
