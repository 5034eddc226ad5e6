"""The host CPU path for experts the GPU does not hold (moe_cpu_expert_ffn,
Tandem-vLLM page, "How it works"): its remainder of the combine against the
oracle's remainder for the same resident set, the host packers against the
packed layouts as the header defines them, and argument checks.  No GPU:
the library is loaded but no CUDA call is made."""
import numpy as np
import pytest

import moe_synth as ms
import oracle
from gpu_common import assert_close

bv = pytest.importorskip("bit_vq_routed_gb300")


@pytest.fixture(scope="module")
def pool():
    p = bv.CpuPool(3)
    yield p
    p.close()


def _host_experts(layer, which):
    hx = bv.HostExperts(layer.spec.E)
    for e in which:
        ex = layer.expert(int(e))
        fmt, pc, ps = bv.host_pack_expert(ex.fmt, ex.codes, ex.scales)
        hx.set(int(e), fmt, pc, ps)
    return hx


def _remainder(pool, layer, x, resident, ref):
    s = layer.spec
    ids, w = ref["ids"], ref["weights"].astype(np.float32)
    status = resident[ids].astype(np.uint8).ravel()
    hx = _host_experts(layer, np.unique(ids.ravel()[status == 0]))
    return bv.moe_cpu_expert_ffn(pool, s.H, s.I, layer.codebook, hx, x, ids, w, status, s.k)


@pytest.mark.parametrize("spec,T", [
    (ms.spec_tiny(0), 4),
    (ms.LayerSpec(H=512, I=256, E=8, k=2, seed=51, fp4_top=3), 6),
    (ms.LayerSpec(H=1024, I=384, E=6, k=3, seed=52, zipf_s=1.1, fp4_top=2), 5),
], ids=["tiny", "mixed", "zipf_mixed"])
def test_cpu_remainder_matches_oracle(pool, spec, T):
    layer = ms.Layer(spec)
    x = ms.tokens(T, spec.H, seed=spec.seed)
    rng = np.random.default_rng(spec.seed)
    resident = rng.random(spec.E) < 0.5
    resident[0], resident[1] = True, False  # both kinds present
    ref = oracle.default.moe_layer(layer, x, resident=resident)
    got = _remainder(pool, layer, x, resident, ref)
    assert np.isfinite(got).all()
    assert_close(got, ref["remainder"], "cpu remainder")


def test_cpu_all_pairs_is_the_whole_layer_and_none_is_zero(pool):
    spec = ms.LayerSpec(H=512, I=256, E=8, k=2, seed=53, fp4_top=2)
    layer = ms.Layer(spec)
    x = ms.tokens(5, spec.H, seed=53)
    ref = oracle.default.moe_layer(layer, x)
    got = _remainder(pool, layer, x, np.zeros(spec.E, bool), ref)
    assert_close(got, ref["out"], "every pair on the CPU")
    none = _remainder(pool, layer, x, np.ones(spec.E, bool), ref)
    assert not none.any()


def test_cpu_result_does_not_depend_on_thread_count():
    spec = ms.LayerSpec(H=512, I=256, E=8, k=2, seed=54)
    layer = ms.Layer(spec)
    x = ms.tokens(7, spec.H, seed=54)
    ref = oracle.default.moe_layer(layer, x)
    outs = []
    for n in (1, 2, 5):
        p = bv.CpuPool(n)
        assert p.threads == n
        outs.append(_remainder(p, layer, x, np.zeros(spec.E, bool), ref))
        p.close()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def _vq2_layout(codes, scales):
    """The packed VQ2 layout as the header states it, by explicit indices."""
    rows, G = codes.shape
    KB = G // 32
    pc = np.zeros(rows * G, np.uint8)
    ps = np.zeros(scales.size, np.uint16)
    for r in range(rows):
        rt, r16 = divmod(r, 16)
        i, h = r16 % 8, r16 // 8
        for q in range(G):
            kb, g = divmod(q, 32)
            pc[(rt * KB + kb) * 512 + 16 * g + 2 * i + h] = codes[r, q]
        for kb in range(KB):
            ps[(rt * KB + kb) * 16 + r16] = scales[r, kb]
    return pc.reshape(codes.shape), ps.reshape(scales.shape)


def _fp4_layout(codes, scales):
    rows, NB = codes.shape
    KT, KB = NB // 32, NB // 16
    pc = np.zeros(rows * NB, np.uint8)
    ps = np.zeros(scales.size, np.uint8)
    for r in range(rows):
        rt, r16 = divmod(r, 16)
        i, hi = r16 % 8, r16 // 8
        for b in range(NB):
            kt, lb = divmod(b, 32)
            s, w = divmod(lb, 8)
            j, up = w % 4, w // 4
            pc[(rt * KT + kt) * 512 + 16 * (4 * i + j) + 4 * s + 2 * hi + up] = codes[r, b]
        for kb in range(KB):
            ps[(rt * KB + kb) * 16 + r16] = scales[r, kb]
    return pc.reshape(codes.shape), ps.reshape(scales.shape)


def test_host_packers_follow_the_documented_layouts():
    rng = np.random.default_rng(5)
    c = rng.integers(0, 256, size=(32, 64), dtype=np.uint8)       # rows 32, K 256
    s = rng.integers(0, 65536, size=(32, 2), dtype=np.uint16)
    pc, ps = bv.moe_vq2_pack_host(c, s)
    ec, es = _vq2_layout(c, s)
    assert np.array_equal(pc, ec) and np.array_equal(ps, es)
    c4 = rng.integers(0, 256, size=(32, 64), dtype=np.uint8)      # rows 32, K 128
    s4 = rng.integers(110, 130, size=(32, 4), dtype=np.uint8)
    pc, ps = bv.moe_fp4_pack_host(c4, s4)
    ec, es = _fp4_layout(c4, s4)
    assert np.array_equal(pc, ec) and np.array_equal(ps, es)


def test_cpu_argument_checks(pool):
    spec = ms.spec_tiny(1)
    layer = ms.Layer(spec)
    x = ms.tokens(2, spec.H, seed=1)
    ids = np.array([[0, 1], [2, 3]], np.int32)
    w = np.full((2, 2), 0.5, np.float32)
    st = np.zeros(4, np.uint8)
    hx = _host_experts(layer, [0, 1, 2])  # expert 3 has no host buffers
    with pytest.raises(bv.MoeError) as ei:
        bv.moe_cpu_expert_ffn(pool, spec.H, spec.I, layer.codebook, hx, x, ids, w, st, 2)
    assert ei.value.status == bv.MOE_ERR_INVALID_ARG and "null buffer" in str(ei.value)
    bad = ids.copy()
    bad[1, 1] = spec.E
    with pytest.raises(bv.MoeError):
        bv.moe_cpu_expert_ffn(pool, spec.H, spec.I, layer.codebook, hx, x, bad, w, st, 2)
    st2 = st.copy()
    st2[3] = 1  # the pair of expert 3 is the GPU's: expert 3 is not read
    out = bv.moe_cpu_expert_ffn(pool, spec.H, spec.I, layer.codebook, hx, x, ids, w, st2, 2)
    assert out.shape == (2, spec.H)
    with pytest.raises(bv.MoeError) as ei:
        bv.moe_cpu_expert_ffn(pool, 200, spec.I, layer.codebook, hx, x, ids, w, st2, 2)
    assert ei.value.status == bv.MOE_ERR_UNSUPPORTED
