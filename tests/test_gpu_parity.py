"""GPU parity of the CUDA path against the CPU oracle on small layers: the
tiny workload, ragged per-expert token counts, degenerate shapes, residency,
determinism and the sign-symmetry invariant.  Every call goes through the
C ABI (ctypes)."""
import numpy as np
import pytest

import moe_synth as ms
import oracle
from gpu_common import (assert_close, assert_routing_exact, device_error_word, device_layer, run,
                        torch_cuda, MAX_REL_RMS, MEAN_REL)

pytestmark = pytest.mark.gpu
O = oracle.default


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


def _check_layer(spec, T, seed=0, resident=None):
    layer = ms.Layer(spec)
    x = ms.tokens(T, spec.H, seed=seed)
    res_ids = None if resident is None else np.nonzero(resident)[0]
    dev, keep = device_layer(layer, T, res_ids)
    g = run(dev, x)
    r = O.moe_layer(layer, x, resident=resident)
    assert_routing_exact(g, r)
    res = np.ones(spec.E, bool) if resident is None else resident
    assert np.array_equal(g["status"], res[r["ids"]].ravel().astype(np.uint8))
    assert_close(g["out"], r["partial"], f"T={T} E={spec.E} k={spec.k}")
    assert device_error_word(dev) == 0
    return layer, x, dev, keep, g, r


def test_tiny_layer_full_parity(torch):
    _check_layer(ms.spec_tiny(0), 4)


def test_tiny_layer_fp4_experts(torch):
    spec = ms.spec_tiny(1)
    spec.fp4_top = 3
    _check_layer(spec, 4, seed=1)


@pytest.mark.parametrize("T", [3, 8, 9, 16, 17, 31])
def test_experts_at_chunk_and_tile_boundaries(torch, T):
    """Every token routes to all three experts (E = k = 3), so each expert gets
    exactly T tokens: the FP4 expert's 16-token chunks hold one n8 tile of
    tokens up to 8 and two from 9, with a second chunk from 17; the two VQ2
    experts take the table path at 3 tokens, then the 32-token mma.sync
    chunks (one to four n8 tiles)."""
    spec = ms.LayerSpec(H=512, I=256, E=3, k=3, seed=40 + T, fp4_top=1)
    _check_layer(spec, T, seed=T)


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (37, 4, 2), (5, 16, 3), (64, 8, 8), (3, 1, 1), (17, 32, 1)])
def test_ragged_and_degenerate_shapes(torch, T, E, k):
    spec = ms.LayerSpec(H=256, I=128, E=E, k=k, seed=T + 10 * E + k)
    _check_layer(spec, T, seed=T)


@pytest.mark.parametrize("H,I,T,E,k", [(512, 256, 1, 16, 4), (1024, 640, 2, 64, 8), (1536, 384, 3, 32, 6),
                                        (4096, 2048, 1, 16, 8), (768, 128, 5, 128, 3),
                                        (256, 128, 1, 1024, 32), (512, 256, 2, 64, 32)])  # the largest E and k
def test_single_token_experts_table_path(torch, H, I, T, E, k):
    # experts that get one token go through the activation-table kernels;
    # K-ranges of 1-4 scale blocks (H, I not multiples of 512) included
    spec = ms.LayerSpec(H=H, I=I, E=E, k=k, seed=H + I + T)
    _check_layer(spec, T, seed=T)


@pytest.mark.parametrize("H,I,E,k,fp4_top", [(512, 256, 16, 4, 16), (1280, 384, 64, 8, 64), (768, 640, 128, 3, 128),
                                              (4096, 2048, 256, 8, 52), (1024, 384, 32, 4, 16), (256, 128, 4, 2, 4),
                                              (512, 256, 8, 1, 8), (512, 256, 64, 32, 64)])  # (last: 32 pairs, one group)
def test_fp4_experts_single_token_e2m1_table_path(torch, H, I, E, k, fp4_top):
    # in single-token calls FP4 experts go through the e2m1 table kernels;
    # K-ranges of 2 to 8 tiles of 64 inputs (H, I not multiples of 512)
    # included
    spec = ms.LayerSpec(H=H, I=I, E=E, k=k, seed=H + I + k, zipf_s=1.1, fp4_top=fp4_top)
    _check_layer(spec, 1, seed=k)


def test_fp4_experts_single_token_non_resident_reported(torch):
    spec = ms.LayerSpec(H=512, I=256, E=16, k=8, seed=17, fp4_top=16)
    res = np.zeros(16, bool)
    res[::2] = True
    _check_layer(spec, 1, seed=17, resident=res)


@pytest.mark.parametrize("H,I,T,E,k,fp4_top", [(512, 256, 2, 16, 4, 16), (1280, 384, 3, 64, 8, 64),
                                                (4096, 2048, 2, 256, 8, 52), (768, 640, 3, 32, 6, 16),
                                                (256, 128, 3, 4, 2, 4), (512, 256, 3, 16, 8, 8)])
def test_fp4_experts_two_and_three_token_calls(torch, H, I, T, E, k, fp4_top):
    # two tokens: the FP4 experts take the e2m1 tables, one pair per token,
    # the pairs grouped by token (experts with two tokens among them), and no
    # mma.sync launch is needed; three tokens: mma.sync for the FP4 experts,
    # tables for the VQ2 ones
    spec = ms.LayerSpec(H=H, I=I, E=E, k=k, seed=H + I + T + k, zipf_s=1.1, fp4_top=fp4_top)
    _check_layer(spec, T, seed=T + k)


@pytest.mark.parametrize("fp4_top", [0, 16])
def test_single_token_no_resident_expert(torch, fp4_top):
    # a single-token call whose routed experts are all missing (VQ2-only
    # table: the self-scheduling table kernels; with FP4 experts: the
    # schedule and the e2m1 kernels): every pair reported, output zero
    spec = ms.LayerSpec(H=512, I=256, E=16, k=4, seed=23, fp4_top=fp4_top)
    layer = ms.Layer(spec)
    x = ms.tokens(1, spec.H, seed=23)
    routed = set(O.moe_layer(layer, x)["ids"].ravel().tolist())
    # with FP4 experts, one FP4 expert the token does not route to is resident
    # (the table then holds FP4 experts, which selects the schedule path)
    keep_ids = [e for e in range(spec.E) if e not in routed][:1] if fp4_top else []
    dev, keep = device_layer(layer, 1, np.array(keep_ids, np.int64))
    g = run(dev, x)
    assert (g["status"] == 0).all()
    assert (g["out"] == 0).all()
    assert device_error_word(dev) == 0


def test_fp4_table_pairs_fused_scatter_matches_per_pair(torch):
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=1280, I=640, E=64, k=8, seed=31, fp4_top=64)
    layer = ms.Layer(spec)
    x = ms.tokens(2, spec.H, seed=31)  # (two token groups of e2m1 pairs)
    dev, keep = device_layer(layer, 2)
    g = run(dev, x)
    xt = torch.from_numpy(x).view(torch.bfloat16).cuda()
    out = torch.zeros(2, spec.H, dtype=torch.float32, device="cuda")
    dev.route(xt)
    dev.experts(xt, bv.MOE_FUSED_SCATTER, out)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert np.abs(o - g["out"]).max() <= 1e-5 * np.abs(g["out"]).max()


def test_wider_hidden_mixed_formats(torch):
    spec = ms.LayerSpec(H=1024, I=384, E=12, k=4, seed=21, zipf_s=1.1, fp4_top=4)
    _check_layer(spec, 24, seed=3)


def test_renormalize_off(torch):
    spec = ms.LayerSpec(H=256, I=128, E=16, k=4, seed=5, renormalize=0)
    _check_layer(spec, 9, seed=5)


def test_non_resident_experts_are_reported_not_substituted(torch):
    spec = ms.LayerSpec(H=512, I=256, E=16, k=4, seed=7, zipf_s=1.1, fp4_top=3)
    res = np.zeros(16, bool)
    res[[0, 3, 4, 9, 10, 15]] = True
    layer, x, dev, keep, g, r = _check_layer(spec, 12, seed=7, resident=res)
    # rows of ypair for skipped pairs are left untouched
    P = 12 * 4
    dev.ypair[:P].fill_(float("nan"))
    g2 = run(dev, x)
    skipped = g2["status"] == 0
    assert skipped.any() and (~skipped).any()
    assert np.isnan(g2["ypair"][g2["pair_to_sorted"][skipped]]).all()
    assert not np.isnan(g2["ypair"][g2["pair_to_sorted"][~skipped]]).any()
    # GPU partial + oracle remainder = oracle whole layer
    assert_close(g2["out"] + r["remainder"], r["out"], "partial + remainder")


def test_per_pair_is_deterministic_and_slot_reload_bit_identical(torch):
    spec = ms.LayerSpec(H=512, I=256, E=8, k=2, seed=8)
    layer = ms.Layer(spec)
    x = ms.tokens(16, 512, seed=8)
    dev, keep = device_layer(layer, 16)
    a = run(dev, x)
    b = run(dev, x)
    assert np.array_equal(a["out"].view(np.uint32), b["out"].view(np.uint32))
    # evict and re-set every expert from freshly packed buffers: same bits
    import bit_vq_routed_gb300 as bv
    for e in range(8):
        dev.evict(e)
    for e in range(8):
        ex = layer.expert(e)
        pc, ps = bv.layer.upload_expert(ex.fmt, ex.codes, ex.scales)
        dev.set_expert(e, ex.fmt, pc, ps)
        keep[e] = (pc, ps)
    c = run(dev, x)
    assert np.array_equal(a["ypair"].view(np.uint32), c["ypair"].view(np.uint32))


def test_fused_scatter_matches_per_pair(torch):
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=512, I=256, E=8, k=3, seed=9)
    layer = ms.Layer(spec)
    x = ms.tokens(20, 512, seed=9)
    dev, keep = device_layer(layer, 20)
    g = run(dev, x)
    xt = torch.from_numpy(x).view(torch.bfloat16).cuda()
    out = torch.zeros(20, 512, dtype=torch.float32, device="cuda")
    dev.route(xt)
    dev.experts(xt, bv.MOE_FUSED_SCATTER, out)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert np.abs(o - g["out"]).max() <= 1e-5 * np.abs(g["out"]).max()


@pytest.mark.parametrize("m", [1, 2])
def test_sign_flip_negates_expert_output_bit_exactly(torch, m):
    # sign-symmetric codebook: flipping every sign bit of the up (m=1) or
    # down (m=2) codes of every expert negates each per-pair y exactly
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=512, I=256, E=4, k=2, seed=12)
    layer = ms.Layer(spec)
    x = ms.tokens(6, 512, seed=12)
    dev, keep = device_layer(layer, 6)
    a = run(dev, x)
    for e in range(4):
        ex = layer.expert(e)
        codes = list(ex.codes)
        codes[m] = codes[m] ^ 0x80
        pc, ps = bv.layer.upload_expert(ex.fmt, codes, ex.scales)
        dev.set_expert(e, ex.fmt, pc, ps)
        keep[e] = (pc, ps)
    b = run(dev, x)
    assert np.array_equal(b["ypair"], -a["ypair"])


def test_empty_batch_is_a_no_op(torch):
    spec = ms.spec_tiny(0)
    layer = ms.Layer(spec)
    dev, keep = device_layer(layer, 4)
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    out = dev.forward(x)
    torch.cuda.synchronize()
    assert out.shape == (0, 256)


def test_workspace_too_small_is_rejected(torch):
    import bit_vq_routed_gb300 as bv
    spec = ms.spec_tiny(0)
    layer = ms.Layer(spec)
    dev, keep = device_layer(layer, 4)
    x = torch.from_numpy(ms.tokens(4, 256, 0)).view(torch.bfloat16).cuda()
    dev.route(x)
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(bv.MoeError) as ei:
        bv.moe_vq2_expert_ffn(dev.table, x, dev.offsets, dev.sorted_pair[:8], dev.weights[:4], 2,
                              bv.MOE_PER_PAIR, dev.ypair[:8], dev.pair_status[:8], small)
    assert ei.value.status == bv.MOE_ERR_WORKSPACE


@pytest.mark.parametrize("T,resident_frac,bf16", [(1, 1.0, False), (1, 0.5, True), (1, 0.0, False), (6, 0.7, True)])
def test_expert_ffn_combine_matches_separate_calls(torch, T, resident_frac, bf16):
    # moe_vq2_expert_ffn_combine == moe_vq2_expert_ffn (per pair) + moe_combine,
    # bit for bit (one token: the combine runs inside the expert kernels)
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=1024, I=512, E=32, k=8, seed=31 + T)
    layer = ms.Layer(spec)
    rng = np.random.default_rng(T)
    res_ids = np.nonzero(rng.random(32) < resident_frac)[0] if resident_frac < 1 else None
    dev, keep = device_layer(layer, T, res_ids)
    x = torch.from_numpy(ms.tokens(T, 1024, seed=T)).view(torch.bfloat16).cuda()
    P = T * 8
    dev.route(x)
    dev.experts(x, bv.MOE_PER_PAIR)
    ref32 = torch.empty(T, 1024, dtype=torch.float32, device="cuda")
    ref16 = torch.empty(T, 1024, dtype=torch.bfloat16, device="cuda")
    bv.moe_combine(dev.ypair[:P], dev.pair_to_sorted[:P], dev.weights[:T], dev.pair_status[:P], 8, ref32,
                   ref16.view(torch.int16) if bf16 else None)
    y_ref = dev.ypair[:P].clone()
    st_ref = dev.pair_status[:P].clone()
    out32 = torch.full((T, 1024), float("nan"), dtype=torch.float32, device="cuda")
    out16 = torch.zeros(T, 1024, dtype=torch.bfloat16, device="cuda")
    dev.experts_combine(x, out32, out16.view(torch.int16) if bf16 else None)
    torch.cuda.synchronize()
    assert torch.equal(dev.pair_status[:P], st_ref)
    done = st_ref.bool()
    assert torch.equal(dev.ypair[:P][done].view(torch.int32), y_ref[done].view(torch.int32))
    assert torch.equal(out32.view(torch.int32), ref32.view(torch.int32))
    if bf16:
        assert torch.equal(out16.view(torch.int16), ref16.view(torch.int16))
    assert device_error_word(dev) == 0
