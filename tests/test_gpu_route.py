"""moe_route (router logits, top-k softmax and permutation in one call; one
kernel for small batches) gives bit for bit what the three separate calls
give, and leaves its workspace counter at zero."""
import numpy as np
import pytest

import moe_synth as ms
from gpu_common import torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


@pytest.mark.parametrize("T,H,E,k,renorm,with_bias", [
    (1, 4096, 256, 8, 1, True), (4, 256, 8, 2, 1, False), (32, 4096, 256, 8, 1, True),
    (64, 1024, 1024, 32, 0, True), (7, 512, 48, 5, 0, False), (16, 2048, 128, 1, 1, True),
    (64, 256, 8, 8, 1, False),  # 512 pairs (two 256-pair chunks), every expert in every warp
    (40, 512, 32, 16, 0, True), (64, 4096, 256, 16, 1, True),  # 640 and 1024 pairs
    (8, 512, 64, 32, 1, True),  # the one-kernel limit: 8 tokens, 256 pairs
    (1, 4096, 1024, 32, 0, True), (1, 512, 48, 5, 1, False),  # one token over a cluster: 1024 and 48 experts
    (1, 8192, 300, 8, 1, True),  # one token, two weight batches per lane (H > 4096), ragged expert count
    (100, 512, 64, 4, 1, True),  # above the one-kernel limit: the three-step fallback
    # from 8192 pairs moe_route sorts over 1024-pair chunks on many CTAs (its
    # workspace), route_stepwise on one CTA (no workspace): the same bits
    (1100, 256, 64, 8, 1, True),    # 8800 pairs: nine chunks, the last one ragged
    (2048, 256, 256, 8, 1, False),  # 16384 pairs: whole chunks
    (1500, 256, 1024, 8, 0, True),  # 1024 experts: 128 KB of per-warp counts per chunk
])
def test_route_matches_stepwise(torch, T, H, E, k, renorm, with_bias):
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=H, I=128, E=E, k=k, seed=T + E + k, zipf_s=1.1 if E >= 64 else None, renormalize=renorm)
    layer = ms.Layer(spec)
    bias = layer.bias if with_bias else None
    dev = bv.MoELayer(H, 128, E, k, T, layer.codebook, layer.w_router, bias, renorm)
    x = torch.from_numpy(ms.tokens(T, H, seed=T)).view(torch.bfloat16).cuda()
    outs = []
    for fused in (False, True):
        for buf in (dev.logits, dev.weights):
            buf.fill_(float("nan"))
        for buf in (dev.ids, dev.offsets, dev.sorted_pair, dev.pair_to_sorted):
            buf.fill_(-7)
        (dev.route if fused else dev.route_stepwise)(x)
        torch.cuda.synchronize()
        P = T * k
        outs.append([a.cpu().numpy().copy() for a in (dev.logits[:T], dev.ids[:T], dev.weights[:T], dev.offsets,
                                                       dev.sorted_pair[:P], dev.pair_to_sorted[:P])])
    for a, b in zip(*outs):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    assert int(dev.route_ws.view(torch.int32)[0].item()) == 0


def test_route_repeated_calls_stay_consistent(torch):
    # the counter returns to zero, so back-to-back calls (and graph replays) work
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=1024, I=128, E=64, k=4, seed=3)
    layer = ms.Layer(spec)
    dev = bv.MoELayer(1024, 128, 64, 4, 8, layer.codebook, layer.w_router, layer.bias)
    xs = [torch.from_numpy(ms.tokens(8, 1024, seed=s)).view(torch.bfloat16).cuda() for s in range(3)]
    ref = []
    for x in xs:
        dev.route_stepwise(x)
        ref.append(dev.sorted_pair[:32].cpu().numpy().copy())
    g = torch.cuda.CUDAGraph()
    xg = xs[0].clone()
    with torch.cuda.graph(g):
        dev.route(xg)
    for rep in range(2):
        for x, r in zip(xs, ref):
            xg.copy_(x)
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(dev.sorted_pair[:32].cpu().numpy(), r)


@pytest.mark.parametrize("T,E,k,zero_first", [(1, 256, 8, True), (1, 256, 8, False), (1, 48, 5, False),
                                              (4, 64, 8, True), (40, 64, 8, True), (3, 1024, 32, True)])
def test_equal_logits_go_to_the_lower_id(torch, T, E, k, zero_first):
    # Router rows duplicated in pairs give bit-equal logits (one fixed summation
    # order); all-zero tokens make every logit equal.  Every routing path (one
    # token over a cluster, the one-kernel path up to 8 tokens, the three steps
    # above) must pick the lower id of equal logits, as the oracle does.
    import oracle
    import bit_vq_routed_gb300 as bv
    H = 512
    spec = ms.LayerSpec(H=H, I=128, E=E, k=k, seed=50 + T)
    layer = ms.Layer(spec)
    w = layer.w_router.copy()
    rng = np.random.default_rng(E + T)
    perm = rng.permutation(E)
    for a, b in zip(perm[0::2], perm[1::2]):  # expert b gets expert a's router row
        w[b] = w[a]
    x = ms.tokens(T, H, seed=60 + T)
    if zero_first:
        x[0] = 0  # token 0: every logit equal
    O = oracle.default
    lg = O.router_logits(x, w, None)
    ids_ref, w_ref = O.route_topk(lg, k, 1)
    if zero_first:
        assert (ids_ref[0] == np.arange(k)).all()
    else:  # the duplicated rows do tie inside this token's selection
        sel = lg[0, ids_ref[0]]
        assert len(np.unique(sel)) < k
    off_ref, sp_ref, p2s_ref = O.permute(ids_ref, E)
    dev = bv.MoELayer(H, 128, E, k, T, layer.codebook, w, None, 1)
    xd = torch.from_numpy(x).view(torch.bfloat16).cuda()
    for fused in (False, True):
        dev.ids.fill_(-7)
        (dev.route if fused else dev.route_stepwise)(xd)
        torch.cuda.synchronize()
        P = T * k
        assert np.array_equal(dev.logits[:T].cpu().numpy().view(np.uint32), lg.view(np.uint32))
        assert np.array_equal(dev.ids[:T].cpu().numpy(), ids_ref), f"fused={fused}"
        assert np.abs(dev.weights[:T].cpu().numpy() - w_ref).max() <= 1e-6
        assert np.array_equal(dev.offsets.cpu().numpy(), off_ref)
        assert np.array_equal(dev.sorted_pair[:P].cpu().numpy(), sp_ref)
        assert np.array_equal(dev.pair_to_sorted[:P].cpu().numpy(), p2s_ref)
        if zero_first:  # equal logits get equal weights
            assert np.allclose(dev.weights[0].cpu().numpy(), 1.0 / k, rtol=0, atol=1e-7)
