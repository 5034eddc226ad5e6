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
