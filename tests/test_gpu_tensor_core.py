"""GPU parity of the tcgen05 (tensor-core) path: experts that receive at
least 32 tokens in one call run FC1 and FC2 as tcgen05.mma contractions over
fp16 weight tiles decoded into shared memory.  Shapes cover ragged token
chunks (counts not a multiple of 128), several weight-row tiles, mixed FP4
experts (which stay on the other path) and fused scatter mode."""
import numpy as np
import pytest

import moe_synth as ms
import oracle
from gpu_common import assert_close, assert_routing_exact, device_error_word, device_layer, run, torch_cuda

pytestmark = pytest.mark.gpu
O = oracle.default


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


@pytest.mark.parametrize("H,I,T,E,k,fp4", [(256, 128, 160, 4, 2, 0), (1024, 512, 300, 8, 4, 0),
                                            (512, 256, 200, 6, 3, 2), (2048, 1024, 96, 2, 2, 0)])
def test_tensor_core_experts_match_oracle(torch, H, I, T, E, k, fp4):
    spec = ms.LayerSpec(H=H, I=I, E=E, k=k, seed=H + T, fp4_top=fp4)
    layer = ms.Layer(spec)
    x = ms.tokens(T, H, seed=T)
    dev, keep = device_layer(layer, T)
    g = run(dev, x)
    r = O.moe_layer(layer, x)
    assert_routing_exact(g, r)
    counts = np.diff(g["offsets"])
    assert (counts[layer.formats == ms.FMT_VQ2] >= 32).any()  # the tensor-core path is exercised
    assert_close(g["out"], r["out"], f"H={H} I={I} T={T}")
    assert device_error_word(dev) == 0


def test_tensor_core_fused_scatter(torch):
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=512, I=256, E=4, k=2, seed=77)
    layer = ms.Layer(spec)
    x = ms.tokens(150, 512, seed=77)
    dev, keep = device_layer(layer, 150)
    g = run(dev, x)
    xt = torch.from_numpy(x).view(torch.bfloat16).cuda()
    out = torch.zeros(150, 512, dtype=torch.float32, device="cuda")
    dev.route(xt)
    dev.experts(xt, bv.MOE_FUSED_SCATTER, out)
    torch.cuda.synchronize()
    assert np.abs(out.cpu().numpy() - g["out"]).max() <= 1e-5 * np.abs(g["out"]).max()
    assert device_error_word(dev) == 0


def test_every_path_in_one_large_call(torch):
    """A call of 160 tokens (at least the split threshold of 128) whose routing
    gives VQ2 experts in every band: 1-3 tokens (activation table), 4-16
    (16-token mma.sync configuration), 17-31 (32-token configuration) and
    32 or more (tcgen05), and an FP4 expert (16-token configuration, in the
    same launch as the small VQ2 experts)."""
    spec = ms.LayerSpec(H=512, I=256, E=48, k=4, seed=91, zipf_s=1.1, fp4_top=1)
    layer = ms.Layer(spec)
    x = ms.tokens(160, 512, seed=91)
    dev, keep = device_layer(layer, 160)
    g = run(dev, x)
    r = O.moe_layer(layer, x)
    assert_routing_exact(g, r)
    counts = np.diff(g["offsets"])
    vq = layer.formats == ms.FMT_VQ2
    for lo, hi in [(1, 3), (4, 16), (17, 31), (32, 160)]:
        assert ((counts >= lo) & (counts <= hi) & vq).any(), (lo, hi)
    assert (counts[~vq] > 0).any()
    assert_close(g["out"], r["out"], "every path, 160 tokens")
    assert device_error_word(dev) == 0
