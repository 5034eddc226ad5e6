"""GraphedStep: one CUDA graph per step over several layers, with the
host-to-device copy of the tokens and the device-to-host copy of the outputs
inside the graph, gives the eager forward's outputs bit for bit."""
import numpy as np
import pytest

import moe_synth as ms
from gpu_common import device_layer, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


@pytest.mark.parametrize("T", [1, 5])
def test_graphed_step_matches_eager_layers(torch, T):
    import bit_vq_routed_gb300 as bv
    specs = [ms.LayerSpec(H=512, I=256, E=16, k=4, seed=70 + L, layer=L) for L in range(3)]
    layers = [ms.Layer(s) for s in specs]
    devs, keeps = zip(*[device_layer(layer, T) for layer in layers])
    toks = [np.stack([ms.tokens(T, 512, seed=80 + b, layer=L) for L in range(3)]) for b in range(2)]
    host_in = [torch.from_numpy(t).view(torch.bfloat16).pin_memory() for t in toks]
    host_out = torch.zeros(3, T, 512, dtype=torch.float32).pin_memory()
    steps = [bv.GraphedStep(devs, h, host_out) for h in host_in]
    for b in (0, 1, 0):
        host_out.zero_()
        steps[b].replay()
        torch.cuda.synchronize()
        for L, dev in enumerate(devs):
            ref = dev.forward(torch.from_numpy(toks[b][L]).view(torch.bfloat16).cuda()).cpu().numpy()
            assert np.array_equal(host_out[L].numpy().view(np.uint32), ref.view(np.uint32)), (b, L)
    with pytest.raises(ValueError):
        bv.GraphedStep(devs, torch.zeros(3, T, 512, dtype=torch.bfloat16), host_out)


@pytest.mark.parametrize("T", [1, 5])
def test_pipelined_steps_match_eager_layers(torch, T):
    """PipelinedSteps: the copies of a step overlap the neighbouring steps'
    layers (two copy streams, double-buffered device tokens and outputs); every
    step's outputs still equal the eager forward's bit for bit."""
    import bit_vq_routed_gb300 as bv
    specs = [ms.LayerSpec(H=512, I=256, E=16, k=4, seed=70 + L, layer=L) for L in range(3)]
    layers = [ms.Layer(s) for s in specs]
    devs, keeps = zip(*[device_layer(layer, T) for layer in layers])
    n = 5
    toks = [np.stack([ms.tokens(T, 512, seed=90 + b, layer=L) for L in range(3)]) for b in range(n)]
    host_in = [torch.from_numpy(t).view(torch.bfloat16).pin_memory() for t in toks]
    host_out = [torch.zeros(3, T, 512, dtype=torch.float32).pin_memory() for _ in range(n)]
    pipe = bv.PipelinedSteps(devs, T)
    for b in range(n):  # enqueued back to back, one synchronisation at the end
        pipe.step(host_in[b], host_out[b])
    pipe.join()
    torch.cuda.synchronize()
    for b in range(n):
        for L, dev in enumerate(devs):
            ref = dev.forward(torch.from_numpy(toks[b][L]).view(torch.bfloat16).cuda()).cpu().numpy()
            assert np.array_equal(host_out[b][L].numpy().view(np.uint32), ref.view(np.uint32)), (b, L)
