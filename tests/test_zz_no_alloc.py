"""The scratch-free expert FFN (moe_vq2_expert_ffn_noalloc) is for callers
that cannot allocate device memory at the point where they run the layer
(a host that owns all device memory through its own arena, a serving loop
that must not allocate mid-step).  It must give what moe_vq2_expert_ffn gives
with a caller workspace.  Two calls in a row, with different tokens, check
that the shared static scratch carries nothing over from one call to the
next.  This file is collected last so a failing run has run everything else
first; it also passes alone in a fresh process."""
import numpy as np
import pytest

import moe_synth as ms
from gpu_common import assert_close, device_layer, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


def _both(torch, dev, x_bits, mode):
    import bit_vq_routed_gb300 as bv
    x = torch.from_numpy(np.ascontiguousarray(x_bits)).view(torch.bfloat16).cuda()
    T = x.shape[0]
    P = T * dev.k
    dev.route(x)
    shape = (P, dev.H) if mode == bv.MOE_PER_PAIR else (T, dev.H)
    ref = torch.zeros(shape, dtype=torch.float32, device="cuda")
    got = torch.zeros(shape, dtype=torch.float32, device="cuda")
    st_ref = torch.zeros(P, dtype=torch.uint8, device="cuda")
    st_got = torch.zeros(P, dtype=torch.uint8, device="cuda")
    bv.moe_vq2_expert_ffn(dev.table, x, dev.offsets, dev.sorted_pair[:P], dev.weights[:T], dev.k, mode,
                          ref, st_ref, dev.ws)
    bv.moe_vq2_expert_ffn_noalloc(dev.table, x, dev.offsets, dev.sorted_pair[:P], dev.weights[:T], dev.k,
                                  mode, got, st_got)
    torch.cuda.synchronize()
    return ref.cpu().numpy(), got.cpu().numpy(), st_ref.cpu().numpy(), st_got.cpu().numpy()


@pytest.mark.parametrize("mode_name", ["per_pair", "fused_scatter"])
def test_noalloc_matches_workspace_entry_point_twice(torch, mode_name):
    import bit_vq_routed_gb300 as bv
    mode = bv.MOE_PER_PAIR if mode_name == "per_pair" else bv.MOE_FUSED_SCATTER
    spec = ms.LayerSpec(H=4096, I=2048, E=16, k=4, seed=31, zipf_s=1.1, fp4_top=3)
    layer = ms.Layer(spec)
    dev, keep = device_layer(layer, 8)
    for call in range(2):
        x = ms.tokens(8 - 3 * call, spec.H, seed=31, stream=call)
        ref, got, st_ref, st_got = _both(torch, dev, x, mode)
        assert np.array_equal(st_ref, st_got)
        assert_close(got, ref, f"noalloc call {call}")


def test_noalloc_single_token_vq2_only_twice(torch):
    """One token on a table of VQ2 experts only: the path without a schedule
    kernel, whose table kernels keep their counters, K-range partial sums
    and error word in the scratch."""
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=4096, I=2048, E=16, k=4, seed=37, fp4_top=0)
    layer = ms.Layer(spec)
    dev, keep = device_layer(layer, 1)
    for call in range(2):
        x = ms.tokens(1, spec.H, seed=37, stream=call)
        ref, got, st_ref, st_got = _both(torch, dev, x, bv.MOE_PER_PAIR)
        assert np.array_equal(st_ref, st_got)
        assert st_got.all()
        assert_close(got, ref, f"single-token noalloc call {call}")


def test_noalloc_rejects_sizes_beyond_its_scratch(torch):
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=256, I=2048, E=8, k=8, seed=1)
    layer = ms.Layer(spec)
    dev, keep = device_layer(layer, 1)
    T = 4096  # needs T*k*I*4 = 256 MiB of scratch, above the fixed 64 MiB
    assert bv.moe_vq2_expert_ffn_workspace_size(T, 8, 8, 256, 2048) > bv.MOE_NOALLOC_SCRATCH_BYTES
    x = torch.zeros(T, 256, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(T, 8, dtype=torch.float32, device="cuda")
    sp = torch.zeros(T * 8, dtype=torch.int32, device="cuda")
    out = torch.zeros(T * 8, 256, dtype=torch.float32, device="cuda")
    st = torch.zeros(T * 8, dtype=torch.uint8, device="cuda")
    with pytest.raises(bv.MoeError) as ei:
        bv.moe_vq2_expert_ffn_noalloc(dev.table, x, dev.offsets, sp, w, 8, bv.MOE_PER_PAIR, out, st)
    assert ei.value.status == bv.MOE_ERR_UNSUPPORTED
    assert "scratch" in str(ei.value)
