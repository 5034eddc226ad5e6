"""The GPU and the host's cores computing one layer together (Tandem-vLLM
page, "How it works": experts that miss the GPU cache are computed by the
CPU in parallel with the GPU): the mixed FP4/VQ2 decode batch of 8 with only
the 96 most routed experts in the GPU slot table; the GPU's partial output
plus the CPU's remainder (moe_cpu_expert_ffn, overlapped with the GPU call)
must equal the oracle's whole layer.  Also: the host packers write the same
bytes as the device packers."""
import numpy as np
import pytest

import moe_synth as ms
import oracle
from gpu_common import assert_close, device_layer, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


def test_host_packers_equal_device_packers(torch):
    import bit_vq_routed_gb300 as bv
    rng = np.random.default_rng(9)
    for fmt, shape, sshape, sdt in [(bv.MOE_FMT_VQ2, (64, 512), (64, 16), np.uint16),
                                    (bv.MOE_FMT_FP4, (64, 512), (64, 32), np.uint8)]:
        c = rng.integers(0, 256, size=shape, dtype=np.uint8)
        s = rng.integers(100, 140, size=sshape).astype(sdt)
        hc, hs = (bv.moe_vq2_pack_host if fmt == bv.MOE_FMT_VQ2 else bv.moe_fp4_pack_host)(c, s)
        dc = torch.empty(shape, dtype=torch.uint8, device="cuda")
        dt = torch.float16 if fmt == bv.MOE_FMT_VQ2 else torch.uint8
        ds = torch.empty(sshape, dtype=dt, device="cuda")
        src_c = torch.from_numpy(c).cuda()
        src_s = torch.from_numpy(s.view(np.int16) if sdt == np.uint16 else s).cuda()
        if fmt == bv.MOE_FMT_VQ2:
            bv.moe_vq2_pack(src_c, src_s.view(torch.float16), dc, ds)
        else:
            bv.moe_fp4_pack(src_c, src_s, dc, ds)
        torch.cuda.synchronize()
        assert np.array_equal(dc.cpu().numpy(), hc)
        assert np.array_equal(ds.cpu().view(torch.int16 if fmt == bv.MOE_FMT_VQ2 else torch.uint8).numpy()
                              .view(sdt), hs)


def test_tandem_mixed_b8_96_resident_matches_oracle(torch):
    import bit_vq_routed_gb300 as bv
    layer = ms.Layer(ms.spec_decode(0, zipf_s=1.1, fp4_top=52))
    s = layer.spec
    T = 8
    res = np.zeros(s.E, bool)
    res[ms.most_popular(layer, 96)] = True
    dev, keep = device_layer(layer, T, resident=np.nonzero(res)[0])
    hx = bv.HostExperts(s.E)
    for e in np.nonzero(~res)[0]:
        ex = layer.expert(int(e))
        hx.set(int(e), *bv.host_pack_expert(ex.fmt, ex.codes, ex.scales))
    pool = bv.CpuPool(0)
    step = bv.TandemForward(dev, pool, hx, T)
    outs = []
    # two steps in a row; token batches whose routing names non-resident
    # experts (3 pairs each; most batches of 8 tokens name one or none)
    for call, seed in enumerate((305, 312)):
        x = ms.tokens(T, s.H, seed=seed)
        xh = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
        out = step.step(xh)
        torch.cuda.synchronize()
        got = out.cpu().numpy().copy()
        ref = oracle.default.moe_layer(layer, x, resident=res)
        assert np.array_equal(dev.ids[:T].cpu().numpy(), ref["ids"])
        st = dev.pair_status[:T * s.k].cpu().numpy()
        sp = dev.sorted_pair[:T * s.k].cpu().numpy()
        want = np.empty(T * s.k, np.uint8)
        want[sp] = res[ref["ids"].ravel()[sp]]
        assert np.array_equal(st, want)  # the GPU skipped exactly the pairs the CPU took
        assert step.last["cpu_pairs"] == int((~res[ref["ids"]]).sum()) > 0
        assert_close(got, ref["out"], f"GPU partial + CPU remainder, step {call}")
        outs.append(got)
    pool.close()
