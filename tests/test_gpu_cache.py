"""The GPU as an expert cache over a host-resident base (vLLM-Moet page,
"2-bit experts on vLLM v0.24.0", "Experts beyond VRAM": a miss is fetched
and the step's graph replayed, bit-identical to a resident forward).

Each step replays the layer's routing graph, reads the routed ids back, has
the cache fetch the misses from page-locked host copies into its slots, and
replays the expert graph; its outputs must equal, bit for bit, those of a
layer with every expert resident.  The resident layer itself
is held to the CPU oracle by the parity tests; one step here is checked
against the oracle too."""
import numpy as np
import pytest

import moe_synth as ms
import oracle
from gpu_common import assert_close, device_error_word, device_layer, experts_fn, run, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


def _cached(layer, T, slots, fmt_for_slots):
    import torch
    import bit_vq_routed_gb300 as bv
    s = layer.spec
    dev = bv.MoELayer(s.H, s.I, s.E, s.k, T, layer.codebook, layer.w_router, layer.bias, s.renormalize)
    slot_bytes = bv.moe_expert_cache_slot_bytes(s.H, s.I, fmt_for_slots)
    # poisoned slots: 0xFF bytes are NaN as fp16 scales, so any byte a fetch
    # failed to overwrite would show in the outputs
    pool = torch.full((slots * slot_bytes,), 0xFF, dtype=torch.uint8, device="cuda")
    cache = bv.ExpertCache(dev.table, pool, slot_bytes)
    f = experts_fn(layer)
    for e in range(s.E):  # even ids: one host block in the slot's layout; odd ids: six buffers
        fmt, codes, scales = f(e)
        if e % 2 == 0:
            cache.set_host_image(e, fmt, bv.host_expert_image(fmt, codes, scales))
        else:
            hc, hs = bv.host_expert(fmt, codes, scales)
            cache.set_host(e, fmt, hc, hs)
    return dev, cache, bv.MissFetchForward(dev, cache, T)


def _steps(spec, T, slots, n_steps, fmt_for_slots=0, seed0=100):
    import torch
    layer = ms.Layer(spec)
    ref, keep = device_layer(layer, T)
    dev, cache, mf = _cached(layer, T, slots, fmt_for_slots)
    P = T * spec.k
    for i in range(n_steps):
        x = ms.tokens(T, spec.H, seed=seed0 + i)
        r = run(ref, x)
        out = mf.step(torch.from_numpy(x).view(torch.bfloat16).cuda())
        torch.cuda.synchronize()
        assert np.array_equal(dev.ids[:T].cpu().numpy(), r["ids"])
        assert (dev.pair_status[:P].cpu().numpy() == 1).all(), f"step {i}: a pair left non-resident"
        assert np.array_equal(dev.ypair[:P].cpu().numpy().view(np.uint32), r["ypair"].view(np.uint32)), i
        assert np.array_equal(out.cpu().numpy().view(np.uint32), r["out"].view(np.uint32)), i
    assert device_error_word(dev) == 0
    return layer, x, out.cpu().numpy(), dev, cache, mf


def test_single_token_misses_fetched_bit_identical(torch):
    # decode shapes, 24 experts in host memory, 10 slots for top-8: most steps
    # evict; one graph captured for all steps
    spec = ms.LayerSpec(H=4096, I=2048, E=24, k=8, seed=31)
    layer, x, out, dev, cache, mf = _steps(spec, T=1, slots=10, n_steps=8)
    st = cache.stats()
    assert st["misses"] > 10 and st["unplaced"] == 0
    assert st["bytes_fetched"] == st["misses"] * 6_684_672
    assert mf.captures == 1 and mf.fetch_steps >= 2 and mf.steps == 8
    held = [e for e in range(24) if cache.slot_of(e) >= 0]
    assert len(held) == 10
    # the last step against the CPU oracle
    r = oracle.default.moe_layer(layer, x)
    assert_close(out, r["out"], "cached layer vs oracle")


def test_small_batch_misses_fetched_bit_identical(torch):
    # four tokens at top-4: experts with 1..4 tokens (table and mma.sync kernels)
    spec = ms.LayerSpec(H=1024, I=512, E=24, k=4, seed=32)
    _, _, _, dev, cache, mf = _steps(spec, T=4, slots=16, n_steps=8)
    st = cache.stats()
    assert st["misses"] >= 16 and st["hits"] > 0
    assert mf.captures == 1


def test_mixed_formats_recapture_and_bit_identical(torch):
    # FP4 experts among the VQ2 ones: the first fetched FP4 expert changes the
    # expert-FFN call's kernel choice, so the graph is captured again once
    spec = ms.LayerSpec(H=1024, I=512, E=16, k=4, seed=33, zipf_s=1.1, fp4_top=4)
    _, _, _, dev, cache, mf = _steps(spec, T=2, slots=8, n_steps=8, fmt_for_slots=1)
    assert mf.captures >= 2
    assert cache.stats()["misses"] >= 8


def test_overflowing_step_reports_unplaced_pairs(torch):
    # 2 slots for a top-4 token: two experts stay out, their pairs are reported
    # (status 0), and the output is the resident part of the layer
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=512, I=256, E=8, k=4, seed=34)
    layer = ms.Layer(spec)
    dev, cache, mf = _cached(layer, 1, 2, bv.MOE_FMT_VQ2)
    x = ms.tokens(1, spec.H, seed=5)
    out = mf.step(torch.from_numpy(x).view(torch.bfloat16).cuda())
    st = dev.pair_status[:4].cpu().numpy()
    assert st.sum() == 2 and cache.stats()["unplaced"] == 2
    ids = dev.ids[:1].cpu().numpy().ravel()
    resident = np.zeros(spec.E, bool)
    resident[[e for e in range(spec.E) if cache.slot_of(e) >= 0]] = True
    assert np.array_equal(st, resident[ids].astype(np.uint8))
    r = oracle.default.moe_layer(layer, x, resident=resident)
    assert_close(out.cpu().numpy(), r["partial"], "resident part")


def test_caller_set_entries_are_left_alone(torch):
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=512, I=256, E=8, k=2, seed=35)
    layer = ms.Layer(spec)
    dev, cache, mf = _cached(layer, 1, 2, bv.MOE_FMT_VQ2)
    ex = layer.expert(3)
    pc, ps = bv.layer.upload_expert(ex.fmt, ex.codes, ex.scales)
    dev.set_expert(3, ex.fmt, pc, ps)
    r = cache.fetch([3, 4])
    assert r["n_fetched"] == 1 and cache.slot_of(3) == -1 and cache.slot_of(4) == 0
    # the caller evicts a cached expert: its slot is free for the next miss
    dev.evict(4)
    r = cache.fetch([5, 6])
    assert r["n_fetched"] == 2 and sorted([cache.slot_of(5), cache.slot_of(6)]) == [0, 1]
    with pytest.raises(bv.MoeError):
        cache.fetch([99])
    # a pageable host buffer is refused by the library's own check
    import ctypes
    pageable = torch.zeros(1 << 16, dtype=torch.uint8)
    d = bv._ExpertDesc()
    d.format = bv.MOE_FMT_VQ2
    for m in range(3):
        d.codes[m] = d.scales[m] = pageable.data_ptr()
    assert cache.lib.moe_expert_cache_set_host(cache.handle, 1, ctypes.byref(d)) == bv.MOE_ERR_UNSUPPORTED
    assert "page-locked" in cache.lib.moe_last_error().decode()


def test_destroy_evicts_the_cached_entries(torch):
    import bit_vq_routed_gb300 as bv
    spec = ms.LayerSpec(H=512, I=256, E=8, k=2, seed=36)
    layer = ms.Layer(spec)
    dev, cache, mf = _cached(layer, 1, 4, bv.MOE_FMT_VQ2)
    x = ms.tokens(1, spec.H, seed=6)
    mf.step(torch.from_numpy(x).view(torch.bfloat16).cuda())
    assert (dev.pair_status[:2].cpu().numpy() == 1).all()
    cache.destroy()
    g = run(dev, x)  # the table no longer points into the pool
    assert (g["status"] == 0).all()
    assert np.array_equal(g["out"], np.zeros_like(g["out"]))
