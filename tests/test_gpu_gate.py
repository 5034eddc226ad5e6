"""The confidence gate over an FP4 delta cache (vLLM-Moet page, "2-bit
experts on vLLM v0.24.0": a delta cache and a confidence gate bring FP4 back
where it matters; its bench table: tau = 0.60): a table of 2E entries with
every expert's 2-bit base at e and the FP4 weights of some experts at E + e.
A pair with router weight >= tau whose expert has FP4 weights in the table is
computed with them, every other pair with the base.  Checked against the
oracle (routing, the gate decision of every pair, the layer output) for
several tau, and with an expert cache filling the FP4 entries on demand."""
import numpy as np
import pytest

import moe_synth as ms
import oracle
from gpu_common import assert_close, experts_fn, torch_cuda

pytestmark = pytest.mark.gpu

H, I, E, K, T = 512, 256, 8, 2, 24


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


def _layers():
    base = ms.Layer(ms.LayerSpec(H=H, I=I, E=E, k=K, seed=71))
    fp4 = ms.Layer(ms.LayerSpec(H=H, I=I, E=E, k=K, seed=72, fp4_top=E))  # every expert FP4
    return base, fp4


def _oracle_gated(base, fp4, x, tau, have):
    O = oracle.default
    lg = O.router_logits(x, base.w_router, base.bias)
    ids, w = O.route_topk(lg, K, 1)
    assert not (np.abs(w - tau) < 1e-5).any()  # no decision within the fp32/fp64 gap
    gate = (w >= tau) & have[ids]
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(K):
            e = int(ids[t, j])
            ex = fp4.expert(e) if gate[t, j] else base.expert(e)
            y = O.expert_ffn(ex, base.codebook, xf[t:t + 1])[0]
            out[t] += w[t, j] * y
    return ids, gate, out


def _gated_layer(torch, base, fp4, have):
    import bit_vq_routed_gb300 as bv
    L = bv.MoELayer(H, I, E, K, T, base.codebook, base.w_router, base.bias, table_experts=2 * E)
    keep = []
    for e in range(E):
        fmt, c, s = experts_fn(base)(e)
        pc, ps = bv.upload_expert(fmt, c, s)
        L.set_expert(e, fmt, pc, ps)
        keep.append((pc, ps))
        if have[e]:
            fmt, c, s = experts_fn(fp4)(e)
            pc, ps = bv.upload_expert(fmt, c, s)
            L.set_expert(E + e, fmt, pc, ps)
            keep.append((pc, ps))
    return L, keep


@pytest.mark.parametrize("tau", [0.6, 0.52, 2.0, 0.0])
def test_gate_matches_oracle(torch, tau):
    import bit_vq_routed_gb300 as bv
    base, fp4 = _layers()
    have = np.zeros(E, bool)
    have[[0, 2, 5, 6]] = True
    L, keep = _gated_layer(torch, base, fp4, have)
    x = ms.tokens(T, H, seed=73)
    ids, gate, ref = _oracle_gated(base, fp4, x, tau, have)
    if tau == 0.6:
        assert 0 < gate.sum() < gate.size  # both kinds of pairs
    g = bv.GatedForward(L, T, tau)
    out = g.step(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(L.ids[:T].cpu().numpy(), ids)
    assert np.array_equal(g.gated.cpu().numpy(), ids + E * gate)
    assert L.pair_status[:T * K].cpu().numpy().all()
    assert_close(out.cpu().numpy(), ref, f"gated layer tau={tau}")


def test_delta_cache_fetches_what_the_gate_wants(torch):
    """FP4 weights of every expert in page-locked host memory, 2 device
    slots: each step fetches the FP4 entries of the pairs with weight >= tau
    (evicting by routing counts); pairs whose FP4 entry did not fit use the
    base.  Two steps in a row, against the oracle with the entries the cache
    held."""
    import bit_vq_routed_gb300 as bv
    base, fp4 = _layers()
    L, keep = _gated_layer(torch, base, fp4, np.zeros(E, bool))
    slot = bv.moe_expert_cache_slot_bytes(H, I, bv.MOE_FMT_FP4)
    pool = torch.empty(2 * slot, dtype=torch.uint8, device="cuda")
    cache = bv.ExpertCache(L.table, pool, slot)
    for e in range(E):
        ex = fp4.expert(e)
        cache.set_host_image(E + e, ex.fmt, bv.host_expert_image(ex.fmt, ex.codes, ex.scales))
    tau = 0.52
    g = bv.GatedForward(L, T, tau, cache=cache)
    for seed in (74, 75):
        x = ms.tokens(T, H, seed=seed)
        out = g.step(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda())
        torch.cuda.synchronize()
        have = np.array([cache.slot_of(E + e) >= 0 for e in range(E)])
        ids, gate, ref = _oracle_gated(base, fp4, x, tau, have)
        assert g.last["wanted"] > 0 and have.sum() >= 1
        assert np.array_equal(g.gated.cpu().numpy(), ids + E * gate)
        assert_close(out.cpu().numpy(), ref, f"delta cache step {seed}")
    cache.destroy()
