"""Activations far outside fp16's range (bf16 outlier channels of 1e3 to
1e5) through every kernel family of the expert FFN, against the oracle at
the stated tolerance.  The fp16 operands of the kernels (table entries, the
gathered activations, silu(g)*u) are scaled by powers of two chosen from the
data, so they cannot overflow; the cases are chosen so that an unscaled fp16
conversion would overflow (table entries and activations above 65504, and
silu(g)*u above 65504, which the test checks on the oracle's fp64 values)."""
import numpy as np
import pytest

import moe_synth as ms
import oracle
from gpu_common import assert_close, assert_routing_exact, device_layer, run, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


def _max_silu_gu(layer, x_bits, ids):
    """Largest |silu(g) * u| over the routed pairs, from the oracle's fp64
    decode of the weights (a precondition of the test, not a result)."""
    O = oracle.default
    x = (np.asarray(x_bits, np.uint32) << 16).view(np.float32).astype(np.float64)
    m = 0.0
    for t in range(x.shape[0]):
        for e in np.unique(ids[t]):
            ex = layer.expert(int(e))
            if ex.fmt == ms.FMT_VQ2:
                Wg = O.decode_vq2(ex.codes[0], ex.scales[0], layer.codebook)
                Wu = O.decode_vq2(ex.codes[1], ex.scales[1], layer.codebook)
            else:
                Wg = O.decode_fp4(ex.codes[0], ex.scales[0])
                Wu = O.decode_fp4(ex.codes[1], ex.scales[1])
            g, u = Wg @ x[t], Wu @ x[t]
            with np.errstate(over="ignore"):  # exp(-g) = inf gives silu(g) = -0, as it should
                m = max(m, float(np.abs(g / (1.0 + np.exp(-g)) * u).max()))
    return m


# (name, spec, tokens): the expert token counts select the kernel family.
CASES = [
    # one token: the activation-table kernels without a schedule
    ("table_t1", ms.LayerSpec(H=4096, I=2048, E=16, k=4, seed=41), 1),
    # three tokens over 16 experts: table pairs of 1..3 tokens per expert
    ("table_t3", ms.LayerSpec(H=4096, I=2048, E=16, k=4, seed=42), 3),
    # 24 tokens over 4 experts (about 12 each): the mma.sync kernels
    ("mma", ms.LayerSpec(H=1024, I=512, E=4, k=2, seed=43), 24),
    # 96 tokens, top-1 of 2 experts (about 48 each): the tcgen05 kernels
    ("tcgen05", ms.LayerSpec(H=1024, I=512, E=2, k=1, seed=44), 96),
    # every expert FP4: the FP4 mma.sync kernels
    ("fp4", ms.LayerSpec(H=1024, I=512, E=8, k=2, seed=45, fp4_top=8), 8),
]


@pytest.mark.parametrize("name,spec,T", CASES, ids=[c[0] for c in CASES])
def test_outlier_activations_match_oracle(torch, name, spec, T):
    layer = ms.Layer(spec)
    x = ms.tokens_outliers(T, spec.H, seed=spec.seed)
    assert np.abs((x.astype(np.uint32) << 16).view(np.float32)).max() > 65504
    ref = oracle.default.moe_layer(layer, x)
    assert _max_silu_gu(layer, x, ref["ids"]) > 65504
    dev, keep = device_layer(layer, T)
    g = run(dev, x)
    assert_routing_exact(g, ref)
    assert g["status"].all()
    assert np.isfinite(g["out"]).all(), f"{name}: non-finite output"
    assert_close(g["out"], ref["out"], name)
    counts = np.bincount(ref["ids"].ravel(), minlength=spec.E)
    if name == "mma":
        assert (counts[counts > 0] >= 4).all() and counts.max() < 32, counts
    if name == "tcgen05":
        assert (counts[counts > 0] >= 32).all(), counts


def test_small_activations_keep_their_precision(torch):
    """Activations around 1e-3 (far below fp16's normal range once multiplied
    by the small weights) on the tensor-core and table paths: the scaling
    brings them up, so the relative error stays that of N(0,1) inputs."""
    spec = ms.LayerSpec(H=1024, I=512, E=4, k=2, seed=46)
    layer = ms.Layer(spec)
    x32 = (ms.tokens(40, spec.H, seed=46).astype(np.uint32) << 16).view(np.float32) * np.float32(1e-3)
    x = (x32.view(np.uint32) >> 16).astype(np.uint16)
    ref = oracle.default.moe_layer(layer, x)
    dev, keep = device_layer(layer, 40)
    g = run(dev, x)
    assert_routing_exact(g, ref)
    assert_close(g["out"], ref["out"], "small activations")
