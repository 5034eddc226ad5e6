"""The VQ2 encoder kernels (moe_vq2_train_codebook, moe_vq2_encode) against
the encoder oracle, bit for bit: the fp32 centroids, the fp16 codebook, the
codes and the scales.  The encoding of a full 2048 x 4096 matrix is compared
on 64 sampled rows (each row's encoding depends on that row alone).  Then a
dense synthetic expert, encoded on the GPU and packed, runs through the
layer against the layer oracle on the encoded weights."""
import numpy as np
import pytest

import moe_synth as ms
import oracle
from oracle import vq2_encoder as enc
from gpu_common import assert_close, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


def test_codebook_training_bit_exact(torch):
    import bit_vq_routed_gb300 as bv
    W = ms.dense_weights(256, 2048, seed=61)
    idx = ms.encoder_init_indices(256 * 512, seed=61)
    cb, C = bv.moe_vq2_train_codebook(torch.from_numpy(W).cuda(), idx, iters=6)
    torch.cuda.synchronize()
    C_o, cb_o = enc.train_codebook(W, idx, 6)
    assert np.array_equal(C.cpu().numpy().view(np.uint32), C_o.view(np.uint32))
    assert np.array_equal(cb.cpu().view(torch.int16).numpy().view(np.uint16), cb_o)


@pytest.mark.parametrize("rows,K,sample", [(128, 1024, None), (2048, 4096, 64)])
def test_encode_bit_exact(torch, rows, K, sample):
    import bit_vq_routed_gb300 as bv
    W = ms.dense_weights(rows, K, seed=62 + rows)
    idx = ms.encoder_init_indices(min(rows, 256) * K // 4, seed=62)
    _, cb_o = enc.train_codebook(W[:min(rows, 256)], idx, 4)
    codes, scales = bv.moe_vq2_encode(torch.from_numpy(W).cuda(), torch.from_numpy(cb_o.view(np.int16)).cuda()
                                      .view(torch.float16), iters=3)
    torch.cuda.synchronize()
    gc = codes.cpu().numpy()
    gs = scales.cpu().view(torch.int16).numpy().view(np.uint16)
    rs = np.arange(rows) if sample is None else np.sort(np.random.default_rng(7).choice(rows, sample, replace=False))
    oc, os_ = enc.encode(W[rs], cb_o, 3)
    assert np.array_equal(gc[rs], oc)
    assert np.array_equal(gs[rs], os_)


def test_encoded_expert_runs_through_the_layer(torch):
    """Dense gate/up/down -> GPU encoder -> packed slots -> the layer, against
    the layer oracle on the encoded weights (the encoder's output is a valid
    expert), and the quantisation error against the dense weights."""
    import bit_vq_routed_gb300 as bv
    H, I, E, k, T = 512, 256, 2, 2, 5
    spec = ms.LayerSpec(H=H, I=I, E=E, k=k, seed=63)
    layer = ms.Layer(spec)
    dense = {e: [ms.dense_weights(*shape, seed=63, stream=3 * e + m)
                 for m, shape in enumerate([(I, H), (I, H), (H, I)])] for e in range(E)}
    idx = ms.encoder_init_indices(I * H // 4, seed=63)
    cb, _ = bv.moe_vq2_train_codebook(torch.from_numpy(dense[0][0]).cuda(), idx, iters=8)
    layer.codebook = cb.cpu().view(torch.int16).numpy().view(np.uint16)
    for e in range(E):
        codes, scales = [], []
        for m in range(3):
            c, s = bv.moe_vq2_encode(torch.from_numpy(dense[e][m]).cuda(), cb, iters=3)
            codes.append(c.cpu().numpy())
            scales.append(s.cpu().view(torch.int16).numpy().view(np.uint16))
        layer._cache[e] = ms.ExpertWeights(ms.FMT_VQ2, codes, scales)
    dev, keep = bv.upload_layer(H, I, E, k, T, layer.codebook, layer.w_router, layer.bias,
                                lambda e: (ms.FMT_VQ2, layer._cache[e].codes, layer._cache[e].scales))
    x = ms.tokens(T, H, seed=63)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    out = dev.forward(xt).cpu().numpy()
    ref = oracle.default.moe_layer(layer, x)
    assert_close(out, ref["out"], "encoded expert")
    # against the dense weights (fp64): what 2.125 bits per weight cost
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    dense_out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = int(ref["ids"][t, j])
            Wg, Wu, Wd = (a.astype(np.float64) for a in dense[e])
            g, u = Wg @ xf[t], Wu @ xf[t]
            dense_out[t] += ref["weights"][t, j] * (Wd @ (g / (1 + np.exp(-g)) * u))
    rel = np.linalg.norm(ref["out"] - dense_out) / np.linalg.norm(dense_out)
    assert rel < 0.6, rel
