"""Shared pieces of the GPU parity tests: building a device layer from the
seeded generator, running it, and the float tolerance."""
import numpy as np
import pytest

import moe_synth as ms

# Layer-output tolerance (the stated gate: fp32 accumulation on bf16
# activations): max |out - ref| <= 2e-2 * rms(ref) and
# sum |out - ref| / sum |ref| <= 2e-3.
MAX_REL_RMS = 2e-2
MEAN_REL = 2e-3
WEIGHT_ATOL = 1e-6


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def tolerance(out, ref):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(out - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return dict(max_err=float(err.max()), rms=rms, max_rel_rms=float(err.max() / rms),
                mean_rel=float(err.sum() / np.abs(ref).sum()))


def assert_close(out, ref, what=""):
    m = tolerance(out, ref)
    assert m["max_rel_rms"] <= MAX_REL_RMS and m["mean_rel"] <= MEAN_REL, f"{what} {m}"
    return m


def experts_fn(layer, cache=False):
    def f(e):
        ex = layer.expert(e, cache=cache)
        return ex.fmt, ex.codes, ex.scales
    return f


def device_layer(layer, T_max, resident=None):
    import bit_vq_routed_gb300 as bv
    s = layer.spec
    return bv.upload_layer(s.H, s.I, s.E, s.k, T_max, layer.codebook, layer.w_router, layer.bias,
                           experts_fn(layer), s.renormalize, resident)


def run(dev, x_bits):
    """Runs a forward pass; returns host copies of everything it produced."""
    import torch
    x = torch.from_numpy(np.ascontiguousarray(x_bits)).view(torch.bfloat16).cuda()
    T = x.shape[0]
    P = T * dev.k
    out = dev.forward(x)
    torch.cuda.synchronize()
    return dict(logits=dev.logits[:T].cpu().numpy(), ids=dev.ids[:T].cpu().numpy(),
                weights=dev.weights[:T].cpu().numpy(), offsets=dev.offsets.cpu().numpy(),
                sorted_pair=dev.sorted_pair[:P].cpu().numpy(),
                pair_to_sorted=dev.pair_to_sorted[:P].cpu().numpy(),
                status=dev.pair_status[:P].cpu().numpy(), ypair=dev.ypair[:P].cpu().numpy(),
                out=out.cpu().numpy().copy())


def device_error_word(dev):
    """The bounded-wait error word of the expert-FFN workspace (0 = none)."""
    import torch
    torch.cuda.synchronize()
    return int(dev.ws[8:12].view(torch.int32).item())


def assert_routing_exact(g, r):
    assert np.array_equal(g["logits"].view(np.uint32), r["logits"].view(np.uint32)), "router logits bits"
    assert np.array_equal(g["ids"], r["ids"])
    assert np.abs(g["weights"] - r["weights"]).max() <= WEIGHT_ATOL
    assert np.array_equal(g["offsets"], r["offsets"])
    assert np.array_equal(g["sorted_pair"], r["sorted_pair"])
    assert np.array_equal(g["pair_to_sorted"], r["pair_to_sorted"])
