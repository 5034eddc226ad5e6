"""The library's boot self-check on the GPU: moe_selftest runs the tiny layer
through every kernel family and compares with the stored oracle values."""
import pytest

from gpu_common import torch_cuda


@pytest.mark.gpu
def test_selftest_passes_and_launches_every_case():
    torch = torch_cuda()
    import bit_vq_routed_gb300 as bv
    n0 = bv.moe_launch_count()
    bv.moe_selftest()
    n1 = bv.moe_launch_count()
    # weights drawn and packed (8 experts x 3 matrices x 2 formats x 4 launches)
    # plus the routing and expert calls of the eight cases
    assert n1 - n0 > 200
    # a second run on another stream gives the same verdict
    s = torch.cuda.Stream()
    bv.moe_selftest(s)
    torch.cuda.synchronize()


@pytest.mark.gpu
def test_selftest_refuses_a_capturing_stream():
    torch = torch_cuda()
    import bit_vq_routed_gb300 as bv
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    x = torch.zeros(4, device="cuda")
    with torch.cuda.graph(g, stream=s):
        with pytest.raises(bv.MoeError) as ei:
            bv.moe_selftest(s)
        x.add_(1)  # the capture stays valid: the refused call enqueued nothing
    assert ei.value.status == bv.MOE_ERR_INVALID_ARG
    g.replay()
    torch.cuda.synchronize()
    assert float(x.sum()) == 4.0


@pytest.mark.gpu
def test_bounded_waits_give_up_and_the_context_stays_usable():
    """Failure detection without a fault: two waits on mbarriers that nothing
    completes (the kernels' bounded-wait pattern, plain and suspending
    try_wait) give up after their limits, record their error codes and
    return; the device then runs the self-check as before."""
    torch = torch_cuda()
    import bit_vq_routed_gb300 as bv
    r = bv.moe_selftest_wait_timeout()
    assert r["codes"] == (1, 2) and r["gave_up"] == (True, True), r
    # the suspending wait's 256 tries with a 1 us hint take at least ~0.1 ms and,
    # like the plain one, end well within a second
    assert 0 <= r["us"][0] < 1_000_000 and 100 <= r["us"][1] < 1_000_000, r
    print("bounded waits gave up after", r["us"], "us")
    bv.moe_selftest()
    torch.cuda.synchronize()
