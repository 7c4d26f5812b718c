"""Failure detection on the GPU without faulting it: a wait that nothing
completes gives up after its bound, reports EP_ERR_TIMEOUT through the status
word, and the context keeps working."""
import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_movement_gb300 import build
    build.build()
    from combine_movement_gb300 import ep as mod
    return mod


def test_bounded_wait_times_out_and_context_survives(ep):
    dev = torch.device("cuda:0")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    t0 = time.perf_counter()
    ep.ep_selftest_wait_timeout(status, 2_000_000)  # 2 ms
    assert ep.ep_get_status(status) == ep.EP_ERR_TIMEOUT
    # the first wait and the drain of the three-stage ring, each bounded
    assert time.perf_counter() - t0 >= 4 * 0.002
    # the device is still usable: a normal layout + dispatch + combine
    from combine_movement_gb300 import workloads as W
    import oracle
    inp = W.make_inputs(W.TINY)
    st2 = torch.zeros(1, dtype=torch.int32, device=dev)
    counts, offsets, slot = ep.get_dispatch_layout(inp.topk_idx.to(dev), 8, status=st2)
    recv = ep.dispatch(inp.x.to(dev), slot, 256, status=st2)
    y = ep.combine(recv, slot, inp.topk_w.to(dev), status=st2)
    assert ep.ep_get_status(st2) == ep.EP_OK
    o = oracle.Oracle()
    _, _, s_ref, _ = o.layout(inp.topk_idx.numpy(), 8)
    assert np.array_equal(slot.cpu().numpy(), s_ref)


def test_selftest_rejects_bad_limits(ep):
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    with pytest.raises(ep.EPError):
        ep.ep_selftest_wait_timeout(status, 0)
    with pytest.raises(ep.EPError):
        ep.ep_selftest_wait_timeout(status, 5_000_000_000)
