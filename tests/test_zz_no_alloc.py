"""ep_get_dispatch_layout_noalloc: the layout call for callers that cannot
allocate device memory (a serving engine whose HBM is already reserved for
weights and KV cache; a latency-critical pipeline where cudaMalloc/cudaFree
could synchronise the device). Its scratch is a static device array inside
the library, so it must give exactly what ep_get_dispatch_layout gives with a
caller-allocated workspace, call after call, while that array is reused.

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from combine_movement_gb300 import workloads as W


@pytest.fixture(scope="module")
def ep():
    from combine_movement_gb300 import build
    build.build()
    from combine_movement_gb300 import ep as mod
    return mod


def test_oversize_is_rejected_before_any_device_work(ep):
    # E=4096 with 65536 entries needs 2 MiB of layout scratch: over the limit.
    T, K, E = 8192, 8, 4096
    assert ep.ep_layout_workspace_bytes(T, K, E) > ep.EP_NOALLOC_SCRATCH_BYTES
    A = 0x10000  # fake aligned address; the call must return before using it
    code = ep.lib.ep_get_dispatch_layout_noalloc(A, T, K, E, A, A, A, None, None)
    assert code == ep.EP_ERR_UNSUPPORTED


def _layout_with_workspace(ep, idx, E):
    counts, offsets, slot = ep.get_dispatch_layout(idx, E)
    return counts, offsets, slot


def _layout_noalloc(ep, idx, E, status):
    T, K = idx.shape
    counts = torch.full((E,), -3, dtype=torch.int32, device=idx.device)
    offsets = torch.full((E + 1,), -3, dtype=torch.int32, device=idx.device)
    slot = torch.full((T, K), -3, dtype=torch.int32, device=idx.device)
    ep.ep_get_dispatch_layout_noalloc(idx, E, counts, offsets, slot, status)
    return counts, offsets, slot


@pytest.mark.gpu
def test_noalloc_matches_workspace_layout_on_consecutive_calls(ep):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    # two different tables in a row, both large enough to use the scratch
    # (smaller tables are laid out by one thread-block cluster, with none)
    cases = [W.sweep(16384, 64),
             W.Workload("noalloc-e512", T=16384, H=64, E=512, K=8, seed=11)]
    for wl in cases:
        assert ep.ep_layout_workspace_bytes(wl.T, wl.K, wl.E) > 0
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for wl in cases:
        idx = W.make_inputs(wl).topk_idx.to(dev)
        want = _layout_with_workspace(ep, idx, wl.E)
        got = _layout_noalloc(ep, idx, wl.E, status)
        assert ep.ep_get_status(status) == ep.EP_OK
        for g, w, name in zip(got, want, ("counts", "offsets", "slot")):
            assert np.array_equal(g.cpu().numpy(), w.cpu().numpy()), f"{wl.name}: {name}"
    # and the first table again, after the second left its counts in the array
    idx = W.make_inputs(cases[0]).topk_idx.to(dev)
    want = _layout_with_workspace(ep, idx, cases[0].E)
    got = _layout_noalloc(ep, idx, cases[0].E, status)
    for g, w in zip(got, want):
        assert torch.equal(g, w)
