"""ep_get_dispatch_layout_noalloc: the layout call for callers that cannot
allocate device memory (a serving engine whose HBM is already reserved for
weights and KV cache; a latency-critical pipeline where cudaMalloc/cudaFree
could synchronise the device). Its scratch is a static device array inside
the library, reused by every call, so each call must still give exactly the
layout the oracle gives, and exactly what ep_get_dispatch_layout gives with a
caller-allocated workspace, call after call, whatever the previous call left
in that array.

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import re
import os

import numpy as np
import pytest
import torch

import oracle
from combine_movement_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ep():
    from combine_movement_gb300 import build
    build.build()
    from combine_movement_gb300 import ep as mod
    return mod


def test_binding_limit_matches_the_header(ep):
    """The binding's copy of the scratch size is the header's #define."""
    text = open(os.path.join(ROOT, "include", "ep.h")).read()
    m = re.search(r"^#define\s+EP_NOALLOC_SCRATCH_BYTES\s+\(1u << (\d+)\)\s*$", text, re.M)
    assert m is not None, "EP_NOALLOC_SCRATCH_BYTES is no longer (1u << n) in include/ep.h"
    assert ep.EP_NOALLOC_SCRATCH_BYTES == 1 << int(m.group(1))


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


def _check(ep, wl: W.Workload, status, dev):
    """One no-allocation call on `wl`'s routing table, checked against the
    oracle's layout and against the workspace call, element by element."""
    idx_cpu = W.make_inputs(wl).topk_idx
    idx = idx_cpu.to(dev)
    c_ref, o_ref, s_ref, st_ref = oracle.Oracle().layout(idx_cpu.numpy(), wl.E)
    got = _layout_noalloc(ep, idx, wl.E, status)
    assert ep.ep_get_status(status) == st_ref == ep.EP_OK
    for g, r, name in zip(got, (c_ref, o_ref, s_ref), ("counts", "offsets", "slot")):
        assert np.array_equal(g.cpu().numpy(), r), f"{wl.name}: {name} differs from the oracle"
    want = _layout_with_workspace(ep, idx, wl.E)
    for g, w, name in zip(got, want, ("counts", "offsets", "slot")):
        assert torch.equal(g, w), f"{wl.name}: {name} differs from the workspace call"


@pytest.mark.gpu
def test_noalloc_matches_oracle_on_consecutive_calls(ep):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    # Tables large enough to need scratch by size (smaller ones are laid out
    # by one thread-block cluster, with none; up to 131,072 entries at
    # E <= 256 a 16-CTA cluster takes them without scratch where the GPU
    # holds one: 16384 x 8 at E = 128 here). The two launch shapes that use
    # it, in a sequence where each call finds the previous one's contents:
    #  - up to 128 tiles: one cooperative launch whose grid barrier keeps
    #    its words in the scratch (20000 x 8 at E = 128 and 512: 20 tiles);
    #  - more tiles: tile + finish launches (140000 x 8 at E = 128: 137
    #    tiles, 70 KB of per-tile counts);
    #  - then a cooperative call with another tile count (9000 x 8 at
    #    E = 1024: 71 tiles), whose flag words still hold earlier targets.
    big = W.Workload("noalloc-137-tiles", T=140000, H=8, E=128, K=8, seed=12)
    small_coop = W.Workload("noalloc-coop-71-tiles", T=9000, H=8, E=1024, K=8, seed=13)
    coop20 = W.Workload("noalloc-coop-20-tiles", T=20000, H=8, E=128, K=8, seed=14)
    cases = [coop20, W.sweep(16384, 64),
             W.Workload("noalloc-e512", T=20000, H=64, E=512, K=8, seed=11),
             big, small_coop, big, coop20]
    for wl in cases:
        assert 0 < ep.ep_layout_workspace_bytes(wl.T, wl.K, wl.E) <= ep.EP_NOALLOC_SCRATCH_BYTES
    assert ep.ep_layout_launches(big.T, big.K, big.E) == 2
    assert ep.ep_layout_launches(small_coop.T, small_coop.K, small_coop.E) == 1
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for wl in cases:
        _check(ep, wl, status, dev)


def _random_tables(n=16, seed=909):
    """Seeded tables of every layout launch shape (one block, one cluster,
    cooperative, tile + finish) within the scratch limit, with masked
    entries, in random order."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        E = int(rng.choice([1, 3, 64, 128, 300, 1024, 4096]))
        K = int(rng.integers(1, min(E, 8) + 1))
        T = int(rng.integers(1, 40000))
        if T * K > 320000:
            continue
        wl = W.Workload(f"noalloc-rand-{len(out)}", T=T, H=8, E=E, K=K, seed=900 + len(out),
                        mask_frac=float(rng.choice([0.0, 0.1])))
        out.append(wl)
    return out


@pytest.mark.gpu
def test_noalloc_random_tables_in_sequence(ep):
    """Sixteen seeded tables through the no-allocation layout one after
    another (whatever the previous call left in the scratch), each against
    the oracle and the workspace call; tables over the scratch limit must be
    refused before any device work."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for wl in _random_tables():
        if ep.ep_layout_workspace_bytes(wl.T, wl.K, wl.E) > ep.EP_NOALLOC_SCRATCH_BYTES:
            A = 0x10000
            code = ep.lib.ep_get_dispatch_layout_noalloc(A, wl.T, wl.K, wl.E, A, A, A, None, None)
            assert code == ep.EP_ERR_UNSUPPORTED
            continue
        _check(ep, wl, status, dev)
