"""The single-cluster layout (routing tables of 2 to 64 rounds of one block,
laid out by one thread-block cluster of up to 8 CTAs that exchange their
per-expert counts through distributed shared memory) must give exactly the
oracle's counts, offsets and slots for every expert count, including counts
that are not a multiple of 4 (the exchanged tables are padded to 16 bytes),
and for every number of CTAs in the cluster.

The library sizes a layout block to keep its per-warp counters within
64 KB of shared memory: warps = clamp(65536 / (4 E), 1, 32), one round =
32 * warps entries; tables of more than one round and at most 64 rounds
take the cluster path (8 CTAs x up to 8 rounds each). The table sizes below
are placed at the edges of that range: 2 CTAs, 5 CTAs, 8 CTAs of one round,
8 CTAs of two rounds, and the largest table of the path.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_movement_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    from combine_movement_gb300 import build
    build.build()
    from combine_movement_gb300 import ep as mod
    return mod


def _round_entries(E: int) -> int:
    warps = max(1, min(32, 65536 // (4 * E)))
    return 32 * warps


def _cases():
    out = []
    for E in (2, 7, 33, 257, 1000, 3001, 4096):
        r = _round_entries(E)
        for label, n in (("2-ctas", r + 1), ("5-ctas", 5 * r - 3), ("8-ctas", 8 * r),
                         ("8-ctas-2-rounds", 8 * r + 1), ("largest", 64 * r)):
            out.append((E, label, n))
    return out


@pytest.mark.parametrize("E,label,n", _cases())
def test_cluster_layout_matches_oracle(ep, E, label, n):
    K = min(8, E)
    T = (n + K - 1) // K
    if T * K > 64 * _round_entries(E):
        T = 64 * _round_entries(E) // K
    # the cluster path is the one multi-round path without a workspace
    assert T * K > _round_entries(E) and ep.ep_layout_workspace_bytes(T, K, E) == 0
    mask = 0.1 if E in (33, 3001) else 0.0
    wl = W.Workload(f"cluster-E{E}-{label}", T=T, H=8, E=E, K=K, seed=E + n, mask_frac=mask)
    idx_cpu = W.make_inputs(wl).topk_idx
    c_ref, o_ref, s_ref, st = oracle.Oracle().layout(idx_cpu.numpy(), E)
    assert st == 0
    dev = torch.device("cuda:0")
    counts, offsets, slot = ep.get_dispatch_layout(idx_cpu.to(dev), E)
    torch.cuda.synchronize()
    assert np.array_equal(counts.cpu().numpy(), c_ref), "counts"
    assert np.array_equal(offsets.cpu().numpy(), o_ref), "offsets"
    assert np.array_equal(slot.cpu().numpy(), s_ref), "slot"


def _wide_cases():
    out = []
    for E in (2, 7, 33, 257, 1000, 3001, 4096):
        r = _round_entries(E)
        # 13 CTAs of 5 rounds, 15 of 7, 16 of 8
        for label, n in (("13-ctas", 64 * r + 1), ("15-ctas", 104 * r - 5), ("largest", 128 * r)):
            out.append((E, label, n))
    return out


@pytest.mark.parametrize("E,label,n", _wide_cases())
def test_wide_cluster_layout_matches_oracle(ep, E, label, n):
    """Tables of 65 to 128 rounds: ep_get_dispatch_layout asks for a
    workspace (by size alone) but lays them out with one cluster of 13 to
    16 CTAs (a non-portable cluster size) where the GPU can hold one, else
    with the cooperative launch; either way exactly the oracle's layout."""
    K = min(8, E)
    T = (n + K - 1) // K
    if T * K > 128 * _round_entries(E):
        T = 128 * _round_entries(E) // K
    assert ep.ep_layout_workspace_bytes(T, K, E) > 0
    mask = 0.1 if E in (33, 3001) else 0.0
    wl = W.Workload(f"wide-E{E}-{label}", T=T, H=8, E=E, K=K, seed=E + n, mask_frac=mask)
    idx_cpu = W.make_inputs(wl).topk_idx
    c_ref, o_ref, s_ref, st = oracle.Oracle().layout(idx_cpu.numpy(), E)
    assert st == 0
    dev = torch.device("cuda:0")
    counts, offsets, slot = ep.get_dispatch_layout(idx_cpu.to(dev), E)
    torch.cuda.synchronize()
    assert np.array_equal(counts.cpu().numpy(), c_ref), "counts"
    assert np.array_equal(offsets.cpu().numpy(), o_ref), "offsets"
    assert np.array_equal(slot.cpu().numpy(), s_ref), "slot"

