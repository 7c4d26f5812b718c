"""Dispatch and combine on a partial SM budget while an arithmetic kernel
holds the other SMs must give exactly the oracle's results, on ordinary
streams and in an SM partition.

"How DeepEP Utilizes TMA Instructions for Minimal SM Usage on Hopper GPUs"
(Minimal SM Occupancy Configuration) limits the communication kernels to a
few SMs so that the rest stay free for the experts' computation. Here the
rest runs an ALU-bound kernel (fp32 fma chains, one 1024-thread CTA per SM
held by a 120 KB shared-memory request, the stand-in of bench.py --overlap)
on a second stream, while batches move on 24 SMs on a high-priority stream,
once with the library's default launch policy and once with launch overlap
forced on (kernels may then start early, beside the foreign work). Every
output of every batch is compared with the oracle bit for bit, and the
events show that the arithmetic kernel was still running when the last
batch finished.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from combine_movement_gb300 import workloads as W
from test_gpu_parity import _custom, assert_parity, gpu_path, oracle_path

pytestmark = pytest.mark.gpu

BUDGET = 24
BATCHES = 4


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    from combine_movement_gb300 import build
    build.build()
    from combine_movement_gb300 import ep as mod
    yield mod
    mod.ep_set_num_sms(0)
    mod.ep_set_launch_overlap(0)


@pytest.fixture(scope="module")
def alu():
    """The ALU-bound stand-in kernel of bench.py, built with nvcc."""
    import bench
    tmp = tempfile.mkdtemp(prefix="ep_overlap_test_")
    src, so = os.path.join(tmp, "spin.cu"), os.path.join(tmp, "libspin.so")
    with open(src, "w") as f:
        f.write(bench._SPIN_SRC)
    subprocess.run(["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC",
                    "-gencode=arch=compute_103a,code=sm_103a", "-o", so, src], check=True)
    lib = ctypes.CDLL(so)
    lib.run_fma.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.run_fma.restype = ctypes.c_int
    return lib


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Batch:
    """One batch's inputs and outputs on the device, and the oracle's
    results for it (identity experts: combine reads the dispatched rows)."""

    def __init__(self, ep, wl: W.Workload, dev):
        inp = W.make_inputs(wl)
        T, H, E, K = wl.T, wl.H, wl.E, wl.K
        self.E = E
        self.x = inp.x.to(dev)
        self.idx = inp.topk_idx.to(dev)
        self.w = inp.topk_w.to(dev)
        self.counts = torch.full((E,), -7, dtype=torch.int32, device=dev)
        self.offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
        self.slot = torch.full((T, K), -7, dtype=torch.int32, device=dev)
        nws = ep.ep_layout_workspace_bytes(T, K, E)
        self.ws = torch.zeros(nws, dtype=torch.uint8, device=dev) if nws else None
        self.recv = torch.zeros((T * K, H), dtype=torch.bfloat16, device=dev)
        self.y = torch.zeros((T, H), dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        o = oracle.Oracle()
        self.c_ref, self.o_ref, self.s_ref, st = o.layout(inp.topk_idx.numpy(), E)
        assert st == 0
        self.r_ref, _, _ = o.dispatch(inp.x_bits(), self.s_ref, T * K)
        self.y_ref = o.combine(self.r_ref, self.s_ref, inp.topk_w.numpy())

    def layout(self, ep, s):
        ep.ep_get_dispatch_layout(self.idx, self.E, self.counts, self.offsets, self.slot, self.ws,
                                  self.status, s)

    def move(self, ep, s):
        ep.ep_dispatch(self.x, self.slot, self.recv, None, None, None, self.status, s)
        ep.ep_combine(self.recv, self.slot, self.w, self.y, self.status, s)

    def check(self, ep):
        assert ep.ep_get_status(self.status) == ep.EP_OK
        assert np.array_equal(self.counts.cpu().numpy(), self.c_ref)
        assert np.array_equal(self.offsets.cpu().numpy(), self.o_ref)
        assert np.array_equal(self.slot.cpu().numpy(), self.s_ref)
        assert np.array_equal(_bits(self.recv), self.r_ref)
        assert np.array_equal(_bits(self.y), self.y_ref)


def _alu_iters(alu, out, grid, stream, target_ms: float) -> int:
    """fma-loop iterations that make the ALU kernel last about target_ms."""
    probe = 20000
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    assert alu.run_fma(out.data_ptr(), grid, probe, stream.cuda_stream) == 0
    e1.record(stream)
    torch.cuda.synchronize()
    return max(probe, int(probe * target_ms / max(e0.elapsed_time(e1), 1e-3)))


def test_sm_partition_splits_the_device(ep):
    """ep_sm_partition: at least the SMs asked for, the rest in the second
    stream, the same streams for the same request."""
    dev = torch.device("cuda:0")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    s, r, n, rn = ep.ep_sm_partition(BUDGET)
    assert s and r and n >= BUDGET and n + rn == sms
    assert ep.ep_sm_partition(BUDGET) == (s, r, n, rn)
    with pytest.raises(ep.EPError):
        ep.ep_sm_partition(sms + 1)


def test_partition_bounds_the_grid_whatever_the_budget(ep):
    """With the budget at all SMs (0), calls into a 24-SM partition still
    launch at most the partition's CTAs per copy kernel and give the
    oracle's results (a larger grid would run in waves, or not at all)."""
    dev = torch.device("cuda:0")
    h, _, n, _ = ep.ep_sm_partition(BUDGET)
    s = torch.cuda.ExternalStream(h, device=dev)
    wl = W.Workload("partition-budget-0", T=1000, H=2048, E=64, K=6, seed=61)
    b = Batch(ep, wl, dev)
    try:
        ep.ep_set_num_sms(0)
        b.layout(ep, s)
        b.move(ep, s)
        torch.cuda.synchronize()
        b.check(ep)
    finally:
        ep.ep_set_num_sms(0)


@pytest.mark.parametrize("where", ["streams", "partition"])
@pytest.mark.parametrize("mode", [0, 1], ids=["default-policy", "launch-overlap-forced"])
@pytest.mark.parametrize("shape", ["decode", "T512-H2048"])
def test_movement_beside_alu_kernel_is_bit_exact(ep, alu, mode, shape, where):
    """`streams`: two ordinary streams, the movement's at high priority.
    `partition`: the movement in an SM partition of 24 SMs and the ALU
    kernel in the partition of the other SMs (ep_sm_partition), where the
    default policy lets the launches of these calls overlap (both shapes
    move at most 64 MB of rows per call)."""
    dev = torch.device("cuda:0")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if shape == "decode":
        # single-block layout: the whole step runs beside the ALU kernel
        wls = [W.Workload(f"ovl-decode-{i}", T=128, H=7168, E=256, K=8, seed=40 + i)
               for i in range(BATCHES)]
    else:
        # the layout is one thread-block cluster, which needs free SMs in one
        # GPC: laid out before the ALU kernel starts, as bench.py --overlap does
        wls = [W.Workload(f"ovl-t512-{i}", T=512, H=2048, E=64, K=8, seed=50 + i)
               for i in range(BATCHES)]
    batches = [Batch(ep, wl, dev) for wl in wls]
    if where == "partition":
        h_move, h_alu, n_move, n_alu = ep.ep_sm_partition(BUDGET)
        s_move = torch.cuda.ExternalStream(h_move, device=dev)
        s_alu = torch.cuda.ExternalStream(h_alu, device=dev)
        grid = n_alu
    else:
        s_move = torch.cuda.Stream(dev, priority=-1)
        s_alu = torch.cuda.Stream(dev)
        grid = sms - BUDGET
    out = torch.zeros(1, device=dev)
    try:
        ep.ep_set_num_sms(BUDGET)
        ep.ep_set_launch_overlap(mode)
        # warm-up (loads the kernels), then clear what it wrote
        batches[0].layout(ep, s_move)
        batches[0].move(ep, s_move)
        torch.cuda.synchronize()
        for b in batches:
            b.counts.fill_(-7), b.offsets.fill_(-7), b.slot.fill_(-7)
            b.recv.zero_(), b.y.zero_()
        iters = _alu_iters(alu, out, grid, s_alu, 20.0)
        if shape != "decode":
            for b in batches:
                b.layout(ep, s_move)
            torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m1 = torch.cuda.Event(enable_timing=True)
        a0.record(s_alu)
        assert alu.run_fma(out.data_ptr(), grid, iters, s_alu.cuda_stream) == 0
        a1.record(s_alu)
        for b in batches:
            if shape == "decode":
                b.layout(ep, s_move)
            b.move(ep, s_move)
        m1.record(s_move)
        torch.cuda.synchronize()
        # the last batch finished while the ALU kernel was still running
        assert a0.elapsed_time(m1) < a0.elapsed_time(a1), "no overlap: ALU kernel ended first"
        for b in batches:
            b.check(ep)
    finally:
        ep.ep_set_num_sms(0)
        ep.ep_set_launch_overlap(0)


@pytest.mark.parametrize("T,H,E,K,mask", [
    (128, 7168, 256, 8, 0.0),   # decode: 14.7 MB of rows, launches overlap in the partition
    (555, 7168, 64, 8, 0.0),    # 63.7 MB: just under the 64 MB size rule
    (600, 7168, 64, 8, 0.0),    # 68.8 MB: just over it, ordinary launch order
    (1000, 2056, 40, 6, 0.1),   # masked entries, rows not a multiple of the column block
    (3, 24, 2, 2, 0.0),         # tiny rows
    (4096, 1024, 128, 8, 0.0),  # 67 MB, a multi-CTA layout
])
@pytest.mark.parametrize("fused", [False, True], ids=["three-calls", "layout-dispatch"])
def test_partition_stream_matches_oracle(ep, T, H, E, K, mask, fused):
    """Every call of the path into a 24-SM partition stream (the default
    launch policy: overlapping launches for calls of at most 64 MB of rows,
    ordinary order above), at the budget of all SMs and of 5, gives the
    oracle's results."""
    dev = torch.device("cuda:0")
    h, _, _, _ = ep.ep_sm_partition(BUDGET)
    s = torch.cuda.ExternalStream(h, device=dev)
    inp = _custom(T, H, E, K, seed=T + E, mask=mask)
    num_recv = int((inp.topk_idx >= 0).sum()) + 2
    ref = oracle_path(inp, num_recv, 1.5)
    try:
        for b in (0, 5):
            with torch.cuda.stream(s):
                got = gpu_path(ep, inp, num_recv, ref.expert_out, num_sms=b, stream=s, fused=fused)
            assert_parity(got, ref)
    finally:
        ep.ep_set_num_sms(0)
