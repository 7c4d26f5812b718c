"""The measured alternatives, each built beside the default library and held
to the same parity bar: the combine that stages expert rows through a
per-warp bulk-copy ring (EP_COMBINE_MODE=1) and the dispatch that copies rows
through registers with 16-byte loads and stores (EP_DISPATCH_MODE=1). Their
timings are in the design notes; here only correctness is checked, through
the same C ABI, against the oracle."""
import ctypes

import numpy as np
import pytest
import torch

from combine_movement_gb300 import build as B
from combine_movement_gb300 import workloads as W
from test_gpu_parity import _custom, bits, from_bits, oracle_path

VARIANTS = {
    "staged-combine": ["-DEP_COMBINE_MODE=1"],
    "register-copy-dispatch": ["-DEP_DISPATCH_MODE=1"],
}


@pytest.fixture(scope="module")
def libs(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = {}
    for name, flags in VARIANTS.items():
        path = B.build(extra_flags=flags, out_dir=str(tmp_path_factory.mktemp(name)))
        lib = ctypes.CDLL(path)
        p, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        lib.ep_set_num_sms.argtypes = [i32]
        lib.ep_layout_workspace_bytes.argtypes = [i64, i32, i32]
        lib.ep_layout_workspace_bytes.restype = sz
        lib.ep_get_dispatch_layout.argtypes = [p, i64, i32, i32, p, p, p, p, sz, p, p]
        lib.ep_dispatch.argtypes = [p, i64, i64, i32, p, p, i64, p, p, p, p, p]
        lib.ep_combine.argtypes = [p, i64, p, p, i64, i64, i32, p, p, p]
        lib.ep_get_status.argtypes = [p, p]
        out[name] = lib
    return out


def _run(lib, inp, num_recv, expert_out, num_sms):
    dev = torch.device("cuda:0")
    T, K = inp.topk_idx.shape
    E, H = inp.wl.E, inp.wl.H
    idx = inp.topk_idx.to(dev)
    w = inp.topk_w.to(dev)
    x = inp.x.to(dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    nws = lib.ep_layout_workspace_bytes(T, K, E)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    recv = torch.full((num_recv, H), 0x7FA5, dtype=torch.int16, device=dev).view(torch.bfloat16)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    eo = from_bits(expert_out).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.ep_set_num_sms(num_sms)
    try:
        assert lib.ep_get_dispatch_layout(idx.data_ptr(), T, K, E, counts.data_ptr(),
                                          offsets.data_ptr(), slot.data_ptr(), ws.data_ptr(), nws,
                                          st.data_ptr(), None) == 0
        assert lib.ep_dispatch(x.data_ptr(), T, H, K, slot.data_ptr(), None, num_recv,
                               recv.data_ptr(), None, None, st.data_ptr(), None) == 0
        assert lib.ep_combine(eo.data_ptr(), num_recv, slot.data_ptr(), w.data_ptr(), T, H, K,
                              y.data_ptr(), st.data_ptr(), None) == 0
        assert lib.ep_get_status(st.data_ptr(), None) == 0
    finally:
        lib.ep_set_num_sms(0)
    return slot.cpu().numpy(), bits(recv), bits(y)


@pytest.mark.gpu
@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("case,budgets", [
    ((2048, 7168, 256, 8, 0.0, "uniform", 1.5), (0, 24)),
    ((3000, 4104, 64, 6, 0.1, "zipf", 1.0), (0, 16)),  # masked, partial last chunk
    ((128, 7168, 256, 8, 0.0, "uniform", 1.0), (0, 24)),
])
def test_variant_parity(libs, variant, case, budgets):
    T, H, E, K, mask, routing, scale = case
    inp = _custom(T, H, E, K, seed=31, mask=mask, routing=routing)
    num_recv = T * K
    ref = oracle_path(inp, num_recv, scale)
    for b in budgets:
        slot, recv, y = _run(libs[variant], inp, num_recv, ref.expert_out, b)
        assert np.array_equal(slot, ref.slot)
        assert np.array_equal(recv, ref.recv_x), "recv_x (incl. untouched canary rows)"
        assert np.array_equal(y, ref.y)
