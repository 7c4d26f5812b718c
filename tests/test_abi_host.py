"""The C-ABI library loads and exports every symbol include/ep.h declares,
and its host-side argument checks answer without touching a GPU (CPU only:
every call below returns before any CUDA runtime call)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ep():
    from combine_movement_gb300 import build
    build.build()
    from combine_movement_gb300 import ep as mod
    return mod


def declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "ep.h")).read()
    return sorted(set(re.findall(r"EP_API\s+[\w\s\*]+?\b(ep_\w+)\s*\(", hdr)))


def test_header_declares_the_four_calls():
    names = declared_symbols()
    for want in ("ep_get_dispatch_layout", "ep_dispatch", "ep_combine", "ep_set_num_sms"):
        assert want in names


def test_library_exports_every_declared_symbol(ep):
    names = declared_symbols()
    assert len(names) >= 9
    lib = ctypes.CDLL(ep.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", ep.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.strip()}
    assert set(names) <= exported
    # hidden visibility: nothing but the ABI (and no C++ internals) leaks out
    assert not [s for s in exported if s.startswith("_ZN2ep")]


def test_sm_budget_is_stored(ep):
    old = ep.ep_get_num_sms()
    try:
        assert ep.ep_set_num_sms(24) == 24
        assert ep.ep_get_num_sms() == 24
        assert ep.ep_set_num_sms(-3) == -1
        assert ep.ep_get_num_sms() == 24
        assert ep.ep_set_num_sms(0) == 0
    finally:
        ep.ep_set_num_sms(old)


def test_launch_overlap_mode_is_stored(ep):
    try:
        assert ep.ep_get_launch_overlap() == 0          # auto by default
        assert ep.ep_set_launch_overlap(1) == 1
        assert ep.ep_get_launch_overlap() == 1
        assert ep.ep_set_launch_overlap(3) == -1        # invalid: unchanged
        assert ep.ep_set_launch_overlap(-1) == -1
        assert ep.ep_get_launch_overlap() == 1
        assert ep.ep_set_launch_overlap(2) == 2
    finally:
        ep.ep_set_launch_overlap(0)


def test_status_strings(ep):
    for code in range(8):
        s = ep.ep_status_string(code)
        assert s and s != "unknown status"
    assert ep.ep_status_string(99) == "unknown status"


def test_workspace_bytes(ep):
    assert ep.ep_layout_workspace_bytes(128, 8, 256) == 0          # one fused launch
    assert ep.ep_layout_workspace_bytes(4096, 8, 256) == 0         # one thread-block cluster
    big = ep.ep_layout_workspace_bytes(16384, 8, 128)              # grid-wide cooperative launch
    assert big > 0 and big % 4 == 0
    assert big % 4 == 0 and big > 4 * 256 * 2                        # barrier words, totals, E x tiles
    assert ep.ep_layout_workspace_bytes(4096, 33, 256) == 0        # invalid -> 0
    assert ep.ep_layout_workspace_bytes(10, 2, 5000) == 0


def test_layout_launch_counts(ep):
    assert ep.ep_layout_launches(128, 8, 256) == 1       # one tile: fused block
    assert ep.ep_layout_launches(4096, 8, 256) == 1      # one thread-block cluster
    assert ep.ep_layout_launches(16384, 8, 128) == 1     # one cooperative launch
    assert ep.ep_layout_launches(20000, 8, 4096) == 2    # many tiles: tile + finish launches
    assert ep.ep_layout_launches(10, 33, 8) == -1


def test_dispatch_tail_percentage_round_trip(ep):
    before = ep.ep_get_dispatch_tail()
    try:
        assert before == 30
        assert ep.ep_set_dispatch_tail(0) == 0 and ep.ep_get_dispatch_tail() == 0
        assert ep.ep_set_dispatch_tail(90) == 90
        assert ep.ep_set_dispatch_tail(91) == -1 and ep.ep_get_dispatch_tail() == 90
        assert ep.ep_set_dispatch_tail(-1) == -1 and ep.ep_get_dispatch_tail() == 90
    finally:
        ep.ep_set_dispatch_tail(before)


def test_combine_tail_percentage_round_trip(ep):
    before = ep.ep_get_combine_tail()
    try:
        assert before == 30
        assert ep.ep_set_combine_tail(0) == 0 and ep.ep_get_combine_tail() == 0
        assert ep.ep_set_combine_tail(91) == -1 and ep.ep_get_combine_tail() == 0
    finally:
        ep.ep_set_combine_tail(before)
    assert ep.lib.ep_combine_launches(4096, 7166, 8, None) == -1    # H % 8 != 0
    assert ep.lib.ep_combine_launches(0, 7168, 8, None) == 0


def test_dispatch_launches_rejects_invalid_sizes(ep):
    # checked before the device is queried (no GPU needed)
    assert ep.lib.ep_dispatch_launches(4096, 7166, 8, None) == -1   # H % 8 != 0
    assert ep.lib.ep_dispatch_launches(4096, 7168, 33, None) == -1  # K above the limit
    assert ep.lib.ep_dispatch_launches(-1, 7168, 8, None) == -1
    assert ep.lib.ep_dispatch_launches(0, 7168, 8, None) == 0       # nothing to launch
    assert ep.lib.ep_layout_dispatch_launches(4096, 7168, 8, 0, None) == -1      # E < 1
    assert ep.lib.ep_layout_dispatch_launches(4096, 7168, 8, 5000, None) == -1   # E too large
    assert ep.lib.ep_layout_dispatch_launches(4096, 7166, 8, 256, None) == -1    # H % 8 != 0


def test_dispatch_chunk_bytes_rejects_invalid_sizes(ep):
    assert ep.ep_dispatch_chunk_bytes(4096, 7166, 8) == -1   # H % 8 != 0
    assert ep.ep_dispatch_chunk_bytes(4096, 7168, 33) == -1  # K above the limit
    assert ep.ep_dispatch_chunk_bytes(-1, 7168, 8) == -1
    assert ep.ep_dispatch_chunk_bytes(1 << 28, 7168, 8) == -1  # T*K overflows int32 slots
    assert ep.ep_dispatch_chunk_bytes(1 << 62, 7168, 8) == -1  # T*K would overflow int64 too


def test_sizes_near_int64_limits_are_refused_before_any_device_call(ep):
    """Limits are checked without forming T*K or H*2, so sizes whose products
    overflow int64 are refused too (UNSUPPORTED), never wrapped into range."""
    lib = ep.lib
    A = 0x10000  # a fake, 16-byte aligned "device" address; never dereferenced
    UNSUP = ep.EP_ERR_UNSUPPORTED
    for T in ((1 << 28), (1 << 62) + 3, (1 << 63) - 1):
        assert ep.ep_layout_workspace_bytes(T, 8, 256) == 0
        assert ep.ep_layout_launches(T, 8, 256) == -1
        assert lib.ep_get_dispatch_layout(A, T, 8, 256, A, A, A, None, 0, None, None) == UNSUP
        assert lib.ep_get_dispatch_layout_noalloc(A, T, 8, 256, A, A, A, None, None) == UNSUP
        assert lib.ep_dispatch(A, T, 7168, 8, A, None, 8, A, None, None, None, None) == UNSUP
        assert lib.ep_combine(A, 8, A, A, T, 7168, 8, A, None, None) == UNSUP
    for H in ((1 << 30), (1 << 62), (1 << 63) - 8):
        assert lib.ep_dispatch(A, 16, H, 8, A, None, 8, A, None, None, None, None) == UNSUP
        assert lib.ep_combine(A, 8, A, A, 16, H, 8, A, None, None) == UNSUP
        assert ep.ep_dispatch_chunk_bytes(16, H, 8) == -1
    # the boundary: 2^31 - 1 (token, expert) pairs pass the size check and
    # stop at the null buffers (INVALID); one token more is refused
    T_max = ((1 << 31) - 1) // 8
    assert lib.ep_dispatch(None, T_max, 7168, 8, None, None, 8, None, None, None, None,
                           None) == ep.EP_ERR_INVALID
    assert lib.ep_dispatch(None, T_max + 1, 7168, 8, None, None, 8, None, None, None, None,
                           None) == UNSUP
    assert lib.ep_combine(A, (1 << 31), A, A, 16, 7168, 8, A, None, None) == UNSUP  # num_recv


def _slice_golden():
    """Per-warp slice figures of DeepEP's intranode kernel, as the pages give
    them (tests/golden/tma_slice_budget.txt, with its citation)."""
    vals = {}
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "tma_slice_budget.txt")):
        line = line.split("#", 1)[0].strip()
        if "=" in line:
            k, v = (x.strip() for x in line.split("=", 1))
            vals[k] = int(v)
    return vals


def test_slice_golden_is_consistent():
    g = _slice_golden()
    assert g["warps"] == g["threads"] // 32
    assert g["smem_bytes"] == g["bytes_per_warp"] * g["warps"]
    assert g["row_bytes"] == 2 * g["hidden"] and g["half_row_bytes"] * 2 == g["row_bytes"]


@pytest.mark.gpu
def test_dispatch_chunk_bytes_plan(ep):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g = _slice_golden()
    try:
        ep.ep_set_num_sms(0)
        # prefill rows of 14336 B: the ring moves them in two chunks, the
        # half rows of DeepEP's receive loop
        assert ep.ep_dispatch_chunk_bytes(4096, g["hidden"], 8) == g["half_row_bytes"]
        # a decode batch is cut finer so every warp gets work, never below 512 B
        c = ep.ep_dispatch_chunk_bytes(128, 7168, 8)
        assert c % 16 == 0 and 512 <= c < 7168
        ep.ep_set_num_sms(24)
        c24 = ep.ep_dispatch_chunk_bytes(128, 7168, 8)
        assert c24 % 16 == 0 and c <= c24 <= 7168
    finally:
        ep.ep_set_num_sms(0)


@pytest.mark.gpu
def test_ring_depth_follows_budget_and_overlap_mode(ep):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    try:
        ep.ep_set_num_sms(0)
        ep.ep_set_launch_overlap(0)
        assert ep.ep_dispatch_ring_stages() == 3       # full budget: launches overlap
        ep.ep_set_num_sms(24)
        assert ep.ep_dispatch_ring_stages() == 4       # shared GPU: no overlap
        ep.ep_set_launch_overlap(1)
        assert ep.ep_dispatch_ring_stages() == 3
        ep.ep_set_num_sms(0)
        ep.ep_set_launch_overlap(2)
        assert ep.ep_dispatch_ring_stages() == 4
    finally:
        ep.ep_set_num_sms(0)
        ep.ep_set_launch_overlap(0)


@pytest.mark.gpu
def test_binding_passes_the_current_stream(ep):
    """With no stream argument the binding passes torch's current stream of
    the current device (the legacy default stream as NULL)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.zeros(1, device="cuda")
    assert ep._stream(None) == (torch.cuda.current_stream().cuda_stream or None)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert ep._stream(None) == s.cuda_stream
    assert ep._stream(s) == s.cuda_stream
    assert ep._stream(None) == (torch.cuda.current_stream().cuda_stream or None)


def _raw(ep):
    return ep.lib


def test_sm_partition_argument_checks(ep):
    """Refused before any CUDA call: fewer than one SM, or no stream out."""
    lib = _raw(ep)
    s = ctypes.c_void_p()
    assert lib.ep_sm_partition(0, ctypes.byref(s), None, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_sm_partition(-3, ctypes.byref(s), None, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_sm_partition(24, None, None, None, None) == ep.EP_ERR_INVALID


def test_host_argument_checks(ep):
    lib = _raw(ep)
    A = 0x10000  # a fake, 16-byte aligned "device" address; never dereferenced
    # dispatch: H not a multiple of 8, K out of range, misaligned x, null slot
    assert lib.ep_dispatch(A, 4, 12, 2, A, None, 8, A, None, None, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_dispatch(A, 4, 16, 33, A, None, 8, A, None, None, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_dispatch(A, 4, 16, 0, A, None, 8, A, None, None, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_dispatch(A + 8, 4, 16, 2, A, None, 8, A, None, None, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_dispatch(A, 4, 16, 2, None, None, 8, A, None, None, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_dispatch(A, 4, 16, 2, A, None, 8, A, A, None, None, None) == ep.EP_ERR_INVALID  # recv_w needs topk_w
    assert lib.ep_dispatch(A, -1, 16, 2, A, None, 8, A, None, None, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_dispatch(A, 1 << 30, 16, 8, A, None, 8, A, None, None, None, None) == ep.EP_ERR_UNSUPPORTED
    assert lib.ep_dispatch(None, 0, 16, 2, None, None, 0, None, None, None, None, None) == ep.EP_OK  # T == 0
    # combine
    assert lib.ep_combine(A, 8, A, A, 4, 16, 2, None, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_combine(A, 8, A, None, 4, 16, 2, A, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_combine(A + 4, 8, A, A, 4, 16, 2, A, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_combine(A, 8, A, A, 4, 10, 2, A, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_combine(None, 0, None, None, 0, 16, 2, None, None, None) == ep.EP_OK
    # layout
    assert lib.ep_get_dispatch_layout(A, 4, 2, 0, A, A, A, None, 0, None, None) == ep.EP_ERR_INVALID
    assert lib.ep_get_dispatch_layout(A, 4, 2, 5000, A, A, A, None, 0, None, None) == ep.EP_ERR_UNSUPPORTED
    assert lib.ep_get_dispatch_layout(A + 4, 4, 2, 8, A, A, A, None, 0, None, None) == ep.EP_ERR_INVALID
    # a table that needs a workspace: missing or too small is refused before any launch
    assert ep.ep_layout_workspace_bytes(16384, 8, 128) > 64
    assert lib.ep_get_dispatch_layout(A, 16384, 8, 128, A, A, A, None, 0, None, None) == ep.EP_ERR_WORKSPACE
    assert lib.ep_get_dispatch_layout(A, 16384, 8, 128, A, A, A, A, 64, None, None) == ep.EP_ERR_WORKSPACE
    assert lib.ep_get_status(None, None) == ep.EP_ERR_INVALID
    # fused layout + dispatch
    ld = lib.ep_layout_dispatch
    assert ld(A, A, 4, 16, 2, 0, None, 8, A, A, A, A, None, None, None, None) == ep.EP_ERR_INVALID
    assert ld(A, A, 4, 16, 2, 5000, None, 8, A, A, A, A, None, None, None, None) == ep.EP_ERR_UNSUPPORTED
    assert ld(A, A, 4, 12, 2, 8, None, 8, A, A, A, A, None, None, None, None) == ep.EP_ERR_INVALID
    assert ld(A + 4, A, 4, 16, 2, 8, None, 8, A, A, A, A, None, None, None, None) == ep.EP_ERR_INVALID
    assert ld(A, A, 4, 16, 2, 8, None, 8, None, A, A, A, None, None, None, None) == ep.EP_ERR_INVALID
