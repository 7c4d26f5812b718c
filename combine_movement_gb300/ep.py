"""Thin Python binding of libep_gb300.so (the C ABI in include/ep.h).

Same entry-point names as the C ABI. This module only marshals arguments:
torch tensors become device pointers, the stream becomes its cudaStream_t
handle. Every step of layout, dispatch and combine runs in the library's CUDA
kernels; importing this module without the built library raises.

Convenience wrappers (``get_dispatch_layout``, ``dispatch``, ``combine``)
allocate outputs with torch and call the same entry points.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libep_gb300.so")

EP_OK = 0
EP_ERR_INVALID = 1
EP_ERR_UNSUPPORTED = 2
EP_ERR_CUDA = 3
EP_ERR_TIMEOUT = 4
EP_ERR_BAD_EXPERT = 5
EP_ERR_BAD_SLOT = 6
EP_ERR_WORKSPACE = 7

EP_MAX_TOPK = 32
EP_MAX_EXPERTS = 4096


def _header_define(name: str) -> int:
    """Integer value of a #define in include/ep.h (the C ABI's own header),
    so sizes the binding checks against cannot drift from it."""
    import re
    hdr = os.path.join(os.path.dirname(_PKG), "include", "ep.h")
    with open(hdr) as f:
        m = re.search(rf"^#define\s+{name}\s+(.+?)\s*$", f.read(), re.M)
    if m is None:
        raise ImportError(f"{name} is not defined in {hdr}")
    expr = re.sub(r"(?<=\d)[uUlL]+\b", "", m.group(1))
    if not re.fullmatch(r"[\d\s()<+*x]+", expr):
        raise ImportError(f"{name} in {hdr}: unexpected expression {m.group(1)!r}")
    return int(eval(expr, {"__builtins__": {}}))  # digits, parentheses, <<, +, * only


# Size of the static scratch array behind ep_get_dispatch_layout_noalloc.
EP_NOALLOC_SCRATCH_BYTES = _header_define("EP_NOALLOC_SCRATCH_BYTES")


class EPError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {ep_status_string(code)} (code {code})")
        self.code = code


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -m combine_movement_gb300.build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    p, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.ep_set_num_sms.argtypes = [i32]
    lib.ep_set_num_sms.restype = i32
    lib.ep_get_num_sms.argtypes = []
    lib.ep_get_num_sms.restype = i32
    lib.ep_set_launch_overlap.argtypes = [i32]
    lib.ep_set_launch_overlap.restype = i32
    lib.ep_get_launch_overlap.argtypes = []
    lib.ep_get_launch_overlap.restype = i32
    lib.ep_set_dispatch_tail.argtypes = [i32]
    lib.ep_set_dispatch_tail.restype = i32
    lib.ep_get_dispatch_tail.argtypes = []
    lib.ep_get_dispatch_tail.restype = i32
    lib.ep_set_combine_tail.argtypes = [i32]
    lib.ep_set_combine_tail.restype = i32
    lib.ep_get_combine_tail.argtypes = []
    lib.ep_get_combine_tail.restype = i32
    lib.ep_combine_launches.argtypes = [i64, i64, i32, p]
    lib.ep_combine_launches.restype = i32
    lib.ep_num_sms_in_effect.argtypes = []
    lib.ep_num_sms_in_effect.restype = i32
    lib.ep_layout_workspace_bytes.argtypes = [i64, i32, i32]
    lib.ep_layout_workspace_bytes.restype = sz
    lib.ep_layout_launches.argtypes = [i64, i32, i32]
    lib.ep_layout_launches.restype = i32
    lib.ep_dispatch_chunk_bytes.argtypes = [i64, i64, i32]
    lib.ep_dispatch_ring_stages.argtypes = []
    lib.ep_dispatch_ring_stages.restype = i32
    lib.ep_dispatch_chunk_bytes.restype = i64
    lib.ep_dispatch_launches.argtypes = [i64, i64, i32, p]
    lib.ep_dispatch_launches.restype = i32
    lib.ep_layout_dispatch_launches.argtypes = [i64, i64, i32, i32, p]
    lib.ep_layout_dispatch_launches.restype = i32
    lib.ep_get_dispatch_layout.argtypes = [p, i64, i32, i32, p, p, p, p, sz, p, p]
    lib.ep_get_dispatch_layout.restype = i32
    lib.ep_dispatch.argtypes = [p, i64, i64, i32, p, p, i64, p, p, p, p, p]
    lib.ep_dispatch.restype = i32
    lib.ep_layout_dispatch.argtypes = [p, p, i64, i64, i32, i32, p, i64, p, p, p, p, p, p, p, p]
    lib.ep_layout_dispatch.restype = i32
    lib.ep_combine.argtypes = [p, i64, p, p, i64, i64, i32, p, p, p]
    lib.ep_combine.restype = i32
    lib.ep_get_dispatch_layout_noalloc.argtypes = [p, i64, i32, i32, p, p, p, p, p]
    lib.ep_get_dispatch_layout_noalloc.restype = i32
    lib.ep_sm_partition.argtypes = [i32, ctypes.POINTER(p), ctypes.POINTER(p),
                                    ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.ep_sm_partition.restype = i32
    lib.ep_selftest_wait_timeout.argtypes = [p, ctypes.c_uint64, p]
    lib.ep_selftest_wait_timeout.restype = i32
    lib.ep_get_status.argtypes = [p, p]
    lib.ep_get_status.restype = i32
    lib.ep_status_string.argtypes = [i32]
    lib.ep_status_string.restype = ctypes.c_char_p
    return lib


lib = _load()


# --------------------------------------------------------------------------
# marshalling helpers

def _ptr(t: Optional[torch.Tensor], dtype=None, what: str = "") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what}: expected a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what}: expected a contiguous tensor")
    return t.data_ptr() if t.numel() > 0 else None


# The current stream's raw handle, read without building a torch.cuda.Stream
# object (about 2 us less per call on the host). Every call passes a CUDA
# tensor first, so CUDA is initialised by the time this runs.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream) -> Optional[int]:
    if stream is None:
        if _raw_stream is not None and _cur_device is not None:
            return _raw_stream(_cur_device()) or None
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _check(code: int, what: str) -> None:
    if code != EP_OK:
        raise EPError(code, what)


# --------------------------------------------------------------------------
# C ABI, same names

def ep_set_num_sms(num_sms: int) -> int:
    return lib.ep_set_num_sms(int(num_sms))


def ep_get_num_sms() -> int:
    return lib.ep_get_num_sms()


def ep_set_launch_overlap(mode: int) -> int:
    return lib.ep_set_launch_overlap(mode)


def ep_get_launch_overlap() -> int:
    return lib.ep_get_launch_overlap()


def ep_set_dispatch_tail(percent: int) -> int:
    return lib.ep_set_dispatch_tail(int(percent))


def ep_get_dispatch_tail() -> int:
    return lib.ep_get_dispatch_tail()


def ep_set_combine_tail(percent: int) -> int:
    return lib.ep_set_combine_tail(int(percent))


def ep_get_combine_tail() -> int:
    return lib.ep_get_combine_tail()


def ep_combine_launches(T: int, H: int, K: int, stream=None) -> int:
    return int(lib.ep_combine_launches(T, H, K, _stream(stream)))


def ep_num_sms_in_effect() -> int:
    return lib.ep_num_sms_in_effect()


def ep_layout_workspace_bytes(T: int, K: int, E: int) -> int:
    return int(lib.ep_layout_workspace_bytes(T, K, E))


def ep_layout_launches(T: int, K: int, E: int) -> int:
    return int(lib.ep_layout_launches(T, K, E))


def ep_dispatch_chunk_bytes(T: int, H: int, K: int) -> int:
    return int(lib.ep_dispatch_chunk_bytes(T, H, K))


def ep_dispatch_ring_stages() -> int:
    return int(lib.ep_dispatch_ring_stages())


def ep_dispatch_launches(T: int, H: int, K: int, stream=None) -> int:
    return int(lib.ep_dispatch_launches(T, H, K, _stream(stream)))


def ep_layout_dispatch_launches(T: int, H: int, K: int, E: int, stream=None) -> int:
    return int(lib.ep_layout_dispatch_launches(T, H, K, E, _stream(stream)))


def ep_status_string(code: int) -> str:
    return lib.ep_status_string(int(code)).decode()


def ep_get_dispatch_layout(topk_idx: torch.Tensor, num_experts: int, counts: torch.Tensor,
                           offsets: torch.Tensor, slot: torch.Tensor,
                           workspace: Optional[torch.Tensor] = None,
                           status: Optional[torch.Tensor] = None, stream=None) -> None:
    T, K = topk_idx.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    code = lib.ep_get_dispatch_layout(
        _ptr(topk_idx, torch.int64, "topk_idx"), T, K, int(num_experts),
        _ptr(counts, torch.int32, "counts"), _ptr(offsets, torch.int32, "offsets"),
        _ptr(slot, torch.int32, "slot"), _ptr(workspace, None, "workspace"), ws_bytes,
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(code, "ep_get_dispatch_layout")


def ep_get_dispatch_layout_noalloc(topk_idx: torch.Tensor, num_experts: int,
                                   counts: torch.Tensor, offsets: torch.Tensor,
                                   slot: torch.Tensor, status: Optional[torch.Tensor] = None,
                                   stream=None) -> None:
    """Layout for callers that cannot allocate: the scratch is the library's
    static device array (EP_NOALLOC_SCRATCH_BYTES), shared by every call."""
    T, K = topk_idx.shape
    code = lib.ep_get_dispatch_layout_noalloc(
        _ptr(topk_idx, torch.int64, "topk_idx"), T, K, int(num_experts),
        _ptr(counts, torch.int32, "counts"), _ptr(offsets, torch.int32, "offsets"),
        _ptr(slot, torch.int32, "slot"), _ptr(status, torch.int32, "status"), _stream(stream))
    _check(code, "ep_get_dispatch_layout_noalloc")




def ep_dispatch(x: torch.Tensor, slot: torch.Tensor, recv_x: torch.Tensor,
                topk_w: Optional[torch.Tensor] = None, recv_w: Optional[torch.Tensor] = None,
                recv_src: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                stream=None) -> None:
    T, H = x.shape
    K = slot.shape[1]
    code = lib.ep_dispatch(
        _ptr(x, torch.bfloat16, "x"), T, H, K, _ptr(slot, torch.int32, "slot"),
        _ptr(topk_w, torch.float32, "topk_w"), recv_x.shape[0],
        _ptr(recv_x, torch.bfloat16, "recv_x"), _ptr(recv_w, torch.float32, "recv_w"),
        _ptr(recv_src, torch.int32, "recv_src"), _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check(code, "ep_dispatch")


def ep_layout_dispatch(topk_idx: torch.Tensor, num_experts: int, x: torch.Tensor,
                       counts: torch.Tensor, offsets: torch.Tensor, slot: torch.Tensor,
                       recv_x: torch.Tensor, topk_w: Optional[torch.Tensor] = None,
                       recv_w: Optional[torch.Tensor] = None,
                       recv_src: Optional[torch.Tensor] = None,
                       status: Optional[torch.Tensor] = None, stream=None) -> None:
    T, H = x.shape
    K = topk_idx.shape[1]
    code = lib.ep_layout_dispatch(
        _ptr(topk_idx, torch.int64, "topk_idx"), _ptr(x, torch.bfloat16, "x"), T, H, K,
        int(num_experts), _ptr(topk_w, torch.float32, "topk_w"), recv_x.shape[0],
        _ptr(counts, torch.int32, "counts"), _ptr(offsets, torch.int32, "offsets"),
        _ptr(slot, torch.int32, "slot"), _ptr(recv_x, torch.bfloat16, "recv_x"),
        _ptr(recv_w, torch.float32, "recv_w"), _ptr(recv_src, torch.int32, "recv_src"),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(code, "ep_layout_dispatch")


def ep_combine(expert_out: torch.Tensor, slot: torch.Tensor, topk_w: torch.Tensor,
               y: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None) -> None:
    T, H = y.shape
    K = slot.shape[1]
    code = lib.ep_combine(
        _ptr(expert_out, torch.bfloat16, "expert_out"), expert_out.shape[0],
        _ptr(slot, torch.int32, "slot"), _ptr(topk_w, torch.float32, "topk_w"), T, H, K,
        _ptr(y, torch.bfloat16, "y"), _ptr(status, torch.int32, "status"), _stream(stream))
    _check(code, "ep_combine")


def ep_sm_partition(num_sms: int) -> Tuple[int, Optional[int], int, int]:
    """(stream, rest_stream, sms, rest_sms) of an SM partition of at least
    num_sms SMs on the current device; the streams are raw cudaStream_t
    handles (wrap them with torch.cuda.ExternalStream)."""
    s, r = ctypes.c_void_p(), ctypes.c_void_p()
    n, rn = ctypes.c_int(), ctypes.c_int()
    _check(lib.ep_sm_partition(int(num_sms), ctypes.byref(s), ctypes.byref(r), ctypes.byref(n),
                               ctypes.byref(rn)), "ep_sm_partition")
    return int(s.value), (int(r.value) if r.value else None), n.value, rn.value


def ep_selftest_wait_timeout(status: torch.Tensor, limit_ns: int, stream=None) -> None:
    _check(lib.ep_selftest_wait_timeout(_ptr(status, torch.int32, "status"), int(limit_ns),
                                        _stream(stream)), "ep_selftest_wait_timeout")


def ep_get_status(status: torch.Tensor, stream=None) -> int:
    return int(lib.ep_get_status(_ptr(status, torch.int32, "status"), _stream(stream)))


# --------------------------------------------------------------------------
# allocating conveniences

def get_dispatch_layout(topk_idx: torch.Tensor, num_experts: int,
                        status: Optional[torch.Tensor] = None, stream=None
                        ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Returns (counts[E], offsets[E+1], slot[T,K]) as int32 CUDA tensors."""
    dev = topk_idx.device
    T, K = topk_idx.shape
    counts = torch.empty(num_experts, dtype=torch.int32, device=dev)
    offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    nbytes = ep_layout_workspace_bytes(T, K, num_experts)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
    ep_get_dispatch_layout(topk_idx, num_experts, counts, offsets, slot, ws, status, stream)
    return counts, offsets, slot


def dispatch(x: torch.Tensor, slot: torch.Tensor, num_recv: int,
             topk_w: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
             stream=None):
    """Returns recv_x [num_recv, H] (and recv_w, recv_src when topk_w is given)."""
    recv_x = torch.empty((num_recv, x.shape[1]), dtype=x.dtype, device=x.device)
    recv_w = recv_src = None
    if topk_w is not None:
        recv_w = torch.empty(num_recv, dtype=torch.float32, device=x.device)
        recv_src = torch.empty(num_recv, dtype=torch.int32, device=x.device)
    ep_dispatch(x, slot, recv_x, topk_w, recv_w, recv_src, status, stream)
    return (recv_x, recv_w, recv_src) if topk_w is not None else recv_x


def combine(expert_out: torch.Tensor, slot: torch.Tensor, topk_w: torch.Tensor,
            status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    T = slot.shape[0]
    y = torch.empty((T, expert_out.shape[1]), dtype=expert_out.dtype, device=expert_out.device)
    ep_combine(expert_out, slot, topk_w, y, status, stream)
    return y
