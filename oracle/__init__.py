"""CPU oracle for MoE dispatch / combine (ctypes wrapper around ep_oracle.c).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg load this package; the library's own code never does. The C
source is a plain single-threaded restatement of what the path computes and
shares nothing with the CUDA library. Parity is pinned for every function
(see tests/test_oracle_pins.py); no function is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_HDR = os.path.join(_HERE, "ep_oracle.h")
LIB_PATH = os.path.join(_HERE, "libep_oracle.so")

OK = 0
BAD_EXPERT = 5

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def build(out_path: str = LIB_PATH, mutant: int = 0) -> str:
    """Compile the oracle with the system C compiler (portable flags only:
    the same source builds on x86_64 and aarch64). ``mutant`` > 0 plants one
    known mistake, for the tests that check the pins catch it."""
    cc = os.environ.get("CC", "gcc")
    cmd = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           f"-DORACLE_MUTANT={int(mutant)}", "-o", out_path, _SRC, "-lm"]
    subprocess.run(cmd, check=True, cwd=_HERE)
    return out_path


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    mt = os.path.getmtime(path)
    return mt < os.path.getmtime(_SRC) or mt < os.path.getmtime(_HDR)


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_layout.argtypes = [p, i64, i32, i32, p, p, p]
    lib.oracle_layout.restype = i32
    lib.oracle_dispatch.argtypes = [p, i64, i64, i32, p, p, p, p, p]
    lib.oracle_dispatch.restype = None
    lib.oracle_combine.argtypes = [p, p, p, i64, i64, i32, p]
    lib.oracle_combine.restype = None
    lib.oracle_pipeline_time.argtypes = [i64, ctypes.c_double, ctypes.c_double]
    lib.oracle_pipeline_time.restype = ctypes.c_double
    lib.oracle_serial_time.argtypes = [i64, ctypes.c_double, ctypes.c_double]
    lib.oracle_serial_time.restype = ctypes.c_double
    return lib


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (building first if missing or stale) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _stale(LIB_PATH):
                build(LIB_PATH)
            _lib = _bind(ctypes.CDLL(LIB_PATH))
        return _lib


def _ptr(a: Optional[np.ndarray]) -> Optional[int]:
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


class Oracle:
    """numpy-facing view of one oracle library (the real one by default)."""

    def __init__(self, lib: Optional[ctypes.CDLL] = None):
        self.lib = lib if lib is not None else load()

    def bf16_to_f32(self, b: int) -> float:
        return self.lib.oracle_bf16_to_f32(int(b))

    def f32_to_bf16(self, f: float) -> int:
        return int(self.lib.oracle_f32_to_bf16_rne(float(f)))

    def layout(self, topk_idx: np.ndarray, E: int):
        """Returns (counts[E], offsets[E+1], slot[T,K], status)."""
        idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
        T, K = idx.shape
        counts = np.empty(max(E, 0), dtype=np.int32)
        offsets = np.empty(max(E, 0) + 1, dtype=np.int32)
        slot = np.empty((T, K), dtype=np.int32)
        st = self.lib.oracle_layout(_ptr(idx), T, K, E, _ptr(counts),
                                    _ptr(offsets), _ptr(slot))
        return counts, offsets, slot, int(st)

    def dispatch(self, x_bits: np.ndarray, slot: np.ndarray, num_recv: int,
                 topk_w: Optional[np.ndarray] = None, fill: int = 0):
        """Returns (recv_x bits [num_recv, H], recv_w, recv_src). Rows no
        (t,k) maps to keep the ``fill`` bit pattern (recv_w NaN, src -1)."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        T, H = x.shape
        s = np.ascontiguousarray(slot, dtype=np.int32)
        K = s.shape[1] if s.ndim == 2 else 0
        recv_x = np.full((num_recv, H), fill, dtype=np.uint16)
        recv_w = recv_src = None
        w = None
        if topk_w is not None:
            w = np.ascontiguousarray(topk_w, dtype=np.float32)
            recv_w = np.full(num_recv, np.nan, dtype=np.float32)
            recv_src = np.full(num_recv, -1, dtype=np.int32)
        self.lib.oracle_dispatch(_ptr(x), T, H, K, _ptr(s), _ptr(w),
                                 _ptr(recv_x), _ptr(recv_w), _ptr(recv_src))
        return recv_x, recv_w, recv_src

    def combine(self, expert_out_bits: np.ndarray, slot: np.ndarray,
                topk_w: np.ndarray) -> np.ndarray:
        eo = np.ascontiguousarray(expert_out_bits, dtype=np.uint16)
        s = np.ascontiguousarray(slot, dtype=np.int32)
        w = np.ascontiguousarray(topk_w, dtype=np.float32)
        T, K = s.shape
        H = eo.shape[1]
        y = np.empty((T, H), dtype=np.uint16)
        self.lib.oracle_combine(_ptr(eo), _ptr(s), _ptr(w), T, H, K, _ptr(y))
        return y

    def pipeline_time(self, N: int, t_load: float, t_compute: float) -> float:
        return self.lib.oracle_pipeline_time(N, t_load, t_compute)

    def serial_time(self, N: int, t_load: float, t_compute: float) -> float:
        return self.lib.oracle_serial_time(N, t_load, t_compute)
