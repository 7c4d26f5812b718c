"""Pins of the CPU oracle: checks against facts that do not come from the
oracle itself (library routines, closed forms, brute force by a different
definition, the pages' worked example and hand-worked fixtures).

Each ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch. tests/test_oracle_pins.py runs them on the real oracle, and
tests/test_oracle_mutants.py runs them on builds with a planted mistake to
show that each mistake is caught.
"""
from __future__ import annotations

import itertools
import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            vals = [int(tok) for tok in v.split()]
            out[k] = vals[0] if len(vals) == 1 else vals
    return out


# --------------------------------------------------------------------------
# bf16 conversions: pinned to torch's bf16 casts (a library routine) and to
# hand-worked rounding cases.

def _torch_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.float().numpy()


def _torch_f32_to_bits(f: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(f.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def check_bf16(o) -> None:
    # Widening: every finite bf16 pattern, against torch.
    rng = np.random.default_rng(11)
    pats = np.arange(0, 1 << 16, 37, dtype=np.uint32).astype(np.uint16)
    ref = _torch_bits_to_f32(pats)
    for b, r in zip(pats, ref):
        got = np.float32(o.bf16_to_f32(int(b)))
        if np.isnan(r):
            assert np.isnan(got)
        else:
            assert got.view(np.uint32) == np.float32(r).view(np.uint32), hex(b)
    # Narrowing: hand-worked ties and boundaries (fp32 bit pattern -> bf16).
    hand = {
        0x3F800000: 0x3F80,  # 1.0
        0x3F808000: 0x3F80,  # exactly half an ulp above 1.0: tie -> even (down)
        0x3F818000: 0x3F82,  # tie with odd kept bit -> rounds up to even
        0x3F808001: 0x3F81,  # just above the tie -> up
        0x3F807FFF: 0x3F80,  # just below the tie -> down
        0xBF808000: 0xBF80,  # negative tie -> even
        0x7F7FFFFF: 0x7F80,  # largest finite fp32 overflows to +inf
        0x80000000: 0x8000,  # -0.0
        0x00000001: 0x0000,  # smallest subnormal rounds to +0
        0x7F800000: 0x7F80,  # +inf stays
    }
    for fbits, want in hand.items():
        f = np.uint32(fbits).view(np.float32)
        assert o.f32_to_bf16(float(f)) == want, (hex(fbits), hex(o.f32_to_bf16(float(f))))
    nan = np.uint32(0x7FC00001).view(np.float32)
    got = o.f32_to_bf16(float(nan))
    assert (got & 0x7F80) == 0x7F80 and (got & 0x007F) != 0
    # Narrowing: random values incl. constructed ties, against torch.
    base = rng.integers(0, 1 << 32, size=4000, dtype=np.uint64).astype(np.uint32)
    ties = (base & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    allb = np.concatenate([base, ties])
    fs = allb.view(np.float32)
    fs = fs[np.isfinite(fs)]
    want = _torch_f32_to_bits(fs)
    for f, w in zip(fs, want):
        assert o.f32_to_bf16(float(f)) == int(w), hex(np.float32(f).view(np.uint32))


# --------------------------------------------------------------------------
# layout

def _layout_by_counting(idx: np.ndarray, E: int):
    """Stable expert-major position of every valid entry, from the counting
    definition: entries of smaller experts, plus entries of the same expert
    that come earlier in (t, k) order. O(R^2), tiny inputs only."""
    flat = idx.reshape(-1)
    n = flat.size
    slot = np.full(n, -1, dtype=np.int64)
    for i in range(n):
        e = flat[i]
        if not (0 <= e < E):
            continue
        before = 0
        for j in range(n):
            ej = flat[j]
            if 0 <= ej < E and (ej < e or (ej == e and j < i)):
                before += 1
        slot[i] = before
    counts = np.array([np.sum(flat == e) for e in range(E)], dtype=np.int64)
    return counts, slot.reshape(idx.shape)


def _layout_by_library(idx: np.ndarray, E: int):
    """The same layout from numpy: bincount for the histogram, cumsum for the
    prefix, and a stable argsort of the expert ids for the receive order."""
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    counts = np.bincount(flat[valid], minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    order = np.nonzero(valid)[0][np.argsort(flat[valid], kind="stable")]
    slot = np.full(flat.size, -1, dtype=np.int64)
    slot[order] = np.arange(order.size)
    return counts, offsets, slot.reshape(idx.shape)


def check_layout_hand(o) -> None:
    g = read_golden("layout_hand_example.txt")
    idx = np.array(g["idx"], dtype=np.int64).reshape(3, 2)
    counts, offsets, slot, st = o.layout(idx, g["E"])
    assert st == 0
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert slot.reshape(-1).tolist() == g["slot"]


def check_layout_bruteforce(o) -> None:
    """All routing tables with T<=3, K<=2, E<=3 and ids in {-1, 0..E-1}."""
    for T, K, E in [(1, 1, 1), (2, 2, 2), (3, 1, 3), (3, 2, 2), (3, 2, 3)]:
        for vals in itertools.product(range(-1, E), repeat=T * K):
            idx = np.array(vals, dtype=np.int64).reshape(T, K)
            counts, offsets, slot, st = o.layout(idx, E)
            c_ref, s_ref = _layout_by_counting(idx, E)
            assert st == 0
            assert np.array_equal(counts, c_ref), (idx, counts, c_ref)
            assert np.array_equal(slot, s_ref), (idx, slot, s_ref)
            assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)


def check_layout_random(o) -> None:
    rng = np.random.default_rng(5)
    cases = [(300, 4, 7, 0.0), (257, 8, 64, 0.1), (1000, 6, 64, 0.0),
             (64, 3, 1, 0.0), (0, 2, 5, 0.0), (50, 1, 3, 0.3)]
    for T, K, E, mask in cases:
        # with repeated experts per token and skew, not only distinct ids
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        idx = rng.choice(E, size=(T, K), p=p / p.sum()).astype(np.int64)
        idx[rng.random((T, K)) < mask] = -1
        counts, offsets, slot, st = o.layout(idx, E)
        c_ref, o_ref, s_ref = _layout_by_library(idx, E)
        assert st == 0
        assert np.array_equal(counts, c_ref)
        assert np.array_equal(offsets, o_ref)
        assert np.array_equal(slot, s_ref)


def check_layout_bad_expert(o) -> None:
    idx = np.array([[0, 7], [-1, 1], [-5, 2]], dtype=np.int64)
    counts, offsets, slot, st = o.layout(idx, 3)
    assert st == 5
    assert counts.tolist() == [1, 1, 1]
    assert slot.tolist() == [[0, -1], [-1, 1], [-1, 2]]


# --------------------------------------------------------------------------
# dispatch: a permutation with replication, checked row by row, plus full
# coverage of the receive buffer (canary) and the per-segment multiset.

def check_dispatch(o) -> None:
    rng = np.random.default_rng(9)
    for T, H, K, E, mask in [(37, 24, 3, 5, 0.0), (64, 8, 8, 16, 0.2), (5, 136, 2, 2, 0.0)]:
        x = rng.integers(0, 1 << 16, size=(T, H), dtype=np.uint16)
        idx = np.stack([rng.permutation(max(E, K))[:K] % E for _ in range(T)]).astype(np.int64)
        idx[rng.random((T, K)) < mask] = -1
        w = rng.random((T, K), dtype=np.float32)
        _, offsets, slot, _ = o.layout(idx, E)
        R = int(offsets[-1])
        canary = 0xDEAD
        recv_x, recv_w, recv_src = o.dispatch(x, slot, R, w, fill=canary)
        covered = np.zeros(R, dtype=np.int64)
        for t in range(T):
            for k in range(K):
                s = slot[t, k]
                if s < 0:
                    continue
                covered[s] += 1
                assert np.array_equal(recv_x[s], x[t])
                assert recv_w[s] == w[t, k]
                assert recv_src[s] == t * K + k
        assert np.all(covered == 1)
        # rows of segment e are exactly the tokens routed to e, in t order
        for e in range(E):
            rows = recv_x[offsets[e]:offsets[e + 1]]
            toks = [t for t in range(T) for k in range(K) if idx[t, k] == e]
            assert np.array_equal(rows, x[toks].reshape(-1, H))


# --------------------------------------------------------------------------
# combine

def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def check_combine_closed_forms(o) -> None:
    rng = np.random.default_rng(21)
    for T, H, K in [(16, 64, 1), (16, 64, 2), (8, 40, 3), (8, 72, 8)]:
        x = torch.from_numpy(rng.standard_normal((T, H), dtype=np.float32)).to(torch.bfloat16)
        xb = _bf16_bits(x)
        idx = np.stack([rng.permutation(16)[:K] for _ in range(T)]).astype(np.int64)
        _, offsets, slot, _ = o.layout(idx, 16)
        recv, _, _ = o.dispatch(xb, slot, int(offsets[-1]))
        # all weights 1, identity experts: partial sums j*x are exact in fp32,
        # so the result is bf16(K*x), computed here by torch.
        ones = np.ones((T, K), dtype=np.float32)
        y = o.combine(recv, slot, ones)
        want = _bf16_bits((x.float() * K).to(torch.bfloat16))
        assert np.array_equal(y, want)
        # one-hot weight on k0 (others exactly 0): returns x itself.
        for k0 in {0, K - 1}:
            oh = np.zeros((T, K), dtype=np.float32)
            oh[:, k0] = 1.0
            assert np.array_equal(o.combine(recv, slot, oh), xb)


def check_combine_error_bound(o) -> None:
    """General weights and distinct expert rows: within the fp32 chain's
    error bound plus half a bf16 ulp of the exact (fp64) weighted sum."""
    rng = np.random.default_rng(23)
    for T, H, K, mask in [(24, 48, 8, 0.0), (40, 16, 6, 0.25), (10, 8, 1, 0.0)]:
        E = 32
        idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int64)
        idx[rng.random((T, K)) < mask] = -1
        _, offsets, slot, _ = o.layout(idx, E)
        R = int(offsets[-1])
        eo = torch.from_numpy(rng.standard_normal((R, H), dtype=np.float32) * 3).to(torch.bfloat16)
        eob = _bf16_bits(eo)
        eof = eo.double().numpy()
        w = (rng.random((T, K), dtype=np.float32) * 2 - 0.5).astype(np.float32)
        y = o.combine(eob, slot, w)
        yf = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).double().numpy()
        exact = np.zeros((T, H))
        mag = np.zeros((T, H))
        for t in range(T):
            for k in range(K):
                s = slot[t, k]
                if s >= 0:
                    exact[t] += np.float64(w[t, k]) * eof[s]
                    mag[t] += abs(np.float64(w[t, k]) * eof[s])
        chain = K * 2.0 ** -24 * mag
        half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact) + chain, 1e-30))) - 8)
        assert np.all(np.abs(yf - exact) <= chain + half_ulp + 1e-30), np.max(np.abs(yf - exact) - chain - half_ulp)


# Exact model of the combine arithmetic, independent of C's fmaf and of any
# float conversion routine: every fused multiply-add is the exact rational
# w*v + acc rounded once to binary32 (round to nearest, ties to even), and
# the final narrowing rounds that binary32 value once to bfloat16 (8
# significant bits, same exponent range). Both are IEEE 754 round-to-nearest
# written out over Fractions.

def _round_binary(q: Fraction, p: int, emin: int = -126, emax: int = 127):
    """q rounded to the nearest binary float with p significant bits and
    exponents emin..emax (gradual underflow), ties to even; a Fraction, or
    +-inf on overflow. Zero comes back as Fraction(0)."""
    if q == 0:
        return Fraction(0)
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if a < Fraction(2) ** e:
        e -= 1
    elif a >= Fraction(2) ** (e + 1):
        e += 1
    quantum = Fraction(2) ** (max(e, emin) - (p - 1))
    m = a / quantum
    n = m.numerator // m.denominator
    rest = m - n
    if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = n * quantum
    if v >= Fraction(2) ** (emax + 1):
        return math.copysign(math.inf, q)
    return v if q > 0 else -v


def _bf16_value(bits: int) -> Fraction:
    """Exact value of a finite bfloat16 bit pattern (sign, 8-bit exponent, 7-bit fraction)."""
    sign = -1 if bits & 0x8000 else 1
    ex = (bits >> 7) & 0xFF
    fr = bits & 0x7F
    assert ex != 0xFF
    if ex == 0:
        return sign * Fraction(fr, 1 << 7) * Fraction(2) ** -126
    return sign * (1 + Fraction(fr, 1 << 7)) * Fraction(2) ** (ex - 127)


def _bf16_bits_of(v: Fraction) -> int:
    """Bits of a bfloat16-representable value (via binary32, where it is exact)."""
    f = np.array([float(v)], dtype=np.float32)
    assert Fraction(float(f[0])) == v
    return int(f.view(np.uint32)[0] >> 16)


def _combine_exact(eo_bits: np.ndarray, slot: np.ndarray, w: np.ndarray) -> np.ndarray:
    T, K = slot.shape
    H = eo_bits.shape[1]
    y = np.zeros((T, H), dtype=np.uint16)
    for t in range(T):
        for h in range(H):
            acc = Fraction(0)
            for k in range(K):
                s = int(slot[t, k])
                if s < 0:
                    continue
                acc = _round_binary(Fraction(float(w[t, k])) * _bf16_value(int(eo_bits[s, h])) + acc, 24)
            y[t, h] = _bf16_bits_of(_round_binary(acc, 8))
    return y


def check_combine_exact(o) -> None:
    """The oracle's combine, bit for bit, against the exact model: random
    weights and rows (some entries masked), and two hand-derived tokens where
    the k order and the single rounding of each fma decide the bf16 output."""
    rng = np.random.default_rng(29)
    for T, H, K, mask in [(16, 24, 8, 0.0), (12, 16, 5, 0.3), (8, 16, 1, 0.0)]:
        E = 24
        idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int64)
        idx[rng.random((T, K)) < mask] = -1
        _, offsets, slot, _ = o.layout(idx, E)
        R = int(offsets[-1])
        eo = torch.from_numpy(rng.standard_normal((R, H), dtype=np.float32) * 4).to(torch.bfloat16)
        eob = _bf16_bits(eo)
        w = rng.standard_normal((T, K), dtype=np.float32)
        assert np.array_equal(o.combine(eob, slot, w), _combine_exact(eob, slot, w))

    # Two tokens, one expert row per (t, k), row r = 3t + k.
    one, big = 0x3F80, 0x4980                   # 1.0 and 2^20 in bfloat16
    small = 0x3F81                              # 1 + 2^-7
    slot = np.array([[0, 1, 2], [3, 4, -1]], dtype=np.int32)
    eob = np.zeros((5, 8), dtype=np.uint16)
    # token 0: rows small, 2^20, -2^20 with weights 1. In k order the first
    # sum rounds small to the 1/8 grid of 2^20, so the result is 1.0 (a
    # reversed order would give small itself).
    eob[0], eob[1], eob[2] = small, big, big | 0x8000
    # token 1: w0 = -(1 + 2^-7 + 2^-20) times 1.0, then w1 = 1 + 2^-20 times
    # (1 + 2^-7): the exact sum is 2^-27, which a fused multiply-add keeps;
    # rounding the product first would cancel to +0.
    eob[3], eob[4] = one, small
    w = np.array([[1.0, 1.0, 1.0],
                  [-(1 + 2.0 ** -7 + 2.0 ** -20), 1 + 2.0 ** -20, 0.0]], dtype=np.float32)
    want = np.array([[0x3F80] * 8, [0x3200] * 8], dtype=np.uint16)   # 1.0 and 2^-27
    assert np.array_equal(_combine_exact(eob, slot, w), want)
    assert np.array_equal(o.combine(eob, slot, w), want)


# --------------------------------------------------------------------------
# pipeline model

def _simulate_two_stage(N: int, tl: float, tc: float) -> float:
    """Event simulation of a double-buffered load/compute pipeline: load i
    starts when load i-1 is done and the buffer it reuses (that of tile i-2)
    has been consumed; compute i starts when load i and compute i-1 are done."""
    load_end = []
    comp_end = []
    for i in range(N):
        start = 0.0
        if i >= 1:
            start = max(start, load_end[i - 1])
        if i >= 2:
            start = max(start, comp_end[i - 2])
        load_end.append(start + tl)
        cs = load_end[i] if i == 0 else max(load_end[i], comp_end[i - 1])
        comp_end.append(cs + tc)
    return comp_end[-1] if N else 0.0


def check_pipeline(o) -> None:
    g = read_golden("pipeline_worked_example.txt")
    assert o.serial_time(g["N"], g["t_load_us"], g["t_compute_us"]) == g["serial_us"]
    assert o.pipeline_time(g["N"], g["t_load_us"], g["t_compute_us"]) == g["pipelined_us"]
    assert o.pipeline_time(1, 3.0, 5.0) == 8.0
    rng = np.random.default_rng(3)
    for _ in range(200):
        N = int(rng.integers(1, 40))
        tl, tc = (float(v) for v in rng.integers(1, 100, size=2))
        assert o.pipeline_time(N, tl, tc) == _simulate_two_stage(N, tl, tc)
        assert o.pipeline_time(N, tl, tc) == o.pipeline_time(N, tc, tl)
        assert o.pipeline_time(N, tl, tc) <= o.serial_time(N, tl, tc)


ALL_CHECKS = {
    "bf16": check_bf16,
    "layout_hand": check_layout_hand,
    "layout_bruteforce": check_layout_bruteforce,
    "layout_random": check_layout_random,
    "layout_bad_expert": check_layout_bad_expert,
    "dispatch": check_dispatch,
    "combine_closed_forms": check_combine_closed_forms,
    "combine_error_bound": check_combine_error_bound,
    "combine_exact": check_combine_exact,
    "pipeline": check_pipeline,
}
