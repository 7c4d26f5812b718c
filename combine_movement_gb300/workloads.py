"""Seeded synthetic MoE routing workloads.

This module only draws inputs. It holds none of the dispatch/combine
arithmetic: no layout, no copy, no reduction. Both the GPU path and the CPU
oracle are fed from here, so the random numbers never have to agree across
languages.

Every workload is a token matrix ``x`` (bf16, ~N(0,1) drawn in fp32 and
rounded to nearest-even by torch), a routing table ``topk_idx`` (int64
[T][K], K distinct experts per token) and routing weights ``topk_w`` (fp32
[T][K], a softmax of N(0,1) logits over the chosen K). The pages study
DeepEP's dispatch (``buffer.dispatch(hidden_states, topk_idx, topk_weights,
num_experts=...)``, "How DeepEP Utilizes TMA Instructions for Minimal SM
Usage on Hopper GPUs", Practical Code Examples); the shapes below are the
synthetic stand-ins used to measure it. No public dataset is involved.

Draw order for a seed: x, then the routing keys, then the weight logits, all
from one ``numpy.random.Generator(PCG64(seed))`` (platform independent).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and routing recipe of one synthetic workload."""

    name: str
    T: int            # tokens
    H: int            # hidden size (bf16 elements per row)
    E: int            # experts
    K: int            # experts per token (top-k)
    seed: int
    routing: str = "uniform"     # "uniform" | "zipf"
    zipf_s: float = 1.2
    expert_scale: float = 1.0    # stand-in expert: y_e = bf16(scale * row)
    mask_frac: float = 0.0       # fraction of (t,k) entries set to -1


# The workloads the library is measured and checked on.
TINY = Workload("tiny", T=128, H=1024, E=8, K=2, seed=0)
DEEPSEEK_PREFILL = Workload("deepseek-v3-prefill", T=4096, H=7168, E=256, K=8,
                            seed=1, expert_scale=1.5)
SKEWED = Workload("skewed-zipf1.2", T=8192, H=4096, E=64, K=6, seed=2,
                  routing="zipf")
DECODE = Workload("decode", T=128, H=7168, E=256, K=8, seed=3)


def sweep(T: int, H: int) -> Workload:
    """One point of the size sweep: 128 experts, top-8, uniform routing."""
    return Workload(f"sweep-T{T}-H{H}", T=T, H=H, E=128, K=8, seed=4)


SWEEP_T = (1024, 4096, 16384)
SWEEP_H = (2048, 7168)

BY_NAME = {w.name: w for w in (TINY, DEEPSEEK_PREFILL, SKEWED, DECODE)}


@dataclasses.dataclass
class Inputs:
    """CPU tensors of one workload instance."""

    wl: Workload
    x: torch.Tensor          # bf16 [T, H]
    topk_idx: torch.Tensor   # int64 [T, K]
    topk_w: torch.Tensor     # float32 [T, K]

    def x_bits(self) -> np.ndarray:
        """x as raw bf16 bit patterns (uint16), the oracle's view."""
        return self.x.view(torch.int16).numpy().view(np.uint16)


def _routing(rng: np.random.Generator, wl: Workload) -> np.ndarray:
    """K distinct experts per token, in draw order.

    Uniform: the first K entries of a uniformly random permutation of the
    experts (argsort of i.i.d. uniform keys). Zipf: K successive draws
    without replacement from p(e) proportional to (e+1)^-s, renormalised over
    the experts not yet drawn; drawn with the Gumbel-top-k construction
    (sort log p(e) + Gumbel noise, descending), which has exactly that law.
    """
    T, E, K = wl.T, wl.E, wl.K
    if K > E:
        raise ValueError("K distinct experts need K <= E")
    u = rng.random((T, E))
    if wl.routing == "uniform":
        keys = u
    elif wl.routing == "zipf":
        logp = -wl.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        gumbel = -np.log(-np.log(np.clip(u, 1e-300, 1.0)))
        keys = -(logp[None, :] + gumbel)
    else:
        raise ValueError(f"unknown routing {wl.routing!r}")
    order = np.argsort(keys, axis=1, kind="stable")
    return np.ascontiguousarray(order[:, :K].astype(np.int64))


def _softmax_weights(rng: np.random.Generator, T: int, K: int) -> np.ndarray:
    logits = rng.standard_normal((T, K), dtype=np.float32).astype(np.float64)
    logits -= logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    p /= p.sum(axis=1, keepdims=True)
    return np.ascontiguousarray(p.astype(np.float32))


def make_inputs(wl: Workload, T: Optional[int] = None) -> Inputs:
    """Draw the inputs of ``wl`` (optionally only its first ``T`` tokens'
    worth of shape, with the same seed)."""
    if T is not None:
        wl = dataclasses.replace(wl, T=T)
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    x32 = rng.standard_normal((wl.T, wl.H), dtype=np.float32)
    x = torch.from_numpy(x32).to(torch.bfloat16)
    del x32
    idx = _routing(rng, wl)
    w = _softmax_weights(rng, wl.T, wl.K)
    if wl.mask_frac > 0.0:
        m = rng.random((wl.T, wl.K)) < wl.mask_frac
        idx[m] = -1
    return Inputs(wl, x.contiguous(), torch.from_numpy(idx), torch.from_numpy(w))


def expert_standin(rows: torch.Tensor, scale: float) -> torch.Tensor:
    """Stand-in for the experts between dispatch and combine.

    Returns ``bf16(scale * float(row))`` per element (round to nearest-even,
    done by torch). Identity when ``scale == 1``. This is the synthetic
    expert, not part of the data-movement method.
    """
    if scale == 1.0:
        return rows.clone()
    return (rows.float() * scale).to(torch.bfloat16)
