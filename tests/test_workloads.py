"""Seeded input generators (CPU only): shapes, determinism, routing laws."""
import numpy as np
import torch

from combine_movement_gb300 import workloads as W


def test_shapes_and_determinism():
    a = W.make_inputs(W.TINY)
    b = W.make_inputs(W.TINY)
    assert a.x.shape == (128, 1024) and a.x.dtype == torch.bfloat16
    assert a.topk_idx.shape == (128, 2) and a.topk_idx.dtype == torch.int64
    assert a.topk_w.shape == (128, 2) and a.topk_w.dtype == torch.float32
    assert torch.equal(a.x.view(torch.int16), b.x.view(torch.int16))
    assert torch.equal(a.topk_idx, b.topk_idx)
    assert torch.equal(a.topk_w, b.topk_w)
    c = W.make_inputs(W.sweep(1024, 2048))
    assert not torch.equal(a.topk_idx[:8], c.topk_idx[:8, :2])


def test_distinct_experts_and_softmax_weights():
    for wl in (W.TINY, W.DECODE, W.SKEWED):
        inp = W.make_inputs(wl)
        idx = inp.topk_idx.numpy()
        assert idx.min() >= 0 and idx.max() < wl.E
        srt = np.sort(idx, axis=1)
        assert np.all(srt[:, 1:] != srt[:, :-1]), "experts of a token must be distinct"
        w = inp.topk_w.numpy().astype(np.float64)
        assert np.all(w > 0)
        assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)


def test_uniform_first_draw_is_uniform():
    inp = W.make_inputs(W.sweep(16384, 2048))
    first = np.bincount(inp.topk_idx.numpy()[:, 0], minlength=128)
    exp = 16384 / 128
    chi2 = float(((first - exp) ** 2 / exp).sum())
    assert chi2 < 200, chi2  # 127 dof: mean 127, sd ~16


def test_zipf_first_draw_follows_law_and_skew():
    inp = W.make_inputs(W.SKEWED)
    idx = inp.topk_idx.numpy()
    p = 1.0 / np.arange(1, 65) ** 1.2
    p /= p.sum()
    first = np.bincount(idx[:, 0], minlength=64)
    exp = p * idx.shape[0]
    chi2 = float(((first - exp) ** 2 / exp).sum())
    assert chi2 < 110, chi2  # 63 dof
    counts = np.bincount(idx.ravel(), minlength=64)
    assert 8.0 < counts.max() / counts.mean() < 12.0


def test_masking_and_expert_standin():
    import dataclasses
    wl = dataclasses.replace(W.TINY, mask_frac=0.25)
    inp = W.make_inputs(wl)
    frac = float((inp.topk_idx == -1).float().mean())
    assert 0.15 < frac < 0.35
    rows = W.make_inputs(W.TINY).x[:4]
    assert torch.equal(W.expert_standin(rows, 1.0).view(torch.int16), rows.view(torch.int16))
    y = W.expert_standin(rows, 1.5)
    assert y.dtype == torch.bfloat16
    assert torch.equal(y.view(torch.int16), (rows.float() * 1.5).to(torch.bfloat16).view(torch.int16))
