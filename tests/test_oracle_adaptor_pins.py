"""Pins of the oracle's 4x temporal merge + adaptor MLP against facts outside the oracle:
a hand-built concatenation, closed forms, LayerNorm invariants, and torch's own functional ops
(an independent library) in float64."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def test_temporal_merge_is_concatenation_of_four_consecutive_frames():
    frames = np.arange(8 * 3, dtype=np.float64).reshape(8, 3)
    merged = oracle.temporal_merge(frames)
    assert merged.shape == (2, 12)
    assert merged[0].tolist() == list(range(0, 12))
    assert merged[1].tolist() == list(range(12, 24))


def test_temporal_merge_rejects_partial_groups():
    with pytest.raises(AssertionError):
        oracle.temporal_merge(np.zeros((6, 2)))


def test_zero_weights_closed_form():
    """W1 = W2 = 0: every row is LayerNorm(b2)."""
    rng = np.random.default_rng(1)
    d, H, E = 8, 6, 5
    frames = rng.standard_normal((12, d))
    b2 = np.array([1.0, -2.0, 0.5, 3.0, 0.0])
    g = np.array([1.0, 2.0, 1.0, 0.5, 1.0])
    be = np.array([0.0, 1.0, 0.0, 0.0, -1.0])
    y = oracle.adaptor(frames, np.zeros((H, 4 * d)), rng.standard_normal(H), np.zeros((E, H)), b2,
                       g, be, eps=0.0)
    mu = b2.mean()
    sd = math.sqrt(((b2 - mu) ** 2).mean())
    expect = (b2 - mu) / sd * g + be
    for row in y:
        np.testing.assert_allclose(row, expect, rtol=1e-13, atol=1e-13)


def test_silu_closed_form_through_identity_weights():
    """d = 1, H = E = 4, W1 = I (on the merged 4 values), W2 = I, eps = 0, unit affine:
    the output is the standardised SiLU of the four frames."""
    frames = np.array([[0.0], [1.0], [-2.0], [3.0]])
    y = oracle.adaptor(frames, np.eye(4), np.zeros(4), np.eye(4), np.zeros(4), np.ones(4),
                       np.zeros(4), eps=0.0)
    s = np.array([0.0, 1 / (1 + math.exp(-1)), -2 / (1 + math.exp(2)), 3 / (1 + math.exp(-3))])
    expect = (s - s.mean()) / math.sqrt(((s - s.mean()) ** 2).mean())
    np.testing.assert_allclose(y[0], expect, rtol=1e-12, atol=1e-12)


def test_layernorm_rows_are_standardised():
    rng = np.random.default_rng(2)
    frames = rng.standard_normal((16, 8))
    y = oracle.adaptor(frames, rng.standard_normal((10, 32)), rng.standard_normal(10),
                       rng.standard_normal((7, 10)), rng.standard_normal(7), np.ones(7),
                       np.zeros(7), eps=1e-12)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose((y ** 2).mean(axis=1), 1.0, rtol=1e-9)


def test_against_torch_functional_float64():
    rng = np.random.default_rng(3)
    d, H, E, T = 16, 12, 10, 5
    frames = rng.standard_normal((4 * T, d))
    w1 = rng.standard_normal((H, 4 * d)) / 8
    b1 = rng.standard_normal(H)
    w2 = rng.standard_normal((E, H)) / 4
    b2 = rng.standard_normal(E)
    g = 1 + 0.1 * rng.standard_normal(E)
    be = 0.1 * rng.standard_normal(E)
    y = oracle.adaptor(frames, w1, b1, w2, b2, g, be, eps=1e-5)
    t = lambda a: torch.from_numpy(a)
    x = t(frames).reshape(T, 4 * d)
    ref = F.layer_norm(F.linear(F.silu(F.linear(x, t(w1), t(b1))), t(w2), t(b2)), (E,), t(g),
                       t(be), eps=1e-5)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
