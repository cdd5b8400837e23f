"""Pins of the oracle's 4x temporal merge + adaptor MLP against facts outside the oracle:
a hand-built concatenation, closed forms, LayerNorm invariants, and torch's own functional ops
(an independent library) in float64."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def pin_temporal_merge_concatenates_four_consecutive_frames():
    frames = np.arange(8 * 3, dtype=np.float64).reshape(8, 3)
    merged = oracle.temporal_merge(frames)
    assert merged.shape == (2, 12)
    assert merged[0].tolist() == list(range(0, 12))
    assert merged[1].tolist() == list(range(12, 24))


def test_temporal_merge_rejects_partial_groups():
    with pytest.raises(AssertionError):
        oracle.temporal_merge(np.zeros((6, 2)))


def pin_zero_weights_closed_form():
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


def pin_silu_closed_form_through_identity_weights():
    """d = 1, H = E = 4, W1 = I (on the merged 4 values), W2 = I, eps = 0, unit affine:
    the output is the standardised SiLU of the four frames."""
    frames = np.array([[0.0], [1.0], [-2.0], [3.0]])
    y = oracle.adaptor(frames, np.eye(4), np.zeros(4), np.eye(4), np.zeros(4), np.ones(4),
                       np.zeros(4), eps=0.0)
    s = np.array([0.0, 1 / (1 + math.exp(-1)), -2 / (1 + math.exp(2)), 3 / (1 + math.exp(-3))])
    expect = (s - s.mean()) / math.sqrt(((s - s.mean()) ** 2).mean())
    np.testing.assert_allclose(y[0], expect, rtol=1e-12, atol=1e-12)


def pin_layernorm_rows_are_standardised():
    rng = np.random.default_rng(2)
    frames = rng.standard_normal((16, 8))
    y = oracle.adaptor(frames, rng.standard_normal((10, 32)), rng.standard_normal(10),
                       rng.standard_normal((7, 10)), rng.standard_normal(7), np.ones(7),
                       np.zeros(7), eps=1e-12)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose((y ** 2).mean(axis=1), 1.0, rtol=1e-9)


def pin_against_torch_functional_float64():
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


PINS = [pin_temporal_merge_concatenates_four_consecutive_frames, pin_zero_weights_closed_form,
        pin_silu_closed_form_through_identity_weights, pin_layernorm_rows_are_standardised,
        pin_against_torch_functional_float64]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__[4:])
def test_pin(pin):
    pin()


# ----------------------------------------------------------------------------------------------
# Planted mistakes: each plausible bug, planted into the oracle on the CPU, must fail a pin.
# A mutant replaces the oracle's merge or adaptor with a copy that differs in one step.
# ----------------------------------------------------------------------------------------------
def _mutant_adaptor(act=None, ddof=0, eps_in_sqrt=True, use_b1=True, swap_affine=False,
                    norm_hidden=False):
    def adaptor(frames, w1, b1, w2, b2, gamma, beta, eps=1e-5):
        x = oracle.temporal_merge(frames)
        h = x @ np.asarray(w1, np.float64).T + (np.asarray(b1, np.float64) if use_b1 else 0.0)
        h = act(h) if act is not None else h / (1.0 + np.exp(-h))
        if norm_hidden:
            h = (h - h.mean(axis=1, keepdims=True)) / np.sqrt(h.var(axis=1, keepdims=True) + eps)
        y = h @ np.asarray(w2, np.float64).T + np.asarray(b2, np.float64)
        mu = y.mean(axis=1, keepdims=True)
        var = y.var(axis=1, ddof=ddof, keepdims=True)
        z = (y - mu) / (np.sqrt(var + eps) if eps_in_sqrt else np.sqrt(var) + eps)
        g, b = np.asarray(gamma, np.float64), np.asarray(beta, np.float64)
        return z * b + g if swap_affine else z * g + b
    return adaptor


def _gelu_tanh(h):
    return 0.5 * h * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (h + 0.044715 * h ** 3)))


ADAPTOR_MUTANTS = {
    "merge_blocked": lambda m: m.setattr(
        oracle, "temporal_merge", lambda f, factor=4: np.concatenate(np.split(np.asarray(f, np.float64), factor), axis=1)),
    "merge_frames_reversed": lambda m: m.setattr(
        oracle, "temporal_merge",
        lambda f, factor=4: np.concatenate([np.asarray(f, np.float64)[factor - 1 - k::factor] for k in range(factor)], axis=1)),
    "silu_as_sigmoid": lambda m: m.setattr(oracle, "adaptor", _mutant_adaptor(act=lambda h: 1.0 / (1.0 + np.exp(-h)))),
    "gelu_for_silu": lambda m: m.setattr(oracle, "adaptor", _mutant_adaptor(act=_gelu_tanh)),
    "layernorm_unbiased_variance": lambda m: m.setattr(oracle, "adaptor", _mutant_adaptor(ddof=1)),
    "eps_outside_sqrt": lambda m: m.setattr(oracle, "adaptor", _mutant_adaptor(eps_in_sqrt=False)),
    "first_bias_dropped": lambda m: m.setattr(oracle, "adaptor", _mutant_adaptor(use_b1=False)),
    "scale_and_shift_swapped": lambda m: m.setattr(oracle, "adaptor", _mutant_adaptor(swap_affine=True)),
    "layernorm_on_hidden_too": lambda m: m.setattr(oracle, "adaptor", _mutant_adaptor(norm_hidden=True)),
}


def _all_pins_pass():
    for pin in PINS:
        pin()
    return True


@pytest.mark.parametrize("name", sorted(ADAPTOR_MUTANTS))
def test_planted_adaptor_mistake_is_caught(name, monkeypatch):
    assert _all_pins_pass()
    with monkeypatch.context() as m:
        ADAPTOR_MUTANTS[name](m)
        with np.errstate(all="ignore"):
            try:
                _all_pins_pass()
                caught = False
            except (AssertionError, ValueError):
                caught = True
    assert caught, f"planted mistake {name} passed every adaptor pin"
