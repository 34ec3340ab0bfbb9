"""Pins for the layer oracle (front end before the recurrence, gated RMSNorm after it).

Each test checks the oracle against something other than its own formula: a
library convolution, special values, exact identities, causality, packing, or
numbers worked out by hand.
"""
import math

import numpy as np
import pytest

from oracle import kda_layer_oracle as lo

RNG = np.random.default_rng(1234)


def _conv_w(H, d, W):
    return RNG.standard_normal((H, d, W))


def test_short_conv_matches_numpy_convolve():
    # One channel at a time, the causal depthwise convolution is np.convolve of the
    # sequence with the (reversed) taps, cut to the sequence length.
    T, H, d, W = 37, 2, 5, 4
    x = RNG.standard_normal((T, H, d))
    w = _conv_w(H, d, W)
    y = lo.short_conv(x, w)
    for h in range(H):
        for c in range(d):
            ref = np.convolve(x[:, h, c], w[h, c, ::-1])[:T]
            np.testing.assert_allclose(y[:, h, c], ref, rtol=0, atol=1e-12)


def test_short_conv_shift_kernel_and_sequence_start():
    # Taps (0, .., 1, 0): the output is the previous token, zero at each sequence start.
    T, H, d, W = 20, 1, 3, 4
    x = RNG.standard_normal((T, H, d))
    w = np.zeros((H, d, W))
    w[..., W - 2] = 1.0
    cu = [0, 7, 20]
    y = lo.short_conv(x, w, cu_seqlens=cu)
    for bos, eos in zip(cu[:-1], cu[1:]):
        assert np.all(y[bos] == 0.0)
        np.testing.assert_array_equal(y[bos + 1:eos], x[bos:eos - 1])


def test_short_conv_is_causal_and_packing_is_exact():
    T, H, d, W = 30, 2, 4, 3
    x = RNG.standard_normal((T, H, d))
    w = _conv_w(H, d, W)
    cu = [0, 11, 30]
    y = lo.short_conv(x, w, cu_seqlens=cu)
    x2 = x.copy()
    x2[17] += 5.0
    y2 = lo.short_conv(x2, w, cu_seqlens=cu)
    np.testing.assert_array_equal(y2[:17], y[:17])
    assert np.all(y2[17] != y[17])
    # packed == separate runs
    for bos, eos in zip(cu[:-1], cu[1:]):
        np.testing.assert_array_equal(lo.short_conv(x[bos:eos], w), y[bos:eos])


def test_sigmoid_family_special_values_and_identities():
    assert lo.logsigmoid(0.0) == pytest.approx(-math.log(2.0), abs=1e-15)
    assert lo.sigmoid(0.0) == pytest.approx(0.5, abs=1e-15)
    x = np.linspace(-60, 60, 241)
    np.testing.assert_allclose(lo.logsigmoid(x) - lo.logsigmoid(-x), x, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lo.sigmoid(x) + lo.sigmoid(-x), 1.0, rtol=0, atol=1e-15)
    assert np.all(lo.logsigmoid(x) <= 0.0)
    assert lo.logsigmoid(-700.0) == pytest.approx(-700.0, rel=1e-15)   # no overflow
    # SiLU: 0 at 0, the identity far right, 0 far left, and x * sigmoid(x) at 1
    assert lo.silu(0.0) == 0.0
    assert lo.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(lo.silu(-40.0)) < 1e-15
    assert lo.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)


def test_frontend_identity_conv_large_inputs_give_unit_directions():
    # Identity taps and large positive inputs: SiLU is the identity to 1e-15, so q and k
    # are the raw rows scaled to unit length (eps = 0), v the raw rows.
    T, H, d, W = 9, 2, 6, 4
    raw = 30.0 + RNG.random((3, T, H, d))
    w = np.zeros((H, d, W))
    w[..., W - 1] = 1.0
    a = RNG.standard_normal((T, H, d))
    b = RNG.standard_normal((T, H))
    q, k, v, la, beta = lo.frontend(raw[0], raw[1], raw[2], w, w, w, a, b, eps=0.0)
    for got, x in ((q, raw[0]), (k, raw[1])):
        np.testing.assert_allclose(np.linalg.norm(got, axis=-1), 1.0, rtol=0, atol=1e-14)
        np.testing.assert_allclose(got, x / np.linalg.norm(x, axis=-1, keepdims=True), rtol=1e-13, atol=0)
    np.testing.assert_allclose(v, raw[2], rtol=1e-13, atol=0)
    np.testing.assert_allclose(la - lo.logsigmoid(-a), a, atol=1e-12)
    np.testing.assert_allclose(beta + lo.sigmoid(-b), 1.0, atol=1e-15)


def test_frontend_l2_norm_with_eps_shrinks_exactly():
    # With eps > 0 the norm of the normalised row is sqrt(s / (s + eps)).
    T, H, d, W = 5, 1, 8, 2
    raw = RNG.standard_normal((T, H, d))
    w = np.zeros((H, d, W))
    w[..., W - 1] = 1.0
    s = np.sum(lo.silu(raw) ** 2, axis=-1)
    q, *_ = lo.frontend(raw, raw, raw, w, w, w, raw, raw[..., 0], eps=0.25)
    np.testing.assert_allclose(np.linalg.norm(q, axis=-1), np.sqrt(s / (s + 0.25)), rtol=1e-13)


def test_gated_rmsnorm_hand_example():
    # o = (3, 4): mean square 12.5; eps = 0, weight 1, gate far open -> (3, 4) / sqrt(12.5).
    o = np.array([[[3.0, 4.0]]])
    out = lo.gated_rmsnorm(o, np.full_like(o, 800.0), np.ones(2), 0.0)
    np.testing.assert_allclose(out[0, 0], [0.848528137423857, 1.131370849898476], rtol=1e-14)
    # gate 0 halves it; weight (2, -1) scales channel by channel
    out0 = lo.gated_rmsnorm(o, np.zeros_like(o), np.array([2.0, -1.0]), 0.0)
    np.testing.assert_allclose(out0[0, 0], [0.848528137423857, -0.565685424949238], rtol=1e-14)


def test_gated_rmsnorm_invariants():
    T, H, dv = 7, 3, 16
    o = RNG.standard_normal((T, H, dv))
    g = RNG.standard_normal((T, H, dv))
    w = RNG.standard_normal(dv)
    open_gate = np.full_like(o, 800.0)
    # unit mean square with eps = 0, weight 1, open gate
    out = lo.gated_rmsnorm(o, open_gate, np.ones(dv), 0.0)
    np.testing.assert_allclose(np.mean(out ** 2, axis=-1), 1.0, rtol=0, atol=1e-14)
    # scale invariance (eps = 0) and the eps shrink factor
    np.testing.assert_allclose(lo.gated_rmsnorm(3.7 * o, g, w, 0.0), lo.gated_rmsnorm(o, g, w, 0.0), rtol=1e-13)
    ms = np.mean(o ** 2, axis=-1, keepdims=True)
    np.testing.assert_allclose(lo.gated_rmsnorm(o, open_gate, np.ones(dv), 0.5),
                               out * np.sqrt(ms / (ms + 0.5)), rtol=1e-13)
    # the gate multiplies channel by channel: gate g vs its mirror -g sum to the open gate
    np.testing.assert_allclose(lo.gated_rmsnorm(o, g, w, 0.0) + lo.gated_rmsnorm(o, -g, w, 0.0),
                               lo.gated_rmsnorm(o, open_gate, w, 0.0), rtol=1e-12, atol=1e-14)
