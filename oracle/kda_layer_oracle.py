"""fp64 CPU oracle for the layer steps around the KDA recurrence -- TEST
INFRASTRUCTURE ONLY (the product path never imports it).

"Kimi K3 architecture: KDA, MLA and MoE", section "Scale: Total vs Active
Parameters and Serving Economics", Visual 1 (the KDA inset) draws one KDA
layer: q and k each pass a projection, a short convolution, SiLU and an L2
norm; v a projection, a short convolution and SiLU; alpha and beta a
projection and a sigmoid; a gate a projection and a sigmoid.  After the KDA
box the output passes a norm and is multiplied by the gate.  The projections
are plain GEMMs outside this library.  This module restates, in plain numpy
fp64, the steps between the projections and the recurrence (``frontend``) and
the step after it (``gated_rmsnorm``).

Readings where the figure is silent:
- the short convolution is depthwise and causal over the tokens of one
  sequence, width W (the figure gives no width; the library takes W <= 4),
  with zero history before the sequence start and no bias:
  y[t, c] = sum_{i<W} w[c, i] * x[t - (W-1) + i, c];
- the L2 norm is over the key dimension of one (token, head):
  x / sqrt(sum x^2 + eps);
- alpha = sigmoid(a_raw) per key channel, so log alpha = logsigmoid(a_raw);
  beta = sigmoid(b_raw) per head;
- "a norm" after the KDA box is an RMSNorm over the value dimension of one
  (token, head) with a weight per value channel shared by the heads:
  o / sqrt(mean o^2 + eps) * weight; the gate is sigmoid(g_raw) per value
  channel.

Parity status: pinned by the CPU tests (library-routine convolution, closed
forms, identities, causality, packing, hand example).
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _bounds(T, cu_seqlens, num_seqs):
    if cu_seqlens is None:
        n = 1 if num_seqs is None else int(num_seqs)
        assert T % n == 0
        return [(i * (T // n), (i + 1) * (T // n)) for i in range(n)]
    cu = [int(c) for c in cu_seqlens]
    assert cu[0] == 0 and cu[-1] == T
    return list(zip(cu[:-1], cu[1:]))


def short_conv(x, w, cu_seqlens=None, num_seqs=None):
    """Causal depthwise convolution per sequence: x [T, H, d], w [H, d, W];
    y[t] = sum_i w[..., i] * x[t - (W-1) + i], zero before the sequence start.
    Tap i reads the input lag = W-1-i tokens back, so each tap adds the
    sequence shifted down by its lag."""
    x, w = _f64(x), _f64(w)
    T = x.shape[0]
    W = w.shape[-1]
    y = np.zeros_like(x)
    for bos, eos in _bounds(T, cu_seqlens, num_seqs):
        n = eos - bos
        for i in range(W):
            lag = W - 1 - i
            if lag < n:
                y[bos + lag:eos] += w[..., i] * x[bos:eos - lag]
    return y


def silu(x):
    x = _f64(x)
    return x / (1.0 + np.exp(-x))


def l2_normalize(x, eps):
    """x / sqrt(sum over the last axis of x^2 + eps)."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def logsigmoid(x):
    """log(1 / (1 + e^-x)) without overflow for either sign."""
    x = _f64(x)
    return -(np.maximum(-x, 0.0) + np.log1p(np.exp(-np.abs(x))))


def sigmoid(x):
    return np.exp(logsigmoid(x))


def frontend(q_raw, k_raw, v_raw, conv_q, conv_k, conv_v, a_raw, b_raw,
             cu_seqlens=None, num_seqs=None, eps=1e-6):
    """Projections -> recurrence inputs: returns (q, k, v, log_alpha, beta), fp64.

    q_raw, k_raw, a_raw: [T, H, dk]; v_raw: [T, H, dv]; b_raw: [T, H];
    conv_q, conv_k: [H, dk, W]; conv_v: [H, dv, W]."""
    q = l2_normalize(silu(short_conv(q_raw, conv_q, cu_seqlens, num_seqs)), eps)
    k = l2_normalize(silu(short_conv(k_raw, conv_k, cu_seqlens, num_seqs)), eps)
    v = silu(short_conv(v_raw, conv_v, cu_seqlens, num_seqs))
    return q, k, v, logsigmoid(a_raw), sigmoid(b_raw)


def gated_rmsnorm(o, g_raw, weight, eps):
    """o [T, H, dv] -> o / sqrt(mean(o^2) + eps) * weight * sigmoid(g_raw), fp64."""
    o, g, w = _f64(o), _f64(g_raw), _f64(weight)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o / rms * w * sigmoid(g)
