"""Independent fp64 formulations used to pin the oracle (CPU only).

Nothing here shares code with the oracle's C loop or with the CUDA library.

* ``unrolled_products`` builds every transition as an explicit dk x dk matrix
  M_t = (I - beta_t k_t k_t^T) Diag(alpha_t) and evaluates the closed form of
  the linear recurrence S_t = M_t S_{t-1} + beta_t k_t v_t^T:

      S_t = (M_t ... M_1) S_0 + sum_{s <= t} (M_t ... M_{s+1}) beta_s k_s v_s^T,
      o_t = S_t^T q_t.

  This is the matrix form of the recurrence that anchors the pages' prose
  ("Kimi K3 Architecture Teardown", Visual 5; "Kimi K3 Architecture: KDA, MoE,
  and Attention", section "Memory as a First-Class Problem").

* ``gated_deltanet`` is the scalar-gate delta rule written in the other common
  orientation (state H = S^T of shape dv x dk, updated on the right):
      H_t = g_t H_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = H_t q_t.
  With g_t = 1 it is DeltaNet.  "Kimi K3 architecture: KDA, MLA and MoE",
  section "KDA is a writable state", names DeltaNet and Gated DeltaNet as the
  rules KDA refines (KDA makes the decay per channel), so KDA with a
  channel-uniform alpha must agree with it.
"""
from __future__ import annotations

import numpy as np


def unrolled_products(q, k, v, log_alpha, beta, S0):
    """One (sequence, head): q, k, log_alpha [T, dk]; v [T, dv]; beta [T];
    S0 [dk, dv].  Returns (out [T, dv], S_T [dk, dv]); intended for T <= 16."""
    q, k, v, la, b, S0 = (np.asarray(x, dtype=np.float64) for x in (q, k, v, log_alpha, beta, S0))
    T, dk = k.shape
    eye = np.eye(dk)
    M = [(eye - b[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(la[t])) for t in range(T)]
    W = [b[t] * np.outer(k[t], v[t]) for t in range(T)]
    out = np.zeros((T, v.shape[1]))
    S_t = S0
    for t in range(T):
        # product M_t ... M_{s+1} for every s, built from scratch for each t
        acc = np.zeros_like(S0)
        for s in range(-1, t + 1):
            P = eye.copy()
            for u in range(t, s, -1):
                P = P @ M[u]
            acc = acc + (P @ S0 if s == -1 else P @ W[s])
        S_t = acc
        out[t] = S_t.T @ q[t]
    return out, S_t


def gated_deltanet(q, k, v, log_g, beta, S0):
    """Scalar gate per token (log_g [T]); state kept as H = S^T [dv, dk]."""
    q, k, v, lg, b, S0 = (np.asarray(x, dtype=np.float64) for x in (q, k, v, log_g, beta, S0))
    T, dk = k.shape
    Hs = S0.T.copy()
    out = np.zeros((T, v.shape[1]))
    for t in range(T):
        g = np.exp(lg[t])
        Hs = g * Hs @ (np.eye(dk) - b[t] * np.outer(k[t], k[t])) + b[t] * np.outer(v[t], k[t])
        out[t] = Hs @ q[t]
    return out, Hs.T
