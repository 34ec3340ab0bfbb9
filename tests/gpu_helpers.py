"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import linear_attention_06_gb300 as kda
from oracle import kda_oracle

TOL = {torch.float32: 1e-4, torch.bfloat16: 5e-3}   # relative L2, from the target spec


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def np64(t):
    return None if t is None else t.detach().float().cpu().numpy().astype(np.float64)


def gpu_prefill(w, cu_on_device=True, **kw):
    dev = w.q.device
    cu = w.cu_seqlens.to(dev) if cu_on_device else w.cu_seqlens
    out, fin = kda.kda_prefill(w.q, w.k, w.v, w.log_alpha, w.beta, w.initial_state, cu,
                               final_state=True, **kw)
    torch.cuda.synchronize()
    return out, fin


def oracle_prefill(w, heads=None):
    """Oracle on the given heads (all if None); returns out [T,h,dv], fin [N,h,dk,dv]."""
    sel = slice(None) if heads is None else list(heads)
    def pick(t):
        return np64(t[:, sel]) if t is not None else None
    h0 = None if w.initial_state is None else np64(w.initial_state[:, sel])
    return kda_oracle.prefill(pick(w.q), pick(w.k), pick(w.v), pick(w.log_alpha), pick(w.beta),
                              h0, cu_seqlens=w.cu_seqlens.numpy())


def compare_prefill(w, heads=None, tol=None, **kw):
    """GPU vs oracle; returns (err_out, err_state) and asserts the tolerance."""
    out, fin = gpu_prefill(w, **kw)
    ro, rf = oracle_prefill(w, heads)
    sel = slice(None) if heads is None else list(heads)
    e_out = rel_l2(np64(out[:, sel]), ro)
    e_fin = rel_l2(np64(fin[:, sel]), rf)
    tol = TOL[w.q.dtype] if tol is None else tol
    assert e_out <= tol and e_fin <= tol, f"{w.name}: out {e_out:.3e} state {e_fin:.3e} > {tol}"
    return e_out, e_fin
