"""fp64 CPU oracle for Kimi Delta Attention (KDA) -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may import this module.  The product path (the CUDA library and its Python
binding) never does.  This module shares no code with the CUDA library; it
compiles and loads ``kda_oracle.c`` from this directory.

The recurrence it computes, token by token in fp64, is

    S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
    o_t = S_t^T q_t

following "Kimi K3 Architecture Teardown" (section "Hybrid Attention for 1M
Tokens", Visual 5: decay each channel, erase the beta-scaled share stored
under the key, write the new pair) and "Kimi K3 Architecture: KDA, MoE, and
Attention" (section "Memory as a First-Class Problem": one beta for erase and
write; the output reads the updated state).

Parity status: pinned (see the CPU test suite: brute-force unrolled products,
closed forms, invariants, mutants and a hand-derived example).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lib = None


def build(out_path: str = _LIB_PATH, mutation: int = 0) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, no FP contraction).

    ``mutation`` > 0 compiles a deliberately wrong variant used only by the
    test that proves the pins catch plausible mistakes.
    """
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", out_path, _SRC, "-lm"]
    if mutation:
        cmd.insert(1, f"-DKDA_ORACLE_MUTATION={int(mutation)}")
    subprocess.run(cmd, check=True)
    return out_path


def _bind(lib):
    i64, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.kda_oracle_prefill.argtypes = [i64, dp, i64, i64, i64, dp, dp, dp, dp, dp,
                                       dp, dp, dp, ip]
    lib.kda_oracle_prefill.restype = ctypes.c_int
    lib.kda_oracle_decode_step.argtypes = [i64, i64, i64, i64, dp, dp, dp, dp, dp,
                                           dp, dp, ip]
    lib.kda_oracle_decode_step.restype = ctypes.c_int
    lib.kda_oracle_max_threads.argtypes = []
    lib.kda_oracle_max_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def load_mutant(mutation: int):
    """Build and load a mutant oracle into a temporary directory."""
    d = tempfile.mkdtemp(prefix="kda_oracle_mut")
    return load(build(os.path.join(d, f"libkda_oracle_m{mutation}.so"), mutation))


def max_threads() -> int:
    return int(load().kda_oracle_max_threads())


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def prefill(q, k, v, log_alpha, beta, initial_state=None, cu_seqlens=None,
            num_seqs=None, num_threads=0, lib=None):
    """Run the oracle over packed sequences.

    q, k, log_alpha: [T, H, dk]; v: [T, H, dv]; beta: [T, H] (any float dtype,
    widened exactly to fp64).  cu_seqlens: [N+1] token offsets; if None, the T
    tokens are split into ``num_seqs`` (default 1) equal sequences.
    initial_state: [N, H, dk, dv] or None (zeros).
    Returns (out [T, H, dv], final_state [N, H, dk, dv]) as fp64 arrays.
    """
    lib = lib or load()
    q, k, v, la, b = _f64(q), _f64(k), _f64(v), _f64(log_alpha), _f64(beta)
    T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        n = 1 if num_seqs is None else int(num_seqs)
        assert T % n == 0
        cu = np.arange(n + 1, dtype=np.int64) * (T // n)
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        n = cu.shape[0] - 1
    assert k.shape == (T, H, dk) and la.shape == (T, H, dk)
    assert v.shape == (T, H, dv) and b.shape == (T, H)
    assert cu[0] == 0 and cu[-1] == T
    h0 = None if initial_state is None else _f64(initial_state)
    if h0 is not None:
        assert h0.shape == (n, H, dk, dv)
    out = np.zeros((T, H, dv), dtype=np.float64)
    fin = np.zeros((n, H, dk, dv), dtype=np.float64)
    rc = lib.kda_oracle_prefill(n, _ptr(cu), H, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                                _ptr(la), _ptr(b), _ptr(h0), _ptr(out), _ptr(fin),
                                int(num_threads))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_prefill failed ({rc})")
    return out, fin


def decode_step(q, k, v, log_alpha, beta, state, num_threads=0, lib=None):
    """One token per sequence.  q, k, log_alpha: [N, H, dk]; v: [N, H, dv];
    beta: [N, H]; state: [N, H, dk, dv].  Returns (out, new_state) in fp64."""
    lib = lib or load()
    q, k, v, la, b = _f64(q), _f64(k), _f64(v), _f64(log_alpha), _f64(beta)
    S = _f64(state).copy()
    N, H, dk = q.shape
    dv = v.shape[2]
    out = np.zeros((N, H, dv), dtype=np.float64)
    rc = lib.kda_oracle_decode_step(N, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(la),
                                    _ptr(b), _ptr(S), _ptr(out), int(num_threads))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_decode_step failed ({rc})")
    return out, S
