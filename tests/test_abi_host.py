"""Host-side tests of the C ABI (no GPU needed).

The library must build for sm_103a, load, export every symbol that
include/kda.h declares, and reject bad arguments on the host before any CUDA
call (so these calls use placeholder pointers that are never dereferenced).
"""
import ctypes
import os
import re

import pytest

from linear_attention_06_gb300 import _lib
from linear_attention_06_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")

FAKE = 0x10000            # 16-byte aligned, never dereferenced
FAKE_MIS = 0x10002        # misaligned


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return _lib.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"kda_prefill", "kda_decode_step", "kda_status_string", "kda_version"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} is declared in kda.h but not exported"


def test_status_strings_and_version(L):
    assert _lib.status_string(0) == "KDA_OK"
    assert _lib.status_string(4) == "KDA_ERR_TIMEOUT"
    assert _lib.status_string(5) == "KDA_ERR_BOUNDS"
    assert _lib.status_string(99) == "KDA_ERR_UNKNOWN"
    assert "sm_103a" in _lib.version()


@pytest.mark.parametrize("cu,T,ok", [
    ([0, 3, 5], 5, True), ([0], 0, True), ([0, 0, 0], 0, True),
    ([1, 3], 3, False), ([0, 3, 2], 2, False), ([0, 3, 5], 6, False)])
def test_check_cu_seqlens(L, cu, T, ok):
    if ok:
        _lib.kda_check_cu_seqlens(cu, T)
    else:
        with pytest.raises(_lib.KdaError):
            _lib.kda_check_cu_seqlens(cu, T)


def shape(n=2, T=128, H=4, dk=128, dv=128, dt=_lib.KDA_BF16):
    return _lib.KdaShape(n, T, H, dk, dv, dt)


def prefill(L, sh, q=FAKE, k=FAKE, v=FAKE, la=FAKE, b=FAKE, h0=None, cu=None, out=FAKE, fin=None):
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return L.kda_prefill(ctypes.byref(sh) if sh is not None else None, p(q), p(k), p(v), p(la),
                         p(b), p(h0), p(cu), p(out), p(fin), None)


def decode(L, sh, q=FAKE, k=FAKE, v=FAKE, la=FAKE, b=FAKE, S=FAKE, out=FAKE):
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return L.kda_decode_step(ctypes.byref(sh), p(q), p(k), p(v), p(la), p(b), p(S), p(out), None)


def test_prefill_rejects_bad_arguments_before_any_cuda_call(L):
    E_ARG, E_UNS = _lib.KDA_ERR_INVALID_ARG, _lib.KDA_ERR_UNSUPPORTED
    assert prefill(L, None) == E_ARG
    for kw in ("q", "k", "v", "la", "b", "out"):
        assert prefill(L, shape(), **{kw: None}) == E_ARG, kw
    assert prefill(L, shape(n=-1)) == E_ARG
    assert prefill(L, shape(T=-5)) == E_ARG
    assert prefill(L, shape(H=0)) == E_ARG
    assert prefill(L, shape(n=0, T=10)) == E_ARG
    assert prefill(L, shape(n=3, T=128)) == E_ARG          # 128 % 3 != 0 without cu_seqlens
    assert prefill(L, shape(dk=96)) == E_UNS
    assert prefill(L, shape(dv=32)) == E_UNS
    assert prefill(L, shape(dt=7)) == E_UNS
    assert prefill(L, shape(), q=FAKE_MIS) == E_UNS
    assert prefill(L, shape(), la=FAKE + 4) == E_UNS
    assert prefill(L, shape(), b=FAKE + 1) == E_UNS          # bf16 beta must be 2-byte aligned
    assert prefill(L, shape(dt=_lib.KDA_F32), b=FAKE + 2) == E_UNS
    assert prefill(L, shape(), h0=FAKE + 8) == E_UNS
    assert prefill(L, shape(), fin=FAKE + 8) == E_UNS
    assert prefill(L, shape(), cu=FAKE + 2) == E_UNS


def test_empty_calls_are_noops(L):
    assert prefill(L, shape(n=0, T=0), q=None, k=None, v=None, la=None, b=None, out=None) == 0
    assert decode(L, shape(n=0, T=0), q=None, k=None, v=None, la=None, b=None, S=None,
                  out=None) == 0


def test_decode_rejects_bad_arguments(L):
    E_ARG, E_UNS = _lib.KDA_ERR_INVALID_ARG, _lib.KDA_ERR_UNSUPPORTED
    assert decode(L, shape(n=4, T=5)) == E_ARG               # one token per sequence
    assert decode(L, shape(n=4, T=4), S=None) == E_ARG
    assert decode(L, shape(n=4, T=4), q=None) == E_ARG
    assert decode(L, shape(n=4, T=4), S=FAKE + 4) == E_UNS
    assert decode(L, shape(n=4, T=4, dk=32)) == E_UNS


def test_valid_call_without_gpu_reports_cuda_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert prefill(L, shape()) == _lib.KDA_ERR_CUDA


def test_selftest_timeout_rejects_limits_out_of_range(L):
    # checked on the host before any CUDA call
    for bad in (0, 999, 1_000_000_001, 2**63):
        assert L.kda_selftest_timeout(bad, None) == _lib.KDA_ERR_INVALID_ARG


def test_decode_multi_token_argument_rules(L):
    E_ARG, E_UNS = _lib.KDA_ERR_INVALID_ARG, _lib.KDA_ERR_UNSUPPORTED
    assert decode(L, shape(n=4, T=4 * 17)) == E_UNS         # more than 16 tokens per sequence
    assert decode(L, shape(n=4, T=0)) == E_ARG
    assert decode(L, shape(n=4, T=10)) == E_ARG              # not a multiple of num_seqs


def test_check_checkpoints_host_rules(L):
    import numpy as np
    def chk(cu, ck_cu, ck_pos):
        cu = np.asarray(cu, dtype=np.int32); a = np.asarray(ck_cu, dtype=np.int32)
        b = np.asarray(ck_pos or [0], dtype=np.int32)
        return L.kda_check_checkpoints(cu.ctypes.data, len(cu) - 1, int(cu[-1]), a.ctypes.data, b.ctypes.data)
    assert chk([0, 200, 264], [0, 3, 4], [64, 128, 200, 64]) == 0
    assert chk([0, 200], [0, 1], [100]) == _lib.KDA_ERR_INVALID_ARG       # not a chunk end
    assert chk([0, 200], [0, 2], [128, 64]) == _lib.KDA_ERR_INVALID_ARG   # not increasing
    assert chk([0, 200], [0, 1], [256]) == _lib.KDA_ERR_INVALID_ARG       # past the end
    assert chk([0, 200], [0, 0], []) == 0


def test_prefill_checkpointed_rejects_null_tables(L):
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    sh = shape()
    args = [ctypes.byref(sh)] + [p(FAKE)] * 5 + [None, None, p(FAKE), None]
    assert L.kda_prefill_checkpointed(*args, None, p(FAKE), p(FAKE), None) == _lib.KDA_ERR_INVALID_ARG
    assert L.kda_prefill_checkpointed(*args, p(FAKE), p(FAKE), p(FAKE + 8), None) == _lib.KDA_ERR_UNSUPPORTED


def frontend_call(L, sh, W=4, eps=1e-6, ptrs=None, conv=FAKE):
    p = ptrs or FAKE
    P = ctypes.c_void_p
    return L.kda_frontend(ctypes.byref(sh), W, ctypes.c_float(eps), P(p), P(p), P(p), P(p), P(p),
                          P(conv), P(conv), P(conv), None, P(p), P(p), P(p), P(p), P(p), None)


@pytest.mark.parametrize("W,eps,code", [(0, 1e-6, 2), (5, 1e-6, 2), (4, -1.0, 1), (4, 0.0, 1),
                                        (4, float("nan"), 1), (4, float("inf"), 1)])
def test_frontend_rejects_width_and_eps(L, W, eps, code):
    assert frontend_call(L, shape(), W=W, eps=eps) == code


def test_frontend_rejects_pointers_and_shapes(L):
    assert frontend_call(L, shape(), conv=0) == 1                 # null conv taps
    assert frontend_call(L, shape(), ptrs=FAKE_MIS) == 2          # misaligned tensors
    assert frontend_call(L, shape(dk=96)) == 2                    # unsupported head size
    assert frontend_call(L, shape(n=3, T=128)) == 1               # T % N without cu_seqlens
    assert frontend_call(L, shape(n=0, T=0)) == 0                 # empty: nothing enqueued


def gated_prefill_call(L, sh, gate=FAKE, w=FAKE, eps=1e-6):
    P = ctypes.c_void_p
    return L.kda_prefill_gated(ctypes.byref(sh), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, None,
                               P(gate), P(w), ctypes.c_float(eps), P(FAKE), None, None)


def test_gated_prefill_rejects_gate_arguments(L):
    assert gated_prefill_call(L, shape(), gate=0) == 1
    assert gated_prefill_call(L, shape(), w=0) == 1
    assert gated_prefill_call(L, shape(), eps=-1.0) == 1
    assert gated_prefill_call(L, shape(), eps=0.0) == 1             # 0/0 on an all-zero row
    assert gated_prefill_call(L, shape(), eps=float("nan")) == 1
    assert gated_prefill_call(L, shape(), gate=FAKE_MIS) == 2
    assert gated_prefill_call(L, shape(n=0, T=0), gate=0) == 0      # empty: nothing checked, nothing enqueued


def test_gated_decode_rejects_gate_arguments(L):
    P = ctypes.c_void_p
    sh = shape(n=4, T=4)
    call = lambda g, w, e: L.kda_decode_step_gated(ctypes.byref(sh), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                                   P(FAKE), P(g), P(w), ctypes.c_float(e), P(FAKE), P(FAKE), None)
    assert call(0, FAKE, 1e-6) == 1
    assert call(FAKE, 0, 1e-6) == 1
    assert call(FAKE, FAKE, -2.0) == 1
    assert call(FAKE, FAKE, 0.0) == 1
    assert call(FAKE_MIS, FAKE, 1e-6) == 2


def split(L, sh, ws=FAKE, nbytes=1 << 40, **kw):
    p = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    a = dict(q=FAKE, k=FAKE, v=FAKE, la=FAKE, b=FAKE, h0=None, cu=None, out=FAKE, fin=None)
    a.update(kw)
    return L.kda_prefill_split(ctypes.byref(sh), p(a["q"]), p(a["k"]), p(a["v"]), p(a["la"]), p(a["b"]),
                               p(a["h0"]), p(a["cu"]), p(a["out"]), p(a["fin"]), p(ws), nbytes, None)


def test_split_workspace_size_depends_on_the_shape_only(L):
    def size(n, T, H):
        b = ctypes.c_size_t(0)
        assert L.kda_prefill_split_workspace_size(ctypes.byref(shape(n=n, T=T, H=H)), ctypes.byref(b)) == 0
        return b.value
    rec = 12 * 8192
    # one long sequence runs in segments of 8192 tokens: two carried fp32 states per head and
    # the records of two segments (8192 / 64 + 1 slots a head each)
    seg_slots = 32 * (8192 // 64 + 1)
    seg_buf = (seg_slots * 4 + 1023) // 1024 * 1024 + seg_slots * rec
    assert size(1, 131072, 32) == 2 * 32 * 128 * 128 * 4 + 2 * seg_buf
    assert size(1, 10 ** 7, 32) == size(1, 131072, 32)           # independent of the length
    slots = 32 * ((16383 + 63) // 64 + 1)                         # below two segments: one pass
    assert size(1, 16383, 32) == (slots * 4 + 1023) // 1024 * 1024 + slots * rec
    slots = 32 * ((131072 + 63) // 64 + 2)                         # two sequences: one pass
    assert size(2, 131072, 32) == (slots * 4 + 1023) // 1024 * 1024 + slots * rec
    assert size(3, 100, 2) == 1024 + 2 * (2 + 3) * rec          # ceil(100/64) + 3 slots a head
    assert size(0, 0, 4) == 0
    assert L.kda_prefill_split_workspace_size(ctypes.byref(shape()), None) == _lib.KDA_ERR_INVALID_ARG
    b = ctypes.c_size_t(7)
    assert L.kda_prefill_split_workspace_size(ctypes.byref(shape(dk=96)), ctypes.byref(b)) == _lib.KDA_ERR_UNSUPPORTED
    assert b.value == 0


def test_split_rejects_bad_workspace_before_any_cuda_call(L):
    E_ARG, E_UNS = _lib.KDA_ERR_INVALID_ARG, _lib.KDA_ERR_UNSUPPORTED
    assert split(L, shape(), ws=None) == E_ARG
    assert split(L, shape(), ws=FAKE + 16) == E_UNS           # not 256-byte aligned
    assert split(L, shape(), nbytes=1024) == E_ARG            # too small
    assert split(L, shape(), q=None) == E_ARG
    assert split(L, shape(n=3, T=128)) == E_ARG
    assert split(L, shape(dk=96)) == E_UNS
    assert split(L, shape(n=0, T=0), ws=None, q=None, k=None, v=None, la=None, b=None, out=None) == 0


def test_prefill_frontend_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    def call(sh, W=4, eps=1e-6, ptrs=FAKE, conv=FAKE, out=FAKE):
        return L.kda_prefill_frontend(ctypes.byref(sh), W, ctypes.c_float(eps), P(ptrs), P(ptrs), P(ptrs), P(ptrs),
                                      P(ptrs), P(conv), P(conv), P(conv), None, None, P(out), None, None)
    E_ARG, E_UNS = _lib.KDA_ERR_INVALID_ARG, _lib.KDA_ERR_UNSUPPORTED
    assert call(shape(), W=0) == E_UNS and call(shape(), W=5) == E_UNS
    assert call(shape(), eps=0.0) == E_ARG and call(shape(), eps=float("nan")) == E_ARG
    assert call(shape(), conv=0) == E_ARG
    assert call(shape(), ptrs=0) == E_ARG
    assert call(shape(), ptrs=FAKE_MIS) == E_UNS
    assert call(shape(dk=64, dv=64)) == E_UNS                  # the tensor-core path only
    assert call(shape(dt=_lib.KDA_F32)) == E_UNS
    assert call(shape(n=3, T=128)) == E_ARG
    assert call(shape(n=0, T=0), ptrs=0, conv=0, out=0) == 0
