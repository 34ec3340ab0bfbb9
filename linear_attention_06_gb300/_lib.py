"""Thin ctypes binding of libkda (argument marshalling only).

Every step of the KDA path runs in the CUDA library; this module only turns
torch tensors into the pointers, sizes and stream that ``include/kda.h``
declares, allocates output tensors when the caller does not pass them, and
raises on a non-OK status.  There is no CPU fallback: if ``libkda.so`` is
missing, loading fails with an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = range(5)
KDA_BF16, KDA_F32 = 0, 1


class KdaShape(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int64),
                ("H", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("dtype", ctypes.c_int)]


class KdaError(RuntimeError):
    def __init__(self, fn, status, name):
        super().__init__(f"{fn} returned {name} ({status})")
        self.status = status


_lib = None


def lib():
    """The loaded libkda (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libkda.so not found at {LIB_PATH}: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, sp = ctypes.c_void_p, ctypes.POINTER(KdaShape)
        L.kda_prefill.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.kda_prefill.restype = ctypes.c_int
        L.kda_decode_step.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.kda_decode_step.restype = ctypes.c_int
        L.kda_check_cu_seqlens.argtypes = [vp, ctypes.c_int32, ctypes.c_int64]
        L.kda_check_cu_seqlens.restype = ctypes.c_int
        L.kda_device_status.argtypes = [vp]
        L.kda_device_status.restype = ctypes.c_int
        L.kda_status_string.argtypes = [ctypes.c_int]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_version.argtypes = []
        L.kda_version.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def version() -> str:
    return lib().kda_version().decode()


def _check(fn, status):
    if status != KDA_OK:
        raise KdaError(fn, status, status_string(status))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def kda_check_cu_seqlens(cu_seqlens, total_tokens: int) -> None:
    """Validate a host cu_seqlens table (list, numpy array or CPU tensor)."""
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu().contiguous()
    st = lib().kda_check_cu_seqlens(ctypes.c_void_p(cu.data_ptr()), cu.numel() - 1,
                                    int(total_tokens))
    _check("kda_check_cu_seqlens", st)


def kda_prefill(q, k, v, log_alpha, beta, initial_state=None, cu_seqlens=None, out=None,
                final_state=None, num_seqs=None, stream=None):
    """KDA prefill over packed sequences (see ``include/kda.h``).

    q, k: [T, H, dk]; v: [T, H, dv]; log_alpha: [T, H, dk] fp32; beta: [T, H];
    all CUDA tensors, q/k/v/beta bf16 or fp32.  ``cu_seqlens`` is a CUDA int32
    tensor, or a host table (validated on the host, then copied); None means
    ``num_seqs`` (default 1) equal sequences.  ``final_state`` may be a tensor
    to fill, True to allocate one, or None.  Returns (out, final_state).
    """
    T, H, dk = q.shape
    dv = v.shape[2]
    host_cu = None
    if cu_seqlens is not None and not (isinstance(cu_seqlens, torch.Tensor) and cu_seqlens.is_cuda):
        host_cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu()
        kda_check_cu_seqlens(host_cu, T)
        cu_seqlens = host_cu.to(q.device, non_blocking=False)
    if cu_seqlens is not None:
        n = cu_seqlens.numel() - 1
    else:
        n = 1 if num_seqs is None else int(num_seqs)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    if final_state is True:
        final_state = torch.empty((n, H, dk, dv), dtype=torch.float32, device=q.device)
    shape = KdaShape(n, T, H, dk, dv, _dtype_code(q))
    st = lib().kda_prefill(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                           _ptr(beta), _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                           _ptr(final_state), _stream(stream))
    _check("kda_prefill", st)
    return out, final_state


def kda_decode_step(q, k, v, log_alpha, beta, state, out=None, stream=None):
    """One decode step: q, k, log_alpha [N, H, dk]; v [N, H, dv]; beta [N, H];
    state [N, H, dk, dv] fp32 updated in place.  Returns out [N, H, dv]."""
    N, H, dk = q.shape
    dv = v.shape[2]
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    shape = KdaShape(N, N, H, dk, dv, _dtype_code(q))
    st = lib().kda_decode_step(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                               _ptr(beta), _ptr(state), _ptr(out), _stream(stream))
    _check("kda_decode_step", st)
    return out


def kda_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(lib().kda_device_status(_stream(stream)))
