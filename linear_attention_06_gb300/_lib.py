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

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT, KDA_ERR_BOUNDS = range(6)
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
        L.kda_prefill_checkpointed.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.kda_prefill_checkpointed.restype = ctypes.c_int
        L.kda_check_checkpoints.argtypes = [vp, ctypes.c_int32, ctypes.c_int64, vp, vp]
        L.kda_check_checkpoints.restype = ctypes.c_int
        L.kda_check_cu_seqlens.argtypes = [vp, ctypes.c_int32, ctypes.c_int64]
        L.kda_check_cu_seqlens.restype = ctypes.c_int
        L.kda_device_status.argtypes = [vp]
        L.kda_device_status.restype = ctypes.c_int
        L.kda_selftest_timeout.argtypes = [ctypes.c_uint64, vp]
        L.kda_selftest_timeout.restype = ctypes.c_int
        L.kda_prefill_gated.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp]
        L.kda_prefill_gated.restype = ctypes.c_int
        L.kda_decode_step_gated.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp]
        L.kda_decode_step_gated.restype = ctypes.c_int
        L.kda_frontend.argtypes = [sp, ctypes.c_int32, ctypes.c_float] + [vp] * 15
        L.kda_frontend.restype = ctypes.c_int
        L.kda_prefill_split.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.kda_prefill_split.restype = ctypes.c_int
        L.kda_prefill_split_workspace_size.argtypes = [sp, ctypes.POINTER(ctypes.c_size_t)]
        L.kda_prefill_split_workspace_size.restype = ctypes.c_int
        L.kda_prefill_frontend.argtypes = [sp, ctypes.c_int32, ctypes.c_float] + [vp] * 13
        L.kda_prefill_frontend.restype = ctypes.c_int
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


def kda_prefill_split_workspace_size(total_tokens: int, num_seqs: int, H: int, dk: int = 128, dv: int = 128,
                                     dtype=torch.bfloat16) -> int:
    """Bytes of workspace kda_prefill_split needs for this shape (see ``include/kda.h``)."""
    shape = KdaShape(int(num_seqs), int(total_tokens), int(H), int(dk), int(dv),
                     KDA_BF16 if dtype == torch.bfloat16 else KDA_F32)
    n = ctypes.c_size_t(0)
    _check("kda_prefill_split_workspace_size", lib().kda_prefill_split_workspace_size(ctypes.byref(shape),
                                                                                      ctypes.byref(n)))
    return int(n.value)


def kda_prefill_split(q, k, v, log_alpha, beta, initial_state=None, cu_seqlens=None, out=None,
                      final_state=None, num_seqs=None, workspace=None, stream=None):
    """kda_prefill for few (sequence, head) pairs and long sequences: a chunk-local
    kernel over every chunk of every head, then a state-chain kernel per (sequence,
    head) (see ``include/kda.h``).  ``workspace`` is a CUDA uint8 tensor of at least
    kda_prefill_split_workspace_size bytes, allocated here when not given.  Returns
    (out, final_state)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is not None and not (isinstance(cu_seqlens, torch.Tensor) and cu_seqlens.is_cuda):
        host_cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu()
        kda_check_cu_seqlens(host_cu, T)
        cu_seqlens = host_cu.to(q.device)
    n = cu_seqlens.numel() - 1 if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    if final_state is True:
        final_state = torch.empty((n, H, dk, dv), dtype=torch.float32, device=q.device)
    shape = KdaShape(n, T, H, dk, dv, _dtype_code(q))
    need = kda_prefill_split_workspace_size(T, n, H, dk, dv, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = lib().kda_prefill_split(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                 _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check("kda_prefill_split", st)
    return out, final_state


def kda_prefill_checkpointed(q, k, v, log_alpha, beta, ckpt_pos, initial_state=None,
                             cu_seqlens=None, out=None, final_state=None, num_seqs=None,
                             stream=None):
    """kda_prefill that also returns the state after chosen token counts.

    ckpt_pos: list (one entry per sequence) of host lists of positions; each is a
    token count from the sequence start, a multiple of 64 or the sequence length.
    The tables are validated on the host, copied to the device, and the saved
    states returned as [total_checkpoints, H, dk, dv] fp32 with the checkpoints
    of sequence 0 first.  Returns (out, final_state, checkpoint_states).
    """
    T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        n = 1 if num_seqs is None else int(num_seqs)
        host_cu = torch.arange(n + 1, dtype=torch.int32) * (T // n)
    elif isinstance(cu_seqlens, torch.Tensor) and cu_seqlens.is_cuda:
        host_cu = cu_seqlens.cpu().to(torch.int32)
    else:
        host_cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu()
    n = host_cu.numel() - 1
    if len(ckpt_pos) != n:
        raise ValueError("ckpt_pos needs one list per sequence")
    counts = [len(p) for p in ckpt_pos]
    ck_cu = torch.tensor([0] + list(torch.tensor(counts).cumsum(0).tolist()) if n else [0], dtype=torch.int32)
    ck_pos = torch.tensor([int(x) for p in ckpt_pos for x in p] or [0], dtype=torch.int32)
    st = lib().kda_check_checkpoints(ctypes.c_void_p(host_cu.contiguous().data_ptr()), n, T,
                                     ctypes.c_void_p(ck_cu.data_ptr()), ctypes.c_void_p(ck_pos.data_ptr()))
    _check("kda_check_checkpoints", st)
    dev = q.device
    d_cu = host_cu.to(dev)
    d_ck_cu, d_ck_pos = ck_cu.to(dev), ck_pos.to(dev)
    total = int(ck_cu[-1])
    ck_states = torch.empty((max(total, 1), H, dk, dv), dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    if final_state is True:
        final_state = torch.empty((n, H, dk, dv), dtype=torch.float32, device=dev)
    shape = KdaShape(n, T, H, dk, dv, _dtype_code(q))
    st = lib().kda_prefill_checkpointed(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                        _ptr(beta), _ptr(initial_state), _ptr(d_cu), _ptr(out),
                                        _ptr(final_state), _ptr(d_ck_cu), _ptr(d_ck_pos),
                                        _ptr(ck_states), _stream(stream))
    _check("kda_prefill_checkpointed", st)
    return out, final_state, ck_states[:total]


def kda_prefill_gated(q, k, v, log_alpha, beta, gate, norm_weight, norm_eps=1e-6, initial_state=None,
                      cu_seqlens=None, out=None, final_state=None, num_seqs=None, stream=None):
    """kda_prefill whose output is RMSNorm(o) * norm_weight * sigmoid(gate) per
    (token, head) (see ``include/kda.h``).  gate: [T, H, dv] like v; norm_weight:
    [dv] fp32.  Returns (out, final_state)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is not None and not (isinstance(cu_seqlens, torch.Tensor) and cu_seqlens.is_cuda):
        host_cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu()
        kda_check_cu_seqlens(host_cu, T)
        cu_seqlens = host_cu.to(q.device)
    n = cu_seqlens.numel() - 1 if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    if final_state is True:
        final_state = torch.empty((n, H, dk, dv), dtype=torch.float32, device=q.device)
    shape = KdaShape(n, T, H, dk, dv, _dtype_code(q))
    st = lib().kda_prefill_gated(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                 _ptr(initial_state), _ptr(cu_seqlens), _ptr(gate), _ptr(norm_weight),
                                 float(norm_eps), _ptr(out), _ptr(final_state), _stream(stream))
    _check("kda_prefill_gated", st)
    return out, final_state


def kda_decode_step_gated(q, k, v, log_alpha, beta, gate, norm_weight, state, norm_eps=1e-6, out=None,
                          stream=None):
    """kda_decode_step whose output is gated like kda_prefill_gated; state in place."""
    rows, H, dk = q.shape
    dv = v.shape[2]
    N = state.shape[0]
    if out is None:
        out = torch.empty((rows, H, dv), dtype=q.dtype, device=q.device)
    shape = KdaShape(N, rows, H, dk, dv, _dtype_code(q))
    st = lib().kda_decode_step_gated(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                     _ptr(beta), _ptr(gate), _ptr(norm_weight), float(norm_eps), _ptr(state),
                                     _ptr(out), _stream(stream))
    _check("kda_decode_step_gated", st)
    return out


def kda_frontend(q_raw, k_raw, v_raw, a_raw, b_raw, conv_q, conv_k, conv_v, cu_seqlens=None,
                 num_seqs=None, eps=1e-6, out=None, stream=None):
    """Layer front end (see ``include/kda.h``): short convolution + SiLU (+ L2 norm
    for q, k), logsigmoid for the decay, sigmoid for beta.

    q_raw, k_raw: [T, H, dk]; v_raw: [T, H, dv]; b_raw: [T, H] (bf16 or fp32);
    a_raw: [T, H, dk] fp32; conv_q, conv_k: [H, dk, W], conv_v: [H, dv, W] fp32.
    Returns (q, k, v, log_alpha, beta) in kda_prefill's input layout, or fills
    ``out`` (a tuple of five tensors) when given."""
    T, H, dk = q_raw.shape
    dv = v_raw.shape[2]
    W = conv_q.shape[-1]
    if cu_seqlens is not None and not (isinstance(cu_seqlens, torch.Tensor) and cu_seqlens.is_cuda):
        host_cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu()
        kda_check_cu_seqlens(host_cu, T)
        cu_seqlens = host_cu.to(q_raw.device)
    n = cu_seqlens.numel() - 1 if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    dev, dt = q_raw.device, q_raw.dtype
    if out is None:
        out = (torch.empty((T, H, dk), dtype=dt, device=dev), torch.empty((T, H, dk), dtype=dt, device=dev),
               torch.empty((T, H, dv), dtype=dt, device=dev),
               torch.empty((T, H, dk), dtype=torch.float32, device=dev),
               torch.empty((T, H), dtype=dt, device=dev))
    q, k, v, la, beta = out
    shape = KdaShape(n, T, H, dk, dv, _dtype_code(q_raw))
    st = lib().kda_frontend(ctypes.byref(shape), int(W), float(eps), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw),
                            _ptr(a_raw), _ptr(b_raw), _ptr(conv_q), _ptr(conv_k), _ptr(conv_v),
                            _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(beta),
                            _stream(stream))
    _check("kda_frontend", st)
    return q, k, v, la, beta


def kda_prefill_frontend(q_raw, k_raw, v_raw, a_raw, b_raw, conv_q, conv_k, conv_v, initial_state=None,
                         cu_seqlens=None, out=None, final_state=None, num_seqs=None, eps=1e-6, stream=None):
    """The layer front end and the prefill in one pass (see ``include/kda.h``): raw
    projections in (as kda_frontend takes them), (out, final_state) out."""
    T, H, dk = q_raw.shape
    dv = v_raw.shape[2]
    W = conv_q.shape[-1]
    if cu_seqlens is not None and not (isinstance(cu_seqlens, torch.Tensor) and cu_seqlens.is_cuda):
        host_cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu()
        kda_check_cu_seqlens(host_cu, T)
        cu_seqlens = host_cu.to(q_raw.device)
    n = cu_seqlens.numel() - 1 if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    if out is None:
        out = torch.empty((T, H, dv), dtype=q_raw.dtype, device=q_raw.device)
    if final_state is True:
        final_state = torch.empty((n, H, dk, dv), dtype=torch.float32, device=q_raw.device)
    shape = KdaShape(n, T, H, dk, dv, _dtype_code(q_raw))
    st = lib().kda_prefill_frontend(ctypes.byref(shape), int(W), float(eps), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw),
                                    _ptr(a_raw), _ptr(b_raw), _ptr(conv_q), _ptr(conv_k), _ptr(conv_v),
                                    _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                    _stream(stream))
    _check("kda_prefill_frontend", st)
    return out, final_state


def kda_decode_step(q, k, v, log_alpha, beta, state, out=None, stream=None):
    """Decode step of T tokens per sequence (see ``include/kda.h``).

    state: [N, H, dk, dv] fp32, updated in place.  q, k, log_alpha: [N*T, H, dk];
    v: [N*T, H, dv]; beta: [N*T, H]; rows n*T .. n*T+T-1 belong to sequence n
    (T = 1 is the one-token step).  Returns out [N*T, H, dv]."""
    rows, H, dk = q.shape
    dv = v.shape[2]
    N = state.shape[0]
    if out is None:
        out = torch.empty((rows, H, dv), dtype=q.dtype, device=q.device)
    shape = KdaShape(N, rows, H, dk, dv, _dtype_code(q))
    st = lib().kda_decode_step(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                               _ptr(beta), _ptr(state), _ptr(out), _stream(stream))
    _check("kda_decode_step", st)
    return out


def kda_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(lib().kda_device_status(_stream(stream)))


def kda_selftest_timeout(limit_ns: int = 1_000_000, stream=None) -> None:
    """Enqueue the timeout-path self test (see ``include/kda.h``): a bounded wait that
    nothing completes gives up after ``limit_ns`` and sets the status word, so the next
    kda_device_status returns KDA_ERR_TIMEOUT."""
    _check("kda_selftest_timeout", lib().kda_selftest_timeout(int(limit_ns), _stream(stream)))
