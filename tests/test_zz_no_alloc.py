"""The no-allocation split prefill (kda_prefill_split_static) through the C ABI.

kda_prefill_split_static is for callers that cannot allocate device memory where they
run (inside another framework's memory pool, under a fixed memory budget, without an
allocator handle): it runs the split prefill on a fixed scratch array owned by the
library.  Here it is called straight through ctypes, twice in a row with different
inputs on the shared array, and each result is compared with kda_prefill_split run on a
caller workspace, within the bf16 tolerance of the other parity tests.  This file is
collected last, and passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import pytest
import torch

from linear_attention_06_gb300 import _lib, workloads
import linear_attention_06_gb300 as kda
from tests.gpu_helpers import np64, oracle_prefill, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 5e-3                                   # relative L2, bf16 inputs


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_06_gb300 import build
    build.build()
    lib = _lib.lib()
    f = lib.kda_prefill_split_static
    f.argtypes = [ctypes.POINTER(_lib.KdaShape)] + [ctypes.c_void_p] * 10
    f.restype = ctypes.c_int
    return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def static_prefill(L, w, cu):
    n = cu.numel() - 1
    out = torch.empty_like(w.v)
    fin = torch.empty((n, w.q.shape[1], 128, 128), dtype=torch.float32, device=DEV)
    shape = _lib.KdaShape(n, w.q.shape[0], w.q.shape[1], 128, 128, _lib.KDA_BF16)
    st = L.kda_prefill_split_static(ctypes.byref(shape), _p(w.q), _p(w.k), _p(w.v), _p(w.log_alpha), _p(w.beta),
                                    _p(w.initial_state), _p(cu), _p(out), _p(fin),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, out, fin


def test_static_scratch_matches_the_workspace_path_twice_in_a_row(L):
    cases = [([300, 150], 4, 201), ([64, 1, 129, 700], 2, 202)]
    for lens, H, seed in cases:                # two calls in a row on the shared array
        cu_h = workloads.cu_from_lengths(lens)
        w = workloads.make_inputs(cu_h[-1], H, 128, 128, seed=seed, cu_seqlens=cu_h, state_std=0.05).to(DEV)
        cu = w.cu_seqlens.to(DEV)
        st, out, fin = static_prefill(L, w, cu)
        assert st == 0, _lib.status_string(st)
        ref_out, ref_fin = kda.kda_prefill_split(w.q, w.k, w.v, w.log_alpha, w.beta, w.initial_state, cu,
                                                 final_state=True)
        torch.cuda.synchronize()
        assert rel_l2(np64(out), np64(ref_out)) <= TOL and rel_l2(np64(fin), np64(ref_fin)) <= TOL
        ro, rf = oracle_prefill(w)
        assert rel_l2(np64(out), ro) <= TOL and rel_l2(np64(fin), rf) <= TOL
    assert kda.kda_device_status() == 0


def test_static_scratch_rejects_shapes_beyond_its_size(L):
    # one 131072-token sequence with 32 heads needs about 6.4 GB of scratch: refused on the
    # host with KDA_ERR_UNSUPPORTED, before any GPU work (the pointers are never read)
    shape = _lib.KdaShape(1, 131072, 32, 128, 128, _lib.KDA_BF16)
    fake = ctypes.c_void_p(0x10000)
    st = L.kda_prefill_split_static(ctypes.byref(shape), fake, fake, fake, fake, fake, None, None, fake, None, None)
    assert st == _lib.KDA_ERR_UNSUPPORTED
