"""GPU parity of the split prefill (kda_prefill_split: a chunk-local kernel over every
chunk of every head, then a state-chain kernel per (sequence, head)) against the fp64
oracle, and its agreement with the fused prefill (kda_prefill) on the same inputs.

Tolerance: relative L2 <= 5e-3 for bf16 inputs, over the whole tensor, separately
for out and the final state.  Full-size workloads are checked on sampled heads.
"""
import numpy as np
import pytest
import torch

import linear_attention_06_gb300 as kda
from linear_attention_06_gb300 import workloads
from tests.gpu_helpers import TOL, gpu_prefill, np64, oracle_prefill, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_06_gb300 import build
    build.build()


def split_prefill(w, **kw):
    out, fin = kda.kda_prefill_split(w.q, w.k, w.v, w.log_alpha, w.beta, w.initial_state,
                                     w.cu_seqlens.to(w.q.device), final_state=True, **kw)
    torch.cuda.synchronize()
    return out, fin


def check(w, heads=None, tol=5e-3):
    out, fin = split_prefill(w)
    ro, rf = oracle_prefill(w, heads)
    sel = slice(None) if heads is None else list(heads)
    e_out, e_fin = rel_l2(np64(out[:, sel]), ro), rel_l2(np64(fin[:, sel]), rf)
    assert e_out <= tol and e_fin <= tol, f"{w.name}: out {e_out:.3e} state {e_fin:.3e}"
    return out, fin


@pytest.mark.parametrize("lens", [[1], [15], [63], [64], [65], [300], [1, 64, 65, 130],
                                  [5, 0, 200, 16, 129], [0, 0, 70]])
def test_split_small_ragged(lens):
    cu = workloads.cu_from_lengths(lens)
    w = workloads.make_inputs(cu[-1], 3, 128, 128, dtype=torch.bfloat16, seed=100 + sum(lens),
                              cu_seqlens=cu, state_std=0.05).to(DEV)
    check(w)


def test_split_agrees_with_fused_prefill():
    cu = [0, 200, 777, 1000]
    w = workloads.make_inputs(cu[-1], 4, 128, 128, seed=101, cu_seqlens=cu, state_std=0.05).to(DEV)
    o_s, f_s = split_prefill(w)
    o_f, f_f = gpu_prefill(w)
    # the same bf16 operands and fp32 accumulation; only the order of a few fp32 additions differs
    assert rel_l2(np64(o_s), np64(o_f)) < 1e-3 and rel_l2(np64(f_s), np64(f_f)) < 1e-4


def test_split_many_short_sequences():
    rng = np.random.default_rng(102)
    lens = [int(v) for v in rng.integers(0, 150, size=200)]
    cu = workloads.cu_from_lengths(lens)
    w = workloads.make_inputs(cu[-1], 2, 128, 128, seed=102, cu_seqlens=cu, state_std=0.05).to(DEV)
    check(w)


def test_split_dense_batch_and_zero_state():
    w = workloads.make_inputs(3 * 256, 2, 128, 128, seed=103, num_seqs=3).to(DEV)
    out, fin = kda.kda_prefill_split(w.q, w.k, w.v, w.log_alpha, w.beta, None, None, final_state=True,
                                     num_seqs=3)
    torch.cuda.synchronize()
    ro, rf = oracle_prefill(w)
    assert rel_l2(np64(out), ro) < 5e-3 and rel_l2(np64(fin), rf) < 5e-3


@pytest.mark.parametrize("mode", ["strong", "minus_inf", "mixed", "beta_one_two"])
def test_split_extreme_decay_and_beta(mode):
    cu = [0, 64, 64 + 150, 400]
    w = workloads.make_inputs(cu[-1], 2, 128, 128, dtype=torch.bfloat16, seed=104,
                              cu_seqlens=cu, state_std=0.05).to(DEV)
    if mode == "strong":
        w.log_alpha.mul_(40.0)                    # every chunk runs token by token
    elif mode == "minus_inf":
        w.log_alpha[10::37, :, ::3] = float("-inf")
    elif mode == "mixed":
        w.log_alpha[:, :, :64] = -30.0
    else:
        w.beta[::2] = 1.0
        w.beta[1::4] = 2.0
    check(w)


def test_split_token_chunk_between_factored_chunks():
    T = 8 * 64
    w = workloads.make_inputs(T, 2, 128, 128, seed=105, cu_seqlens=[0, T], state_std=0.05).to(DEV)
    w.log_alpha[64 * 3 + 17, :, ::5] = float("-inf")
    check(w)


def test_split_workspace_is_reusable_and_results_deterministic():
    cu = [0, 300, 450]
    w = workloads.make_inputs(cu[-1], 2, 128, 128, seed=106, cu_seqlens=cu, state_std=0.05).to(DEV)
    need = kda.kda_prefill_split_workspace_size(cu[-1], 2, 2)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device=DEV)    # stale contents
    o1, f1 = split_prefill(w, workspace=ws)
    o2, f2 = split_prefill(w, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    assert kda.kda_device_status() == 0


def test_split_long_prefill_sampled_heads_and_resume():
    w = workloads.long_prefill(device=DEV)
    T = w.total_tokens
    m = T // 2
    out, fin = check(w, heads=[0, 31])
    o1, s1 = kda.kda_prefill_split(w.q[:m], w.k[:m], w.v[:m], w.log_alpha[:m], w.beta[:m], None, None,
                                   final_state=True)
    o2, s2 = kda.kda_prefill_split(w.q[m:], w.k[m:], w.v[m:], w.log_alpha[m:], w.beta[m:], s1, None,
                                   final_state=True)
    torch.cuda.synchronize()
    # the split lands on a chunk boundary: the same records and the same chain
    assert torch.equal(torch.cat([o1, o2]), out) and torch.equal(s2, fin)


@pytest.mark.parametrize("T", [16384, 20000, 24577])
def test_split_segmented_single_sequence(T):
    # one sequence of at least 16384 tokens runs in 8192-token segments (chunk records of the
    # next segment built while the chains run), the fp32 state carried between segments: a
    # ragged last segment, an initial state, and agreement with the fused prefill and the oracle
    w = workloads.make_inputs(T, 4, 128, 128, seed=108 + T % 97, cu_seqlens=[0, T], state_std=0.05).to(DEV)
    out, fin = check(w, heads=[1])
    o_f, f_f = gpu_prefill(w)
    assert rel_l2(np64(out), np64(o_f)) < 1e-3 and rel_l2(np64(fin), np64(f_f)) < 1e-4
    assert kda.kda_device_status() == 0


def test_split_segmented_results_do_not_depend_on_the_workspace_contents():
    T = 17000
    w = workloads.make_inputs(T, 2, 128, 128, seed=109, cu_seqlens=[0, T], state_std=0.05).to(DEV)
    need = kda.kda_prefill_split_workspace_size(T, 1, 2)
    ws = torch.full((need,), 0x5A, dtype=torch.uint8, device=DEV)
    o1, f1 = split_prefill(w, workspace=ws)
    ws.fill_(0xC3)
    o2, f2 = split_prefill(w, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_split_varlen_full_size_sampled_heads():
    w = workloads.varlen_prefill(device=DEV)
    check(w, heads=[0, 31])


def test_split_unsupported_shape_runs_the_plain_prefill():
    cu = [0, 77, 200]
    w = workloads.make_inputs(cu[-1], 2, 64, 64, dtype=torch.float32, seed=107, cu_seqlens=cu,
                              state_std=0.05).to(DEV)
    out, fin = split_prefill(w)                   # no workspace needed for these shapes
    ro, rf = oracle_prefill(w)
    assert rel_l2(np64(out), ro) < TOL[torch.float32] and rel_l2(np64(fin), rf) < TOL[torch.float32]
