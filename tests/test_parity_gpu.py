"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (relative L2 over the whole tensor, separately for out and for the
final state): 1e-4 for fp32 inputs, 5e-3 for bf16 inputs.  Full-size
workloads are checked on sampled heads: every (sequence, head) pair is an
independent recurrence, so the oracle computes the sampled heads exactly.
"""
import numpy as np
import pytest
import torch

import linear_attention_06_gb300 as kda
from linear_attention_06_gb300 import workloads
from tests.gpu_helpers import (TOL, compare_prefill, gpu_prefill, np64, oracle_prefill,
                               rel_l2)
from oracle import kda_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_06_gb300 import build
    build.build()


# ---- the tiny fp32 workload (B=1, H=2, T=256, d=64) ---------------------------------
def test_tiny_fp32_workload():
    w = workloads.tiny_fp32().to(DEV)
    e_out, e_fin = compare_prefill(w)
    assert e_out < 1e-4 and e_fin < 1e-4


# ---- small shapes: ragged tails, short sequences, both head sizes, both dtypes ------
@pytest.mark.parametrize("lens", [[1], [15], [17], [63], [64], [65], [100], [300],
                                  [1, 64, 65, 130], [5, 0, 200, 16, 129]])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_small_ragged_d128(lens, dtype):
    cu = workloads.cu_from_lengths(lens)
    w = workloads.make_inputs(cu[-1], 3, 128, 128, dtype=dtype, seed=sum(lens),
                              cu_seqlens=cu, state_std=0.05).to(DEV)
    compare_prefill(w)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_small_head_sizes(dk, dv, dtype):
    cu = [0, 77, 77 + 190]
    w = workloads.make_inputs(cu[-1], 2, dk, dv, dtype=dtype, seed=dk + dv,
                              cu_seqlens=cu, state_std=0.05).to(DEV)
    compare_prefill(w)


def test_many_short_sequences_span_many_waves():
    # 400 sequences x 4 heads = 1600 blocks (about ten waves of one block per SM), every
    # chunk a ragged last chunk, lengths 0..40 with empty sequences among them
    rng = np.random.default_rng(400)
    lens = [int(v) for v in rng.integers(0, 41, size=400)]
    cu = workloads.cu_from_lengths(lens)
    w = workloads.make_inputs(cu[-1], 4, 128, 128, seed=400, cu_seqlens=cu, state_std=0.05).to(DEV)
    compare_prefill(w)


def test_dense_batch_without_cu_seqlens():
    w = workloads.make_inputs(4 * 150, 2, 128, 128, seed=5, num_seqs=4).to(DEV)
    out, fin = kda.kda_prefill(w.q, w.k, w.v, w.log_alpha, w.beta, None, None,
                               final_state=True, num_seqs=4)
    torch.cuda.synchronize()
    ro, rf = oracle_prefill(w)
    assert rel_l2(np64(out), ro) < 5e-3 and rel_l2(np64(fin), rf) < 5e-3


def test_host_cu_seqlens_is_validated_and_copied():
    cu = [0, 33, 140]
    w = workloads.make_inputs(cu[-1], 2, 128, 128, seed=6, cu_seqlens=cu).to(DEV)
    compare_prefill(w, cu_on_device=False)
    with pytest.raises(kda.KdaError):
        kda.kda_prefill(w.q, w.k, w.v, w.log_alpha, w.beta, None, [0, 50, 40],
                        final_state=True)


# ---- decay and write-strength edge cases --------------------------------------------
def test_no_write_no_decay_keeps_state():
    cu = [0, 90, 200]
    w = workloads.make_inputs(cu[-1], 2, 128, 128, seed=7, cu_seqlens=cu, state_std=0.05).to(DEV)
    w.beta.zero_()
    w.log_alpha.zero_()
    out, fin = gpu_prefill(w)
    assert torch.equal(fin, w.initial_state)


@pytest.mark.parametrize("mode", ["strong", "minus_inf", "mixed", "beta_one_two"])
def test_extreme_decay_and_beta(mode):
    cu = [0, 64, 64 + 150]
    w = workloads.make_inputs(cu[-1], 2, 128, 128, dtype=torch.bfloat16, seed=8,
                              cu_seqlens=cu, state_std=0.05).to(DEV)
    if mode == "strong":
        w.log_alpha.mul_(40.0)                    # ~ -2 per token: e^-128 over a chunk
    elif mode == "minus_inf":
        w.log_alpha[10::37, :, ::3] = float("-inf")
    elif mode == "mixed":
        w.log_alpha[:, :, :64] = -30.0            # half the channels forget at once
    else:
        w.beta[::2] = 1.0
        w.beta[1::4] = 2.0
    compare_prefill(w)


@pytest.mark.parametrize("token_chunk", [2, 3, 5])
def test_token_chunk_between_tensor_core_chunks(token_chunk):
    # One chunk whose decay leaves the tensor-core range (a -inf gate) in the middle of
    # a run of ordinary chunks: the slots it shares with later chunks must be handed
    # back in order.
    T = 8 * 64
    w = workloads.make_inputs(T, 2, 128, 128, dtype=torch.bfloat16, seed=31, cu_seqlens=[0, T],
                              state_std=0.05).to(DEV)
    w.log_alpha[64 * token_chunk + 17, :, ::5] = float("-inf")
    compare_prefill(w)


# ---- full-size workloads, sampled heads ---------------------------------------------
def test_prefill_bf16_full_size_sampled_heads():
    w = workloads.prefill_bf16(device=DEV)
    compare_prefill(w, heads=[0, 13, 31])


def test_long_prefill_resume_equals_full_run():
    w = workloads.long_prefill(device=DEV)
    T = w.total_tokens
    m = T // 2
    full_out, full_fin = gpu_prefill(w)
    o1, s1 = kda.kda_prefill(w.q[:m], w.k[:m], w.v[:m], w.log_alpha[:m], w.beta[:m],
                             None, None, final_state=True)
    o2, s2 = kda.kda_prefill(w.q[m:], w.k[m:], w.v[m:], w.log_alpha[m:], w.beta[m:],
                             s1, None, final_state=True)
    torch.cuda.synchronize()
    # the split lands on a chunk boundary and the kernels are deterministic
    assert torch.equal(torch.cat([o1, o2]), full_out)
    assert torch.equal(s2, full_fin)
    heads = [0, 31]
    ro, rf = oracle_prefill(w, heads)
    assert rel_l2(np64(full_out[:, heads]), ro) < 5e-3
    assert rel_l2(np64(full_fin[:, heads]), rf) < 5e-3


def test_varlen_full_size_sampled_heads():
    w = workloads.varlen_prefill(device=DEV)
    compare_prefill(w, heads=[0, 31])


def test_decode_full_size():
    w = workloads.decode_inputs(device=DEV)
    S = w.initial_state.clone()
    out = kda.kda_decode_step(w.q, w.k, w.v, w.log_alpha, w.beta, S)
    torch.cuda.synchronize()
    ro, rS = kda_oracle.decode_step(np64(w.q), np64(w.k), np64(w.v), np64(w.log_alpha),
                                    np64(w.beta), np64(w.initial_state))
    assert rel_l2(np64(out), ro) < 5e-3
    assert rel_l2(np64(S), rS) < 5e-3


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_small(dk, dv, dtype):
    n = 37
    w = workloads.make_inputs(n, 3, dk, dv, dtype=dtype, seed=dk * 3 + dv,
                              cu_seqlens=list(range(n + 1)), state_std=0.05).to(DEV)
    S = w.initial_state.clone()
    out = kda.kda_decode_step(w.q, w.k, w.v, w.log_alpha, w.beta, S)
    torch.cuda.synchronize()
    ro, rS = kda_oracle.decode_step(np64(w.q), np64(w.k), np64(w.v), np64(w.log_alpha),
                                    np64(w.beta), np64(w.initial_state))
    assert rel_l2(np64(out), ro) < TOL[dtype] and rel_l2(np64(S), rS) < TOL[dtype]


# ---- internal invariants ------------------------------------------------------------
def test_decode_equals_one_token_prefill():
    n = 64
    w = workloads.make_inputs(n, 4, 128, 128, seed=21, cu_seqlens=list(range(n + 1)),
                              state_std=0.05).to(DEV)
    S = w.initial_state.clone()
    o_d = kda.kda_decode_step(w.q, w.k, w.v, w.log_alpha, w.beta, S)
    o_p, S_p = gpu_prefill(w)
    assert rel_l2(np64(o_d), np64(o_p)) < 5e-3 and rel_l2(np64(S), np64(S_p)) < 5e-3


def test_varlen_equals_separate_runs():
    lens = [70, 1, 300, 64]
    cu = workloads.cu_from_lengths(lens)
    w = workloads.make_inputs(cu[-1], 2, 128, 128, seed=22, cu_seqlens=cu, state_std=0.05).to(DEV)
    out, fin = gpu_prefill(w)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        o_n, f_n = kda.kda_prefill(w.q[s:e], w.k[s:e], w.v[s:e], w.log_alpha[s:e], w.beta[s:e],
                                   w.initial_state[n:n + 1].contiguous(), None, final_state=True)
        torch.cuda.synchronize()
        assert torch.equal(o_n, out[s:e]) and torch.equal(f_n[0], fin[n])


def test_final_state_may_alias_initial_state():
    cu = [0, 100, 250]
    w = workloads.make_inputs(cu[-1], 2, 128, 128, seed=23, cu_seqlens=cu, state_std=0.05).to(DEV)
    _, ref = gpu_prefill(w)
    S = w.initial_state.clone()
    kda.kda_prefill(w.q, w.k, w.v, w.log_alpha, w.beta, S, w.cu_seqlens.to(DEV), final_state=S)
    torch.cuda.synchronize()
    assert torch.equal(S, ref)


def test_recurrent_and_chunk_paths_agree(monkeypatch):
    cu = [0, 200, 333]
    w = workloads.make_inputs(cu[-1], 2, 128, 128, seed=24, cu_seqlens=cu, state_std=0.05).to(DEV)
    o_a, f_a = gpu_prefill(w)
    monkeypatch.setenv("KDA_PREFILL_IMPL", "recurrent")
    o_b, f_b = gpu_prefill(w)
    assert rel_l2(np64(o_a), np64(o_b)) < 5e-3 and rel_l2(np64(f_a), np64(f_b)) < 5e-3


def test_timeout_path_sets_and_clears_the_status_word():
    # a bounded wait that nothing completes (1 ms): no fault, the context stays usable
    assert kda.kda_device_status() == 0
    kda.kda_selftest_timeout(1_000_000)
    assert kda.kda_device_status() == 4                    # KDA_ERR_TIMEOUT
    assert kda.kda_device_status() == 0                    # read and cleared
    w = workloads.make_inputs(64, 2, 128, 128, seed=77).to(DEV)
    compare_prefill(w)                                     # the library still runs
    assert kda.kda_device_status() == 0


def test_device_status_is_clean():
    assert kda.kda_device_status() == 0


# ---- multi-token decode (T tokens per sequence through the decode path) -------------
# At dk = dv = 128 a bf16 step of 2..16 tokens takes the chunk form (tensor cores, T <= 8 and
# T <= 16 instances), or its fp32 token loop when the decay over the step passes e^-60 in some
# channel; fp32 inputs and other head sizes keep the token loop of the one-token kernel.
@pytest.mark.parametrize("T", [2, 5, 8, 9, 16])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_multi_token_matches_oracle(T, dtype):
    n = 24
    cu = [T * i for i in range(n + 1)]
    w = workloads.make_inputs(n * T, 4, 128, 128, dtype=dtype, seed=30 + T, cu_seqlens=cu,
                              state_std=0.05).to(DEV)
    S = w.initial_state.clone()
    out = kda.kda_decode_step(w.q, w.k, w.v, w.log_alpha, w.beta, S)
    torch.cuda.synchronize()
    ro, rf = oracle_prefill(w)
    assert rel_l2(np64(out), ro) < TOL[dtype] and rel_l2(np64(S), rf) < TOL[dtype]


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 64), (64, 64)])
def test_decode_multi_token_other_head_sizes(dk, dv):
    n, T = 12, 6
    cu = [T * i for i in range(n + 1)]
    w = workloads.make_inputs(n * T, 3, dk, dv, seed=31, cu_seqlens=cu, state_std=0.05).to(DEV)
    S = w.initial_state.clone()
    out = kda.kda_decode_step(w.q, w.k, w.v, w.log_alpha, w.beta, S)
    torch.cuda.synchronize()
    ro, rf = oracle_prefill(w)
    assert rel_l2(np64(out), ro) < TOL[torch.bfloat16] and rel_l2(np64(S), rf) < TOL[torch.bfloat16]


def test_decode_multi_token_strong_decay_mixed_with_chunk_form():
    # sequences 0, 5 and 11 decay past e^-60 within the step (some channels reach -inf): their
    # (sequence, head) blocks run token by token, the others in the chunk form, in one launch
    n, T, H = 12, 16, 4
    cu = [T * i for i in range(n + 1)]
    w = workloads.make_inputs(n * T, H, 128, 128, seed=32, cu_seqlens=cu, state_std=0.05)
    for seq in (0, 5, 11):
        w.log_alpha[seq * T:(seq + 1) * T] *= 100.0
    w.log_alpha[5 * T + 3, 1, :7] = -float("inf")            # a full reset of a few channels
    d = w.to(DEV)
    S = d.initial_state.clone()
    out = kda.kda_decode_step(d.q, d.k, d.v, d.log_alpha, d.beta, S)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(S).all()
    ro, rf = oracle_prefill(w)
    assert rel_l2(np64(out), ro) < TOL[torch.bfloat16] and rel_l2(np64(S), rf) < TOL[torch.bfloat16]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_multi_token_agrees_with_repeated_single_steps(dtype):
    # the chunk form (bf16) is an exact rewrite of T one-token steps, not the same sequence of
    # roundings: it agrees within the tolerance of the dtype; fp32 runs the one-token kernel's
    # loop T times and gives the same bits
    n, T, H = 16, 7, 4
    cu = [T * i for i in range(n + 1)]
    w = workloads.make_inputs(n * T, H, 128, 128, dtype=dtype, seed=40, cu_seqlens=cu, state_std=0.05).to(DEV)
    S_multi = w.initial_state.clone()
    out_multi = kda.kda_decode_step(w.q, w.k, w.v, w.log_alpha, w.beta, S_multi)
    S_step = w.initial_state.clone()
    rows = torch.arange(n, device=DEV) * T
    outs = torch.empty_like(out_multi)
    for t in range(T):
        r = rows + t
        outs[r] = kda.kda_decode_step(w.q[r].contiguous(), w.k[r].contiguous(), w.v[r].contiguous(),
                                      w.log_alpha[r].contiguous(), w.beta[r].contiguous(), S_step)
    torch.cuda.synchronize()
    assert rel_l2(np64(out_multi), np64(outs)) < TOL[dtype]
    assert rel_l2(np64(S_multi), np64(S_step)) < TOL[dtype]
    if dtype == torch.float32:
        assert torch.equal(out_multi, outs) and torch.equal(S_multi, S_step)


def test_decode_two_tokens_equals_two_single_steps_bitwise():
    # a two-token step runs the one-token kernel's loop twice on the state in registers (the
    # chunk form starts at three tokens): the same arithmetic in the same order as two calls
    # of the one-token step, so out and the state are equal bit for bit
    n, T, H = 16, 2, 4
    cu = [T * i for i in range(n + 1)]
    w = workloads.make_inputs(n * T, H, 128, 128, dtype=torch.bfloat16, seed=41, cu_seqlens=cu,
                              state_std=0.05).to(DEV)
    S_two = w.initial_state.clone()
    out_two = kda.kda_decode_step(w.q, w.k, w.v, w.log_alpha, w.beta, S_two)
    S_one = w.initial_state.clone()
    rows = torch.arange(n, device=DEV) * T
    outs = torch.empty_like(out_two)
    for t in range(T):
        r = rows + t
        outs[r] = kda.kda_decode_step(w.q[r].contiguous(), w.k[r].contiguous(), w.v[r].contiguous(),
                                      w.log_alpha[r].contiguous(), w.beta[r].contiguous(), S_one)
    torch.cuda.synchronize()
    assert torch.equal(out_two, outs) and torch.equal(S_two, S_one)


@pytest.mark.parametrize("T", [4, 16])
def test_decode_multi_token_full_size_sampled_sequences(T):
    # the bench's multi-token step (256 sequences x 32 heads, one launch of the chunk form on
    # every SM), checked on sampled (sequence, head) pairs against the oracle
    n, H = 256, 32
    cu = [T * i for i in range(n + 1)]
    w = workloads.make_inputs(n * T, H, 128, 128, seed=13 + T, cu_seqlens=cu, state_std=0.05)
    d = w.to(DEV)
    S = d.initial_state.clone()
    out = kda.kda_decode_step(d.q, d.k, d.v, d.log_alpha, d.beta, S)
    torch.cuda.synchronize()
    seqs, heads = [0, 77, 128, 255], [0, 13, 31]
    rows = np.concatenate([np.arange(T * i, T * (i + 1)) for i in seqs])
    pick = lambda t: np64(t[rows][:, heads])          # noqa: E731
    ro, rf = kda_oracle.prefill(pick(w.q), pick(w.k), pick(w.v), pick(w.log_alpha), pick(w.beta),
                                np64(w.initial_state[seqs][:, heads]), cu_seqlens=[T * i for i in range(len(seqs) + 1)])
    assert rel_l2(np64(out)[rows][:, heads], ro) < TOL[torch.bfloat16]
    assert rel_l2(np64(S)[seqs][:, heads], rf) < TOL[torch.bfloat16]


def test_decode_multi_token_zero_beta_is_pure_decay():
    # beta = 0: no erase and no write, so the state is only decayed: S = Diag(e^G) S0 exactly
    # up to the fp32 product of the decay factors, and o_t = (e^{g_t} o q_t)^T S0
    n, T, H = 6, 10, 2
    cu = [T * i for i in range(n + 1)]
    w = workloads.make_inputs(n * T, H, 128, 128, seed=41, cu_seqlens=cu, state_std=0.05)
    w.beta.zero_()
    d = w.to(DEV)
    S = d.initial_state.clone()
    out = kda.kda_decode_step(d.q, d.k, d.v, d.log_alpha, d.beta, S)
    torch.cuda.synchronize()
    la = np64(w.log_alpha).reshape(n, T, H, 128)
    G = la.sum(axis=1)                                        # [n, H, dk]
    S_ref = np.exp(G)[..., None] * np64(w.initial_state)
    assert rel_l2(np64(S), S_ref) < 1e-5
    g = np.cumsum(la, axis=1)
    o_ref = np.einsum("nthk,nhkv->nthv", np.exp(g) * np64(w.q).reshape(n, T, H, 128), np64(w.initial_state))
    assert rel_l2(np64(out).reshape(n, T, H, 128), o_ref) < TOL[torch.bfloat16]


# ---- checkpoint emission during prefill ---------------------------------------------
def oracle_checkpoints(w, ck, heads=None):
    """fp64 oracle state after each checkpoint position: each sequence is run as a chain of
    oracle prefills over the segments between its positions, every segment starting from the
    previous one's final state (the resume property the oracle is pinned to)."""
    sel = slice(None) if heads is None else list(heads)
    cu = [int(x) for x in w.cu_seqlens]
    pick = lambda t, s, e: np64(t[s:e, sel])          # noqa: E731
    states = []
    for n, positions in enumerate(ck):
        S = None if w.initial_state is None else np64(w.initial_state[n:n + 1, sel])
        done = 0
        for p in positions:
            s, e = cu[n] + done, cu[n] + p
            _, S = kda_oracle.prefill(pick(w.q, s, e), pick(w.k, s, e), pick(w.v, s, e),
                                      pick(w.log_alpha, s, e), pick(w.beta, s, e), S,
                                      cu_seqlens=[0, e - s])
            states.append(S[0])
            done = p
    return np.stack(states)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_checkpoints_match_oracle_and_prefix_runs(dtype):
    lens = [200, 64, 300, 30]
    cu = workloads.cu_from_lengths(lens)
    ck = [[64, 128, 200], [64], [192, 256, 300], [30]]
    w = workloads.make_inputs(cu[-1], 3, 128, 128, dtype=dtype, seed=50, cu_seqlens=cu,
                              state_std=0.05).to(DEV)
    out, fin, cks = kda.kda_prefill_checkpointed(w.q, w.k, w.v, w.log_alpha, w.beta, ck,
                                                 w.initial_state, cu, final_state=True)
    torch.cuda.synchronize()
    # every checkpoint against the fp64 oracle's state at that position
    ref = oracle_checkpoints(w, ck)
    assert rel_l2(np64(cks), ref) <= TOL[dtype]
    for c in range(ref.shape[0]):                      # and each one on its own
        assert rel_l2(np64(cks[c]), ref[c]) <= TOL[dtype], c
    ro, rf = oracle_prefill(w)
    assert rel_l2(np64(out), ro) <= TOL[dtype] and rel_l2(np64(fin), rf) <= TOL[dtype]
    # the same call without checkpoints gives the same out and final state, bit for bit
    ref_out, ref_fin = gpu_prefill(w)
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    # and a checkpoint equals the final state of a prefill over the same prefix
    c = 0
    for n, positions in enumerate(ck):
        for p in positions:
            s, e = cu[n], cu[n] + p
            _, f = kda.kda_prefill(w.q[s:e], w.k[s:e], w.v[s:e], w.log_alpha[s:e], w.beta[s:e],
                                   w.initial_state[n:n + 1].contiguous(), None, final_state=True)
            torch.cuda.synchronize()
            assert torch.equal(cks[c], f[0]), (n, p)
            c += 1


def test_checkpoints_full_size_sampled_heads():
    # the benchmark prefill (4 x 8192 tokens, 32 heads) saving every sequence's state each
    # 1024 tokens; sampled heads against the oracle's chained segments
    w = workloads.prefill_bf16(device=DEV)
    B, T = 4, 8192
    ck = [list(range(1024, T + 1, 1024)) for _ in range(B)]
    out, fin, cks = kda.kda_prefill_checkpointed(w.q, w.k, w.v, w.log_alpha, w.beta, ck, None,
                                                 w.cu_seqlens, final_state=True)
    torch.cuda.synchronize()
    heads = [0, 31]
    ref = oracle_checkpoints(w, ck, heads)
    got = np64(cks[:, heads])
    assert rel_l2(got, ref) <= 5e-3
    for c in range(ref.shape[0]):
        assert rel_l2(got[c], ref[c]) <= 5e-3, c
    ro, rf = oracle_prefill(w, heads)
    assert rel_l2(np64(out[:, heads]), ro) <= 5e-3 and rel_l2(np64(fin[:, heads]), rf) <= 5e-3


@pytest.mark.parametrize("impl", ["tensor_core", "recurrent"])
def test_checkpoint_nonpositive_positions_do_not_drop_later_ones(impl, monkeypatch):
    # Straight through the C ABI (no host validation): a position <= 0 is skipped like any
    # other bad position, and the valid checkpoints after it are still written.
    import ctypes
    from linear_attention_06_gb300 import _lib
    if impl == "recurrent":
        monkeypatch.setenv("KDA_PREFILL_IMPL", "recurrent")
    lens = [256, 192]
    cu = workloads.cu_from_lengths(lens)
    w = workloads.make_inputs(cu[-1], 2, 128, 128, seed=52, cu_seqlens=cu, state_std=0.05).to(DEV)
    ck = [[0, 64, 192], [-5, 128]]
    d_cu = torch.tensor(cu, dtype=torch.int32, device=DEV)
    ck_cu = torch.tensor([0, 3, 5], dtype=torch.int32, device=DEV)
    ck_pos = torch.tensor([p for ps in ck for p in ps], dtype=torch.int32, device=DEV)
    cks = torch.full((5, 2, 128, 128), float("nan"), device=DEV)
    out = torch.empty_like(w.v)
    shape = _lib.KdaShape(2, cu[-1], 2, 128, 128, _lib.KDA_BF16)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = _lib.lib().kda_prefill_checkpointed(ctypes.byref(shape), p(w.q), p(w.k), p(w.v), p(w.log_alpha),
                                             p(w.beta), p(w.initial_state), p(d_cu), p(out), None, p(ck_cu),
                                             p(ck_pos), p(cks), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 0
    assert torch.isnan(cks[0]).all() and torch.isnan(cks[3]).all()      # the bad positions
    ref = oracle_checkpoints(w, [[64, 192], [128]])
    for got, r in zip((cks[1], cks[2], cks[4]), ref):
        assert rel_l2(np64(got), r) <= 5e-3


def test_checkpoint_positions_off_chunk_ends_are_not_written():
    import ctypes
    from linear_attention_06_gb300 import _lib
    lens = [256]
    w = workloads.make_inputs(256, 2, 128, 128, seed=51, cu_seqlens=[0, 256]).to(DEV)
    with pytest.raises(kda.KdaError):           # the host validator rejects 100
        kda.kda_prefill_checkpointed(w.q, w.k, w.v, w.log_alpha, w.beta, [[64, 100]], None, [0, 256])
    # straight through the C ABI, the device skips the bad position and writes the good one
    d_cu = torch.tensor([0, 256], dtype=torch.int32, device=DEV)
    ck_cu = torch.tensor([0, 2], dtype=torch.int32, device=DEV)
    ck_pos = torch.tensor([100, 128], dtype=torch.int32, device=DEV)
    cks = torch.full((2, 2, 128, 128), float("nan"), device=DEV)
    out = torch.empty_like(w.v)
    shape = _lib.KdaShape(1, 256, 2, 128, 128, _lib.KDA_BF16)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = _lib.lib().kda_prefill_checkpointed(ctypes.byref(shape), p(w.q), p(w.k), p(w.v), p(w.log_alpha),
                                             p(w.beta), None, p(d_cu), p(out), None, p(ck_cu), p(ck_pos),
                                             p(cks), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 0
    assert torch.isnan(cks[0]).all()
    _, f = kda.kda_prefill(w.q[:128], w.k[:128], w.v[:128], w.log_alpha[:128], w.beta[:128], None, None,
                           final_state=True)
    torch.cuda.synchronize()
    assert torch.equal(cks[1], f[0])
