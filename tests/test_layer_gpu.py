"""GPU parity for the layer steps around the recurrence: the front end
(kda_frontend) against the fp64 layer oracle on the same seeded raw inputs.

Tolerances (relative L2 over each output tensor): bf16 outputs 5e-3 (one bf16
rounding is about 2e-3); fp32 outputs 1e-5 (the kernel's exp/log are fp32
approximations with a few ulp of error).
"""
import numpy as np
import pytest
import torch

import linear_attention_06_gb300 as kda
from linear_attention_06_gb300 import workloads
from oracle import kda_layer_oracle as lo
from tests.gpu_helpers import np64, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_06_gb300 import build
    build.build()


def run_frontend(x, heads=None, eps=1e-6, num_seqs=None):
    d = x.to(DEV)
    cu = None if num_seqs is not None else d.cu_seqlens
    got = kda.kda_frontend(d.q_raw, d.k_raw, d.v_raw, d.a_raw, d.b_raw, d.conv_q, d.conv_k, d.conv_v,
                           cu_seqlens=cu, num_seqs=num_seqs, eps=eps)
    torch.cuda.synchronize()
    sel = slice(None) if heads is None else list(heads)
    ref = lo.frontend(np64(x.q_raw[:, sel]), np64(x.k_raw[:, sel]), np64(x.v_raw[:, sel]),
                      np64(x.conv_q[sel]), np64(x.conv_k[sel]), np64(x.conv_v[sel]),
                      np64(x.a_raw[:, sel]), np64(x.b_raw[:, sel]),
                      cu_seqlens=x.cu_seqlens.numpy(), eps=eps)
    return [np64(g[:, sel]) for g in got], ref


def check(got, ref, dtype):
    tol = 5e-3 if dtype == torch.bfloat16 else 1e-5
    names = ["q", "k", "v", "log_alpha", "beta"]
    for name, g, r in zip(names, got, ref):
        t = 1e-5 if name == "log_alpha" else tol
        e = rel_l2(g, r)
        assert e <= t, f"{name}: rel L2 {e:.3e} > {t}"


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_frontend_varlen_widths(W, dtype):
    cu = [0, 1, 77, 77, 200, 333]          # a one-token and an empty sequence, ragged runs
    x = workloads.make_layer_inputs(cu[-1], 2, 128, 128, W=W, dtype=dtype, seed=40 + W, cu_seqlens=cu)
    got, ref = run_frontend(x)
    check(got, ref, dtype)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
def test_frontend_head_sizes(dk, dv):
    x = workloads.make_layer_inputs(150, 3, dk, dv, W=4, dtype=torch.bfloat16, seed=50, cu_seqlens=[0, 70, 150])
    got, ref = run_frontend(x)
    check(got, ref, torch.bfloat16)


def test_frontend_dense_split_and_eps():
    x = workloads.make_layer_inputs(4 * 96, 2, 128, 128, W=4, dtype=torch.float32, seed=51, num_seqs=4)
    got, ref = run_frontend(x, num_seqs=4, eps=0.5)
    check(got, ref, torch.float32)


def test_frontend_full_size_sampled_heads():
    # the benchmark shape: B=4 sequences of 8192 tokens, H=32, d=128, bf16
    # drawn on the device (the host draw of 0.8G values is slow); both sides read these tensors
    x = workloads.make_layer_inputs(4 * 8192, 32, 128, 128, W=4, dtype=torch.bfloat16, seed=1, num_seqs=4,
                                    device=DEV)
    got, ref = run_frontend(x, heads=[0, 17, 31], num_seqs=4)
    check(got, ref, torch.bfloat16)


def test_frontend_output_feeds_prefill():
    # the front end's outputs are valid kda_prefill inputs: unit-norm q and k, log_alpha <= 0
    x = workloads.make_layer_inputs(512, 4, 128, 128, W=4, dtype=torch.bfloat16, seed=52, num_seqs=2).to(DEV)
    q, k, v, la, beta = kda.kda_frontend(x.q_raw, x.k_raw, x.v_raw, x.a_raw, x.b_raw, x.conv_q, x.conv_k,
                                         x.conv_v, num_seqs=2)
    out, fin = kda.kda_prefill(q, k, v, la, beta, None, None, num_seqs=2, final_state=True)
    torch.cuda.synchronize()
    assert torch.all(la <= 0)
    n = q.float().norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-2)
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()


# ---- gated output (RMSNorm x weight x sigmoid(gate)) after the recurrence ----------

def gated_ref(w, x, heads=None, eps=1e-6):
    from tests.gpu_helpers import oracle_prefill
    sel = slice(None) if heads is None else list(heads)
    ro, rf = oracle_prefill(w, heads)
    return lo.gated_rmsnorm(ro, np64(x.g_raw[:, sel]), np64(x.norm_weight), eps), rf


def run_gated(w, x, eps=1e-6):
    d = w.to(DEV)
    out, fin = kda.kda_prefill_gated(d.q, d.k, d.v, d.log_alpha, d.beta, x.g_raw.to(DEV),
                                     x.norm_weight.to(DEV), norm_eps=eps, initial_state=d.initial_state,
                                     cu_seqlens=d.cu_seqlens, final_state=True)
    plain_out, plain_fin = kda.kda_prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.initial_state, d.cu_seqlens,
                                           final_state=True)
    torch.cuda.synchronize()
    return out, fin, plain_fin


@pytest.mark.parametrize("mode", ["plain", "token_chunks", "ragged_only"])
def test_prefill_gated_tensor_core_path(mode):
    cu = [0, 64, 214, 300] if mode != "ragged_only" else [0, 37, 100]
    w = workloads.make_inputs(cu[-1], 2, 128, 128, dtype=torch.bfloat16, seed=61, cu_seqlens=cu, state_std=0.05)
    if mode == "token_chunks":
        w.log_alpha[70::41, :, ::4] = float("-inf")   # some chunks run token by token
    x = workloads.make_layer_inputs(cu[-1], 2, 128, 128, dtype=torch.bfloat16, seed=62, cu_seqlens=cu)
    out, fin, plain_fin = run_gated(w, x)
    ro, rf = gated_ref(w, x)
    e_out = rel_l2(np64(out), ro)
    assert e_out <= 5e-3, f"gated out rel L2 {e_out:.3e}"
    assert torch.equal(fin, plain_fin)                 # the gate does not touch the state
    assert rel_l2(np64(fin), rf) <= 5e-3


def test_prefill_gated_recurrent_path_fp32():
    cu = [0, 50, 130]
    w = workloads.make_inputs(cu[-1], 2, 64, 64, dtype=torch.float32, seed=63, cu_seqlens=cu)
    x = workloads.make_layer_inputs(cu[-1], 2, 64, 64, dtype=torch.float32, seed=64, cu_seqlens=cu)
    out, fin, _ = run_gated(w, x, eps=1e-5)
    ro, _ = gated_ref(w, x, eps=1e-5)
    assert rel_l2(np64(out), ro) <= 1e-4


def test_prefill_gated_full_size_sampled_heads():
    w = workloads.prefill_bf16(device=DEV)
    x = workloads.make_layer_inputs(w.total_tokens, 32, 128, 128, dtype=torch.bfloat16, seed=65,
                                    num_seqs=4, device=DEV)
    out, fin, plain_fin = run_gated(w, x)
    heads = [3, 30]
    ro, _ = gated_ref(w, x, heads=heads)
    assert rel_l2(np64(out[:, heads]), ro) <= 5e-3
    assert torch.equal(fin, plain_fin)


@pytest.mark.parametrize("T", [1, 2, 5, 16])
def test_decode_gated(T):
    from oracle import kda_oracle
    n = 6
    cu = [T * i for i in range(n + 1)]
    w = workloads.make_inputs(n * T, 4, 128, 128, dtype=torch.bfloat16, seed=66 + T, cu_seqlens=cu,
                              state_std=0.05)
    x = workloads.make_layer_inputs(n * T, 4, 128, 128, dtype=torch.bfloat16, seed=67, cu_seqlens=cu)
    d = w.to(DEV)
    S = d.initial_state.clone()
    out = kda.kda_decode_step_gated(d.q, d.k, d.v, d.log_alpha, d.beta, x.g_raw.to(DEV), x.norm_weight.to(DEV),
                                    S, norm_eps=1e-6)
    torch.cuda.synchronize()
    ro, rf = kda_oracle.prefill(np64(w.q), np64(w.k), np64(w.v), np64(w.log_alpha), np64(w.beta),
                                np64(w.initial_state), cu_seqlens=cu)
    ref = lo.gated_rmsnorm(ro, np64(x.g_raw), np64(x.norm_weight), 1e-6)
    assert rel_l2(np64(out), ref) <= 5e-3
    assert rel_l2(np64(S), rf) <= 5e-3


@pytest.mark.parametrize("impl", ["tensor_core", "recurrent"])
def test_prefill_gated_all_zero_rows_stay_finite(impl, monkeypatch):
    # beta = 0 from a zero state leaves S = 0, so every output row is exactly zero; the gated
    # output must then be zero (eps > 0 is required), never 0/0
    if impl == "recurrent":
        monkeypatch.setenv("KDA_PREFILL_IMPL", "recurrent")
    cu = [0, 70, 200]
    w = workloads.make_inputs(cu[-1], 2, 128, 128, dtype=torch.bfloat16, seed=68, cu_seqlens=cu)
    w.beta.zero_()
    x = workloads.make_layer_inputs(cu[-1], 2, 128, 128, dtype=torch.bfloat16, seed=69, cu_seqlens=cu)
    out, fin, _ = run_gated(w, x, eps=1e-6)
    assert torch.isfinite(out.float()).all()
    assert torch.count_nonzero(out) == 0 and torch.count_nonzero(fin) == 0
    ro, _ = gated_ref(w, x, eps=1e-6)
    assert np.all(ro == 0.0)


def test_decode_gated_all_zero_rows_stay_finite():
    n, T = 4, 3
    cu = [T * i for i in range(n + 1)]
    w = workloads.make_inputs(n * T, 2, 128, 128, dtype=torch.bfloat16, seed=70, cu_seqlens=cu)
    x = workloads.make_layer_inputs(n * T, 2, 128, 128, dtype=torch.bfloat16, seed=71, cu_seqlens=cu)
    d = w.to(DEV)
    d.beta.zero_()
    S = torch.zeros((n, 2, 128, 128), dtype=torch.float32, device=DEV)
    out = kda.kda_decode_step_gated(d.q, d.k, d.v, d.log_alpha, d.beta, x.g_raw.to(DEV), x.norm_weight.to(DEV),
                                    S, norm_eps=1e-6)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.count_nonzero(out) == 0


# ---- the front end fused into the prefill (kda_prefill_frontend) --------------------

def fused_layer_ref(x, heads=None, h0=None, eps=1e-6):
    """fp64 oracle: the layer front end, then the recurrence, on the same raw inputs."""
    from oracle import kda_oracle
    sel = slice(None) if heads is None else list(heads)
    cu = x.cu_seqlens.numpy()
    q, k, v, la, b = lo.frontend(np64(x.q_raw[:, sel]), np64(x.k_raw[:, sel]), np64(x.v_raw[:, sel]),
                                 np64(x.conv_q[sel]), np64(x.conv_k[sel]), np64(x.conv_v[sel]),
                                 np64(x.a_raw[:, sel]), np64(x.b_raw[:, sel]), cu_seqlens=cu, eps=eps)
    return kda_oracle.prefill(q, k, v, la, b, None if h0 is None else np64(h0[:, sel]), cu_seqlens=cu)


def run_fused_layer(x, h0=None, eps=1e-6):
    d = x.to(DEV)
    out, fin = kda.kda_prefill_frontend(d.q_raw, d.k_raw, d.v_raw, d.a_raw, d.b_raw, d.conv_q, d.conv_k,
                                        d.conv_v, initial_state=h0, cu_seqlens=d.cu_seqlens, final_state=True,
                                        eps=eps)
    torch.cuda.synchronize()
    return out, fin


@pytest.mark.parametrize("W", [1, 2, 3, 4])
def test_prefill_frontend_matches_oracle(W):
    # ragged sequences: the convolution's halo crosses chunk boundaries inside a sequence and
    # restarts at each sequence start (one-token and empty sequences included)
    cu = [0, 1, 77, 77, 200, 333, 500]
    x = workloads.make_layer_inputs(cu[-1], 2, 128, 128, W=W, dtype=torch.bfloat16, seed=80 + W, cu_seqlens=cu)
    h0 = torch.randn((6, 2, 128, 128), generator=torch.Generator().manual_seed(81), dtype=torch.float32) * 0.05
    out, fin = run_fused_layer(x, h0=h0.to(DEV))
    ro, rf = fused_layer_ref(x, h0=h0)
    assert rel_l2(np64(out), ro) <= 5e-3 and rel_l2(np64(fin), rf) <= 5e-3


def test_prefill_frontend_agrees_with_two_pass_path():
    cu = [0, 300, 640, 700]
    x = workloads.make_layer_inputs(cu[-1], 3, 128, 128, W=4, dtype=torch.bfloat16, seed=82, cu_seqlens=cu)
    out, fin = run_fused_layer(x, eps=1e-5)
    d = x.to(DEV)
    q, k, v, la, b = kda.kda_frontend(d.q_raw, d.k_raw, d.v_raw, d.a_raw, d.b_raw, d.conv_q, d.conv_k, d.conv_v,
                                      cu_seqlens=d.cu_seqlens, eps=1e-5)
    o2, f2 = kda.kda_prefill(q, k, v, la, b, None, d.cu_seqlens, final_state=True)
    torch.cuda.synchronize()
    assert rel_l2(np64(out), np64(o2)) <= 5e-3 and rel_l2(np64(fin), np64(f2)) <= 5e-3


def test_prefill_frontend_token_by_token_chunks():
    # decay logits far below zero make log alpha ~ a_raw, so some chunks leave the factored
    # range and run token by token from the processed tiles
    cu = [0, 64, 64 + 150, 400]
    x = workloads.make_layer_inputs(cu[-1], 2, 128, 128, W=4, dtype=torch.bfloat16, seed=83, cu_seqlens=cu)
    x.a_raw[70:90, :, ::3] = -200.0
    out, fin = run_fused_layer(x)
    ro, rf = fused_layer_ref(x)
    assert rel_l2(np64(out), ro) <= 5e-3 and rel_l2(np64(fin), rf) <= 5e-3


def test_prefill_frontend_full_size_sampled_heads():
    x = workloads.make_layer_inputs(4 * 8192, 32, 128, 128, W=4, dtype=torch.bfloat16, seed=84, num_seqs=4,
                                    device=DEV)
    out, fin = run_fused_layer(x)
    heads = [0, 31]
    ro, rf = fused_layer_ref(x, heads=heads)
    assert rel_l2(np64(out[:, heads]), ro) <= 5e-3 and rel_l2(np64(fin[:, heads]), rf) <= 5e-3
