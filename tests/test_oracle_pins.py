"""Pins for the fp64 oracle (CPU only, no GPU).

Each test checks the oracle against something other than itself: a
hand-derived example, an independent unrolled-product formulation, closed
forms and invariants of the recurrence
    S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = S_t^T q_t,
and the special cases the pages name (DeltaNet, Gated DeltaNet: "Kimi K3
architecture: KDA, MLA and MoE", section "KDA is a writable state").  The last
test builds mutant oracles with one planted mistake each and checks that the
pins catch every one of them.
"""
import json
import os

import numpy as np
import pytest

from oracle import kda_oracle
from tests.bruteforce import gated_deltanet, unrolled_products

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")


def rand_case(rng, T, H, dk, dv, unit_keys=False, n=1, alpha_lo=0.3):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    la = np.log(rng.uniform(alpha_lo, 1.0, (T, H, dk)))
    b = rng.uniform(0.0, 1.0, (T, H))
    h0 = rng.standard_normal((n, H, dk, dv))
    return q, k, v, la, b, h0


def run_golden(lib=None):
    with open(GOLDEN) as f:
        ex = json.load(f)["examples"]
    errs = []
    for e in ex:
        T = len(e["beta"])
        dk, dv = e["dk"], e["dv"]
        q = np.array(e["q"]).reshape(T, 1, dk)
        k = np.array(e["k"]).reshape(T, 1, dk)
        v = np.array(e["v"]).reshape(T, 1, dv)
        la = np.log(np.array(e["alpha"])).reshape(T, 1, dk)
        b = np.array(e["beta"]).reshape(T, 1)
        h0 = np.array(e["initial_state"]).reshape(1, 1, dk, dv)
        out, fin = kda_oracle.prefill(q, k, v, la, b, h0, lib=lib)
        errs.append(max(np.abs(out[:, 0] - np.array(e["out"])).max(),
                        np.abs(fin[0, 0] - np.array(e["final_state"])).max()))
    return max(errs)


def test_hand_examples():
    assert run_golden() < 1e-13


def brute_force_error(rng, lib=None, T=12, H=2, dk=8, dv=6):
    q, k, v, la, b, h0 = rand_case(rng, T, H, dk, dv)
    out, fin = kda_oracle.prefill(q, k, v, la, b, h0, lib=lib)
    err = 0.0
    for h in range(H):
        o_ref, s_ref = unrolled_products(q[:, h], k[:, h], v[:, h], la[:, h], b[:, h], h0[0, h])
        err = max(err, np.abs(out[:, h] - o_ref).max() / np.abs(o_ref).max(),
                  np.abs(fin[0, h] - s_ref).max() / np.abs(s_ref).max())
    return err


@pytest.mark.parametrize("T,dk,dv", [(1, 4, 4), (5, 8, 6), (12, 6, 8), (16, 8, 8)])
def test_bruteforce_unrolled_products(T, dk, dv):
    rng = np.random.default_rng(100 + T)
    assert brute_force_error(rng, T=T, dk=dk, dv=dv) < 1e-12


def test_p1_no_write_no_decay_keeps_state():
    rng = np.random.default_rng(1)
    q, k, v, la, b, h0 = rand_case(rng, 40, 3, 16, 12)
    la[:] = 0.0
    b[:] = 0.0
    out, fin = kda_oracle.prefill(q, k, v, la, b, h0)
    assert np.array_equal(fin[0], h0[0])
    ref = np.einsum("hij,thi->thj", h0[0], q)
    assert np.abs(out - ref).max() < 1e-12


def test_p2_unit_key_retrieval():
    rng = np.random.default_rng(2)
    q, k, v, la, b, h0 = rand_case(rng, 50, 2, 16, 12, unit_keys=True)
    la[:] = 0.0
    b[:] = 1.0
    out, _ = kda_oracle.prefill(k, k, v, la, b, h0)  # query with the key just written
    assert np.abs(out - v).max() < 1e-12


def test_p3_resume_equals_full_run():
    rng = np.random.default_rng(3)
    q, k, v, la, b, h0 = rand_case(rng, 300, 2, 16, 16)
    full_out, full_fin = kda_oracle.prefill(q, k, v, la, b, h0)
    for m in (1, 64, 137):
        o1, s1 = kda_oracle.prefill(q[:m], k[:m], v[:m], la[:m], b[:m], h0)
        o2, s2 = kda_oracle.prefill(q[m:], k[m:], v[m:], la[m:], b[m:], s1)
        assert np.array_equal(np.concatenate([o1, o2]), full_out)
        assert np.array_equal(s2, full_fin)


def test_p5_decay_only_closed_form():
    rng = np.random.default_rng(5)
    q, k, v, la, b, h0 = rand_case(rng, 30, 2, 8, 5, alpha_lo=0.5)
    b[:] = 0.0
    out, fin = kda_oracle.prefill(q, k, v, la, b, h0)
    g = np.exp(np.cumsum(la, axis=0))                       # [T, H, dk]
    S_t = g[:, :, :, None] * h0[0][None]                    # [T, H, dk, dv]
    ref_out = np.einsum("thij,thi->thj", S_t, q)
    assert np.abs(fin[0] - S_t[-1]).max() < 1e-12
    assert np.abs(out - ref_out).max() < 1e-12


def test_p6_special_cases_gated_deltanet_and_deltanet():
    rng = np.random.default_rng(6)
    q, k, v, la, b, h0 = rand_case(rng, 25, 2, 8, 6, unit_keys=True)
    scalar = np.log(rng.uniform(0.5, 1.0, (25, 2)))
    la_scalar = np.repeat(scalar[:, :, None], 8, axis=2)
    for log_g in (scalar, np.zeros_like(scalar)):           # Gated DeltaNet, DeltaNet
        la_use = la_scalar if log_g is scalar else np.zeros_like(la_scalar)
        out, fin = kda_oracle.prefill(q, k, v, la_use, b, h0)
        for h in range(2):
            o_ref, s_ref = gated_deltanet(q[:, h], k[:, h], v[:, h], log_g[:, h], b[:, h], h0[0, h])
            assert np.abs(out[:, h] - o_ref).max() < 1e-12 * np.abs(o_ref).max()
            assert np.abs(fin[0, h] - s_ref).max() < 1e-12 * np.abs(s_ref).max()


def test_p7_householder_preserves_frobenius_norm():
    rng = np.random.default_rng(7)
    q, k, v, la, b, h0 = rand_case(rng, 64, 2, 16, 8, unit_keys=True)
    la[:] = 0.0
    b[:] = 2.0
    v[:] = 0.0
    for T in (1, 7, 64):
        _, fin = kda_oracle.prefill(q[:T], k[:T], v[:T], la[:T], b[:T], h0)
        n0 = np.linalg.norm(h0[0], axis=(1, 2))
        n1 = np.linalg.norm(fin[0], axis=(1, 2))
        assert np.abs(n1 - n0).max() < 1e-12 * n0.max()


def test_p8_orthonormal_keys_closed_form():
    rng = np.random.default_rng(8)
    dk, dv, T = 16, 8, 12
    qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = qm[:, :T].T.reshape(T, 1, dk)                       # orthonormal rows
    q = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    la = np.zeros((T, 1, dk))
    b = np.ones((T, 1))
    h0 = rng.standard_normal((1, 1, dk, dv))
    _, fin = kda_oracle.prefill(q, k, v, la, b, h0)
    S0 = h0[0, 0]
    ref = S0 + sum(np.outer(k[t, 0], v[t, 0] - S0.T @ k[t, 0]) for t in range(T))
    assert np.abs(fin[0, 0] - ref).max() < 1e-12


def test_p9_varlen_equals_separate_runs():
    rng = np.random.default_rng(9)
    lens = [1, 17, 64, 5, 100]
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, la, b, _ = rand_case(rng, int(cu[-1]), 2, 8, 8)
    h0 = rng.standard_normal((len(lens), 2, 8, 8))
    out, fin = kda_oracle.prefill(q, k, v, la, b, h0, cu_seqlens=cu)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        o_n, f_n = kda_oracle.prefill(q[s:e], k[s:e], v[s:e], la[s:e], b[s:e], h0[n:n + 1])
        assert np.array_equal(out[s:e], o_n)
        assert np.array_equal(fin[n], f_n[0])


def test_empty_sequences_leave_state_unchanged():
    rng = np.random.default_rng(10)
    cu = np.array([0, 0, 3, 3])
    q, k, v, la, b, _ = rand_case(rng, 3, 1, 4, 4)
    h0 = rng.standard_normal((3, 1, 4, 4))
    _, fin = kda_oracle.prefill(q, k, v, la, b, h0, cu_seqlens=cu)
    assert np.array_equal(fin[0], h0[0]) and np.array_equal(fin[2], h0[2])


def test_decode_step_equals_one_token_prefill():
    rng = np.random.default_rng(11)
    q, k, v, la, b, h0 = rand_case(rng, 6, 3, 8, 8, n=6)
    out_d, S_d = kda_oracle.decode_step(q, k, v, la, b, h0)
    out_p, S_p = kda_oracle.prefill(q, k, v, la, b, h0, cu_seqlens=np.arange(7))
    assert np.array_equal(out_d, out_p) and np.array_equal(S_d, S_p)


@pytest.mark.parametrize("mutation", [1, 2, 3, 4, 5, 6])
def test_pins_catch_planted_mistakes(mutation):
    lib = kda_oracle.load_mutant(mutation)
    caught = run_golden(lib) > 1e-6
    caught = caught or brute_force_error(np.random.default_rng(77), lib=lib, dk=6, dv=6) > 1e-6
    assert caught, f"mutation {mutation} slipped through the pins"
