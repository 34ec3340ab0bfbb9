"""Seeded synthetic KDA workloads (input generators only).

This module holds no part of the KDA recurrence: it only draws inputs with the
shapes and distributions of the K3-shaped workloads, and is shared by the
tests, the benchmark and the smoke check.  Both the CUDA path and the CPU
oracle receive exactly the tensors produced here.

Recipe (per workload; all draws from one ``torch.Generator`` seeded with the
workload's seed, in the order q, k, v, alpha-noise, beta-noise, state,
lengths):
  q, k   ~ N(0, 1), L2-normalised per (token, head) in fp32, then cast to the
           input dtype (the library expects normalised q and k; it does not
           normalise them itself).
  v      ~ N(0, 1), cast to the input dtype.
  log_alpha = logsigmoid(N(mu, 1)) per (token, head, key channel), fp32
           (alpha = sigmoid(N(mu, 1)); mu = 2 for the tiny fp32 case, 3 else).
  beta   = sigmoid(N(0, 1)) per (token, head), in the input dtype.
  initial state: zeros, or N(0, 0.05) (standard deviation 0.05) in fp32.
  varlen lengths: floor(exp(U(ln 128, ln 32768))) per sequence.

Layer inputs (``make_layer_inputs``, for the front end before the recurrence and
the gated output after it; raw draws only, in the order q, k, v, a, b, gate,
conv q, conv k, conv v, norm weight):
  q_raw, k_raw, v_raw ~ N(0, 1) in the input dtype (projection outputs);
  a_raw ~ N(mu, 1) fp32 (decay logits; logsigmoid of it is log_alpha);
  b_raw ~ N(0, 1), gate logits g_raw ~ N(0, 1) in the input dtype;
  convolution taps ~ N(0, 1/W) fp32 (width W), norm weight ~ 1 + N(0, 0.1) fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass
class Workload:
    name: str
    q: torch.Tensor            # [T, H, dk]
    k: torch.Tensor            # [T, H, dk]
    v: torch.Tensor            # [T, H, dv]
    log_alpha: torch.Tensor    # [T, H, dk] fp32
    beta: torch.Tensor         # [T, H]
    initial_state: torch.Tensor | None   # [N, H, dk, dv] fp32 or None
    cu_seqlens: torch.Tensor   # [N+1] int32 (host copy)
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.numel()) - 1

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[0])

    def to(self, device):
        def mv(t):
            return None if t is None else t.to(device)
        return Workload(self.name, mv(self.q), mv(self.k), mv(self.v), mv(self.log_alpha),
                        mv(self.beta), mv(self.initial_state), self.cu_seqlens.clone(),
                        dict(self.meta))


def _normal(shape, gen, device, mean=0.0, std=1.0):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std + mean


def make_inputs(T, H, dk, dv, dtype=torch.bfloat16, seed=0, alpha_mu=3.0,
                cu_seqlens=None, num_seqs=1, state_std=None, device="cpu",
                name="custom"):
    """Draw one packed workload.  ``cu_seqlens`` (list or tensor) overrides the
    equal split into ``num_seqs`` sequences."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    q = _normal((T, H, dk), gen, device)
    k = _normal((T, H, dk), gen, device)
    v = _normal((T, H, dv), gen, device)
    q = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    log_alpha = torch.nn.functional.logsigmoid(_normal((T, H, dk), gen, device, mean=alpha_mu))
    beta = torch.sigmoid(_normal((T, H), gen, device))
    if cu_seqlens is None:
        assert T % num_seqs == 0
        cu = torch.arange(num_seqs + 1, dtype=torch.int32) * (T // num_seqs)
    else:
        cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu()
    n = int(cu.numel()) - 1
    h0 = None
    if state_std is not None:
        h0 = _normal((n, H, dk, dv), gen, device, std=state_std)
    return Workload(name, q.to(dtype), k.to(dtype), v.to(dtype), log_alpha.contiguous(),
                    beta.to(dtype), h0, cu,
                    dict(T=T, H=H, dk=dk, dv=dv, dtype=str(dtype).replace("torch.", ""),
                         seed=seed, alpha_mu=alpha_mu))


@dataclass
class LayerInputs:
    name: str
    q_raw: torch.Tensor        # [T, H, dk]
    k_raw: torch.Tensor        # [T, H, dk]
    v_raw: torch.Tensor        # [T, H, dv]
    a_raw: torch.Tensor        # [T, H, dk] fp32
    b_raw: torch.Tensor        # [T, H]
    g_raw: torch.Tensor        # [T, H, dv]
    conv_q: torch.Tensor       # [H, dk, W] fp32
    conv_k: torch.Tensor       # [H, dk, W] fp32
    conv_v: torch.Tensor       # [H, dv, W] fp32
    norm_weight: torch.Tensor  # [dv] fp32
    cu_seqlens: torch.Tensor   # [N+1] int32 (host copy)

    def to(self, device):
        f = {k: (v.to(device) if isinstance(v, torch.Tensor) and k != "cu_seqlens" else v)
             for k, v in self.__dict__.items()}
        f["cu_seqlens"] = self.cu_seqlens.clone()
        return LayerInputs(**f)


def make_layer_inputs(T, H, dk, dv, W=4, dtype=torch.bfloat16, seed=0, alpha_mu=3.0,
                      cu_seqlens=None, num_seqs=1, device="cpu", name="layer"):
    """Raw projection outputs and layer weights for the front end and the gated
    output (see the module docstring for the recipe)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    q = _normal((T, H, dk), gen, device)
    k = _normal((T, H, dk), gen, device)
    v = _normal((T, H, dv), gen, device)
    a = _normal((T, H, dk), gen, device, mean=alpha_mu)
    b = _normal((T, H), gen, device)
    g = _normal((T, H, dv), gen, device)
    std = 1.0 / math.sqrt(W)
    cq = _normal((H, dk, W), gen, device, std=std)
    ck = _normal((H, dk, W), gen, device, std=std)
    cv = _normal((H, dv, W), gen, device, std=std)
    nw = _normal((dv,), gen, device, mean=1.0, std=0.1)
    if cu_seqlens is None:
        assert T % num_seqs == 0
        cu = torch.arange(num_seqs + 1, dtype=torch.int32) * (T // num_seqs)
    else:
        cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu()
    return LayerInputs(name, q.to(dtype), k.to(dtype), v.to(dtype), a.contiguous(), b.to(dtype),
                       g.to(dtype), cq, ck, cv, nw, cu)


def varlen_lengths(num_seqs, seed, lo=128, hi=32768):
    """floor(exp(U(ln lo, ln hi))) per sequence, from a CPU generator."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed) + 1_000_003)
    u = torch.rand((num_seqs,), generator=gen, dtype=torch.float64)
    lens = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).floor().to(torch.int64)
    return [int(x) for x in lens.clamp(lo, hi)]


def cu_from_lengths(lengths):
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return cu


# ---------------------------------------------------------------------------
# The five K3-shaped workloads.
# ---------------------------------------------------------------------------

def tiny_fp32(device="cpu"):
    """B=1, H=2, T=256, dk=dv=64, fp32, zero initial state, alpha=sigmoid(N(2,1)), seed 0."""
    return make_inputs(256, 2, 64, 64, dtype=torch.float32, seed=0, alpha_mu=2.0,
                       num_seqs=1, device=device, name="prefill_tiny_fp32_B1_H2_T256_d64")


def prefill_bf16(device="cpu", B=4, T=8192, H=32, d=128, seed=1):
    """B=4, H=32, T=8192, dk=dv=128, bf16 q/k/v/beta, fp32 log_alpha, zero state."""
    return make_inputs(B * T, H, d, d, dtype=torch.bfloat16, seed=seed, alpha_mu=3.0,
                       num_seqs=B, device=device, name=f"prefill_bf16_B{B}_H{H}_T{T}_d{d}")


def decode_inputs(device="cpu", N=256, H=32, d=128, seed=2):
    """256 sequences x H=32 x dk=dv=128, one token each; state ~ N(0, 0.05) fp32."""
    return make_inputs(N, H, d, d, dtype=torch.bfloat16, seed=seed, alpha_mu=3.0,
                       cu_seqlens=list(range(N + 1)), state_std=0.05, device=device,
                       name=f"decode_N{N}_H{H}_d{d}")


def long_prefill(device="cpu", T=131072, H=32, d=128, seed=3):
    """B=1, H=32, T=131072, dk=dv=128 bf16; the resume test splits it at T/2."""
    return make_inputs(T, H, d, d, dtype=torch.bfloat16, seed=seed, alpha_mu=3.0,
                       num_seqs=1, device=device, name=f"long_prefill_T{T}_H{H}_d{d}")


def varlen_prefill(device="cpu", num_seqs=64, H=32, d=128, seed=4):
    """64 log-uniform(128, 32768) lengths packed with cu_seqlens, per-sequence
    initial states ~ N(0, 0.05)."""
    lens = varlen_lengths(num_seqs, seed)
    cu = cu_from_lengths(lens)
    return make_inputs(cu[-1], H, d, d, dtype=torch.bfloat16, seed=seed, alpha_mu=3.0,
                       cu_seqlens=cu, state_std=0.05, device=device,
                       name=f"varlen_prefill_N{num_seqs}_H{H}_d{d}")
