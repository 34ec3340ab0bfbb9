"""Run every entry point once on a library built with -DKDA_CHECK_BOUNDS and check
that no kernel skipped a global-memory access because its index left its buffer.

Executed in a child process by tests/test_bounds_gpu.py (so that it loads its own
copy of the library); prints one line per case and "bounds ok" at the end, and
exits non-zero on the first case whose status is not KDA_OK.
"""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main() -> int:
    from linear_attention_06_gb300 import _lib
    from linear_attention_06_gb300 import build as _build
    _lib.LIB_PATH = _build.build(extra_flags=["-DKDA_CHECK_BOUNDS"], tag="bounds")
    _lib._lib = None

    import torch

    import linear_attention_06_gb300 as kda
    from linear_attention_06_gb300 import workloads

    dev = torch.device("cuda")
    failures = []

    def check(name):
        st = kda.kda_device_status()
        print(f"{name}: {_lib.status_string(st)}", flush=True)
        if st != _lib.KDA_OK:
            failures.append(name)

    assert kda.kda_device_status() == _lib.KDA_OK

    # prefill: tensor-core path (ragged chunks, empty and one-token sequences, initial and
    # final states), the token-by-token chunks, and the fp32 recurrent path for each head size
    lens = [1, 64, 65, 130, 0, 17, 200]
    cu = workloads.cu_from_lengths(lens)
    for dtype, dk, dv in ((torch.bfloat16, 128, 128), (torch.float32, 128, 128), (torch.bfloat16, 64, 128),
                          (torch.float32, 128, 64), (torch.bfloat16, 64, 64)):
        w = workloads.make_inputs(cu[-1], 3, dk, dv, dtype=dtype, seed=dk + dv, cu_seqlens=cu,
                                  state_std=0.05).to(dev)
        kda.kda_prefill(w.q, w.k, w.v, w.log_alpha, w.beta, w.initial_state,
                        torch.tensor(cu, dtype=torch.int32, device=dev), final_state=True)
        check(f"prefill {dtype} dk={dk} dv={dv}")
        ck = [sorted({p for p in (64, 128, L) if 0 < p <= L}) for L in lens]
        kda.kda_prefill_checkpointed(w.q, w.k, w.v, w.log_alpha, w.beta, ck, w.initial_state, cu)
        check(f"prefill with checkpoints {dtype} dk={dk} dv={dv}")
    w = workloads.make_inputs(cu[-1], 2, 128, 128, seed=8, cu_seqlens=cu, state_std=0.05).to(dev)
    w.log_alpha.mul_(40.0)                                   # every chunk token by token
    kda.kda_prefill(w.q, w.k, w.v, w.log_alpha, w.beta, w.initial_state,
                    torch.tensor(cu, dtype=torch.int32, device=dev), final_state=True)
    check("prefill, token-by-token chunks")
    # the split prefill: ragged sequences in one pass, a token-by-token chunk among them, and one
    # long sequence run in segments (the chunk-local pass of the next segment overlapping the chains)
    w = workloads.make_inputs(cu[-1], 3, 128, 128, seed=10, cu_seqlens=cu, state_std=0.05).to(dev)
    w.log_alpha[70:72].mul_(400.0)
    kda.kda_prefill_split(w.q, w.k, w.v, w.log_alpha, w.beta, w.initial_state,
                          torch.tensor(cu, dtype=torch.int32, device=dev), final_state=True)
    check("split prefill, ragged")
    ws_ = workloads.make_inputs(17000, 2, 128, 128, seed=11, cu_seqlens=[0, 17000], state_std=0.05).to(dev)
    kda.kda_prefill_split(ws_.q, ws_.k, ws_.v, ws_.log_alpha, ws_.beta, ws_.initial_state,
                          torch.tensor([0, 17000], dtype=torch.int32, device=dev), final_state=True)
    check("split prefill, one sequence in segments")
    # the front end fused into the prefill (ragged sequences, halo rows at sequence starts)
    x = workloads.make_layer_inputs(cu[-1], 3, 128, 128, W=4, seed=12, cu_seqlens=cu).to(dev)
    kda.kda_prefill_frontend(x.q_raw, x.k_raw, x.v_raw, x.a_raw, x.b_raw, x.conv_q, x.conv_k, x.conv_v,
                             cu_seqlens=cu, final_state=True)
    check("prefill with the front end fused")
    wd = workloads.make_inputs(4 * 128, 2, 128, 128, seed=9, num_seqs=4).to(dev)
    kda.kda_prefill(wd.q, wd.k, wd.v, wd.log_alpha, wd.beta, None, None, final_state=True, num_seqs=4)
    check("prefill, dense batch without cu_seqlens")

    # the layer around the recurrence: front end for every width and both dtypes, gated output
    for dtype in (torch.bfloat16, torch.float32):
        for W in (1, 2, 3, 4):
            x = workloads.make_layer_inputs(cu[-1], 3, 128, 128, W=W, dtype=dtype, seed=W,
                                            cu_seqlens=cu).to(dev)
            q, k, v, la, b = kda.kda_frontend(x.q_raw, x.k_raw, x.v_raw, x.a_raw, x.b_raw, x.conv_q,
                                              x.conv_k, x.conv_v, cu_seqlens=cu)
            check(f"front end {dtype} W={W}")
        kda.kda_prefill_gated(q, k, v, la, b, x.g_raw, x.norm_weight, cu_seqlens=cu)
        check(f"gated prefill {dtype}")
    x = workloads.make_layer_inputs(cu[-1], 2, 64, 128, W=4, seed=5, cu_seqlens=cu).to(dev)
    kda.kda_frontend(x.q_raw, x.k_raw, x.v_raw, x.a_raw, x.b_raw, x.conv_q, x.conv_k, x.conv_v,
                     cu_seqlens=cu)
    check("front end dk=64 dv=128")

    # decode: one, two, five and sixteen tokens per sequence, plain and gated, every head size
    for T in (1, 2, 5, 16):
        for dk, dv in ((128, 128), (64, 128), (128, 64), (64, 64)):
            n = 9
            c = [T * i for i in range(n + 1)]
            d = workloads.make_inputs(n * T, 3, dk, dv, seed=T + dk, cu_seqlens=c, state_std=0.05).to(dev)
            S = d.initial_state.clone()
            kda.kda_decode_step(d.q, d.k, d.v, d.log_alpha, d.beta, S)
            check(f"decode T={T} dk={dk} dv={dv}")
            g = workloads.make_layer_inputs(n * T, 3, dk, dv, seed=T, cu_seqlens=c).to(dev)
            kda.kda_decode_step_gated(d.q, d.k, d.v, d.log_alpha, d.beta, g.g_raw, g.norm_weight, S)
            check(f"gated decode T={T} dk={dk} dv={dv}")

    # multi-token decode: fp32 (the one-token kernel's loop), and bf16 steps whose decay sends them
    # token by token
    for T in (5, 16):
        n = 9
        c = [T * i for i in range(n + 1)]
        d = workloads.make_inputs(n * T, 3, 128, 128, dtype=torch.float32, seed=T, cu_seqlens=c,
                                  state_std=0.05).to(dev)
        kda.kda_decode_step(d.q, d.k, d.v, d.log_alpha, d.beta, d.initial_state.clone())
        check(f"decode fp32 T={T}")
        d = workloads.make_inputs(n * T, 3, 128, 128, seed=T + 1, cu_seqlens=c, state_std=0.05).to(dev)
        d.log_alpha.mul_(200.0)
        kda.kda_decode_step(d.q, d.k, d.v, d.log_alpha, d.beta, d.initial_state.clone())
        check(f"decode strong decay T={T}")

    if failures:
        print("index checks failed:", ", ".join(failures))
        return 1
    print("bounds ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
