"""Cycle profile of the tensor-core prefill kernel, by phase (diagnostic tool).

    python -m linear_attention_06_gb300.phase_profile --mode phase
    python -m linear_attention_06_gb300.phase_profile --mode trace

Each mode builds a separately configured copy of the library under
``_build/<mode>/`` and leaves the package's own ``libkda.so`` alone; the product
build contains none of the code below.

``phase`` (``-DKDA_PHASE_TIMING``): the first thread of each role adds the SM
clock it spends in each phase of its chunk loop to a counter, summed over all
blocks; printed as cycles per chunk.  The clock reads and counter updates slow
the kernel by about a quarter, so the shares matter more than the totals.

``trace`` (``-DKDA_TRACE_EVENTS``): for a window of 12 consecutive chunks
(five windows across the sequence, each read after three launches), block 0
records the clock at which each of the four tensor-core product groups is
issued (by the issuing thread) and the clock at which an extra observer warp,
probing the groups' completion barriers without blocking, first sees it
complete; a stamp later than the issue of a product that waits for that group
is replaced by that issue.  From this it prints how long each group takes from
issue to completion, and the share of the time in which the tensor pipe holds
products ("GEMM phases": the union of the issue-to-completion intervals) that
their arithmetic needs at the pipe's dense bf16 rate of 8192 flop per SM cycle
(an M=128, N=256, K=16 product per 128 cycles); stamps can only be late, so
that share is a lower bound.  Only block 0 is instrumented and the events stay
in shared memory until the block ends; the launch time is printed so that it can
be set against the uninstrumented kernel's (the stamped block runs a few per
cent slower).

The workload is the benchmark prefill: B=4 sequences of T=8192 tokens, H=32
heads, dk=dv=128, bf16 inputs, zero initial state.
"""
from __future__ import annotations

import argparse
import ctypes
import statistics

from . import _lib
from . import build as _build

FLOP_PER_SM_CYCLE = 8192
TRACE_CHUNKS, TRACE_EVENTS = 12, 8        # the kernel's traced window of block 0
TRACE_WINDOWS = (16, 40, 64, 88, 112)     # first chunks of the windows traced in turn
MMA_N64 = 2 * 128 * 64 * 16           # one M=128, N=64, K=16 product
MMA_N128 = 2 * 128 * 128 * 16         # one M=128, N=128, K=16 product

# product groups of one chunk: (name, issue event, completion event, flops)
GROUPS = [
    ("Gram [Khat; Qhat] Kb^T (8 x N64, both operands in smem)", 0, 1, 8 * MMA_N64),
    ("W'^T = Khat^T T^T, U^T = V^T T^T (8 x N64, smem)", 2, 3, 8 * MMA_N64),
    ("Delta^T = U^T - Ss^T W'^T (8 x N64, A in TMEM)", 4, 5, 8 * MMA_N64),
    ("O^T, S^T += Delta^T Kb (12 x N64 + 4 x N128, A in TMEM)", 6, 7, 12 * MMA_N64 + 4 * MMA_N128),
]

# phase counter slots of the kernel's diagnostic build
PHASES = {
    0: "P: wait for log alpha", 4: "P: suffix sums", 2: "P: wait for Kb/P slot", 3: "P: wait for q/k",
    5: "P: operand tiles", 25: "P: Gram issue",
    26: "S: wait for Gram", 6: "S: read Gram", 15: "S: UT solve", 7: "S: wait for v / U slot",
    1: "S: W'/U issue",
    8: "B: wait for W'/U", 9: "B: decay state", 10: "B: read W'", 24: "B: Delta issue",
    11: "B: wait for Delta", 12: "B: pack Delta", 22: "B: hand to issuer", 16: "B: store output",
    13: "B: wait for state/output", 14: "B: chunk end sync",
    18: "Q: wait for alpha/v slot", 19: "Q: load alpha/v", 20: "Q: wait for q/k slot", 21: "Q: load q/k",
}
SOLVE_STEPS = {27: "diagonal blocks", 28: "32x32 halves", 29: "B A^-1", 30: "lower-left quarter"}


def _load(mode: str):
    flag = {"phase": "-DKDA_PHASE_TIMING", "trace": "-DKDA_TRACE_EVENTS"}[mode]
    path = _build.build(extra_flags=[flag], tag=mode)
    _lib.LIB_PATH = path
    _lib._lib = None
    return _lib.lib()


def _run(kda, wl, cu, launches):
    import torch
    ms = []
    for _ in range(launches):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        kda.kda_prefill(wl.q, wl.k, wl.v, wl.log_alpha, wl.beta, None, cu, final_state=True)
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    return ms


def _union(intervals):
    total, end = 0, None
    for a, b in sorted(intervals):
        if end is None or a > end:
            total += b - a
            end = b
        elif b > end:
            total += b - end
            end = b
    return total


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--mode", choices=["phase", "trace"], default="trace")
    args = ap.parse_args(argv)

    L = _load(args.mode)
    import torch

    import linear_attention_06_gb300 as kda
    from linear_attention_06_gb300 import workloads

    wl = workloads.prefill_bf16(device="cuda")
    cu = wl.cu_seqlens.cuda()
    nblocks = wl.cu_seqlens.numel() - 1
    H = wl.q.shape[1]
    nch = wl.q.shape[0] // nblocks // 64
    print(f"workload {wl.name}: {nblocks} sequences x {H} heads, {nch} chunks each")

    if args.mode == "phase":
        L.kda_debug_phase_cycles.argtypes = [ctypes.c_void_p, ctypes.c_int]
        buf = (ctypes.c_ulonglong * 32)()
        _run(kda, wl, cu, 2)
        L.kda_debug_phase_cycles(buf, 1)
        ms = _run(kda, wl, cu, 1)
        L.kda_debug_phase_cycles(buf, 1)
        chunks = nblocks * H * nch
        print(f"launch {ms[0]:.3f} ms (phase-timed build)")
        for role in "PSBQ":
            idx = [i for i, n in PHASES.items() if n.startswith(role + ":")]
            tot = sum(buf[i] for i in idx)
            print(f"role {role}: {tot / chunks:8.0f} cycles per chunk")
            for i in idx:
                print(f"  {PHASES[i]:28s} {buf[i] / chunks:8.0f}  {100.0 * buf[i] / max(tot, 1):5.1f}%")
            if role == "S":
                for i, n in SOLVE_STEPS.items():
                    print(f"    (solve: {n:20s} {buf[i] / chunks:8.0f})")
        return

    L.kda_debug_trace.argtypes = [ctypes.c_void_p]
    L.kda_debug_set_trace_first.argtypes = [ctypes.c_int]
    ms, windows = [], []
    for first in TRACE_WINDOWS:
        if first + TRACE_CHUNKS > nch:
            continue
        if L.kda_debug_set_trace_first(first) != 0:
            raise RuntimeError("kda_debug_set_trace_first failed")
        ms += _run(kda, wl, cu, 3)
        tr = (ctypes.c_uint32 * (TRACE_CHUNKS * TRACE_EVENTS))()
        if L.kda_debug_trace(tr) != 0:
            raise RuntimeError("kda_debug_trace failed")
        windows.append((first, _window([[tr[i * TRACE_EVENTS + e] for e in range(TRACE_EVENTS)]
                                        for i in range(TRACE_CHUNKS)], first)))
    need_all = sum(g[3] for g in GROUPS) / FLOP_PER_SM_CYCLE
    print(f"launch {statistics.median(ms):.3f} ms (median of {len(ms)}; only block 0 traced)")
    print(f"tensor arithmetic per chunk: {need_all:.0f} cycles at the dense rate")
    for first, w in windows:
        print(f"  chunks {first}..{first + TRACE_CHUNKS - 1}: period {w['period']:.0f}, GEMM phases "
              f"{w['busy']:.0f} cycles per chunk, utilisation {100.0 * need_all / w['busy']:.1f}%, "
              f"{w['late']} of {4 * TRACE_CHUNKS} stamps replaced by a dependent issue")
    period = statistics.mean(w["period"] for _, w in windows)
    busy = statistics.mean(w["busy"] for _, w in windows)
    print(f"over {len(windows)} windows: period {period:.0f} cycles per chunk, tensor arithmetic "
          f"{100.0 * need_all / period:.1f}% of it")
    print("issue to completion, cycles (median over the traced chunks) and arithmetic share:")
    for g, (name, _, _, fl) in enumerate(GROUPS):
        d = statistics.median(v for _, w in windows for v in w["dur"][g])
        need = fl / FLOP_PER_SM_CYCLE
        print(f"  {name:58s} {d:7.0f}  needs {need:5.0f}  ({100.0 * need / d:5.1f}%)")
    print(f"GEMM phases (tensor pipe holds products): {busy:.0f} cycles per chunk "
          f"({100.0 * busy / period:.1f}% of the period); tensor-pipe utilisation over them "
          f"{100.0 * need_all / busy:.1f}% of the dense bf16 rate (a lower bound: stamps can only be late)")


def _window(raw, first):
    """Period, per-group issue-to-completion cycles and GEMM-phase cycles per chunk of one
    traced window (raw: TRACE_CHUNKS x TRACE_EVENTS 32-bit clocks)."""
    if any(v == 0 for row in raw for v in row):
        raise RuntimeError(f"window {first}: trace events missing")
    base = raw[0][0]
    ev = [[(v - base) % (1 << 32) for v in row] for row in raw]   # 32-bit clock, relative
    rows = range(TRACE_CHUNKS)
    for i in rows:
        for _, s, e, _ in GROUPS:
            if ev[i][e] < ev[i][s]:
                raise RuntimeError(f"chunk {first + i}: completion before issue ({s}/{e})")
    period = (ev[-1][0] - ev[0][0]) / (TRACE_CHUNKS - 1)
    # A completion stamp can trail the true completion (the watching warp sleeps between
    # probes).  Each group's completion is also bounded by the issue of a product that
    # waits for it: W'/U of chunk n by Gram n (team S reads the Gram first), Delta by
    # W'/U (group B waits for them), state/output by Delta (group B packs Delta first),
    # Gram of chunk n+2 by state/output n (it frees the slots that Gram reuses).
    done = [[ev[i][1], ev[i][3], ev[i][5], ev[i][7]] for i in rows]
    bound = [[ev[i][2], ev[i][4], ev[i][6], ev[i + 2][0] if i + 2 < TRACE_CHUNKS else None] for i in rows]
    tight = [[d if b is None else min(d, b) for d, b in zip(done[i], bound[i])] for i in rows]
    late = sum(1 for i in rows for d, t in zip(done[i], tight[i]) if t < d)
    dur = [[tight[i][g] - ev[i][GROUPS[g][1]] for i in rows] for g in range(4)]
    # union over a span inside the window (Gram issue of its third to its second-last chunk),
    # where every product in flight belongs to a traced chunk
    t0, t1 = ev[2][0], ev[TRACE_CHUNKS - 2][0]
    spans = [(max(ev[i][GROUPS[g][1]], t0), min(tight[i][g], t1)) for i in rows for g in range(4)]
    busy = _union([(a, b) for a, b in spans if b > a]) / ((t1 - t0) / period)
    return {"period": period, "busy": busy, "dur": dur, "late": late}


if __name__ == "__main__":
    main()
