#!/usr/bin/env python
"""KDA on GB300: prefill tokens/s (H=32, d=128) and decode-step HBM GB/s.

One step = one KDA prefill pass (kda_prefill, C ABI) over the bf16 workload
B=4, H=32, T=8192, dk=dv=128 (q, k, v, beta bf16; log_alpha fp32; zero initial
state; final states returned), inputs resident in HBM.  The decode step
(kda_decode_step, 256 sequences x H=32, fp32 state in place) is timed in the
same run and reported under "decode".  Inputs are larger than L2 (1.6 GB and
1.1 GB), so no flush is needed between iterations.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (one process per GPU, launched by torch.distributed.run) every rank
runs its own batch (weak scaling, no data-path collective); timing is the max
over ranks.  --impl reference times the fp64 CPU oracle on a bounded sample of
the same workload (host cores) and prints the same JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (H=32,d=128) + decode-step HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
WORKLOAD = "kda_prefill_bf16_B4_H32_T8192_d128"
B, T, H, D = 4, 8192, 32, 128
DEC_N = 256
CKPT_EVERY = 1024          # checkpointed prefill: a state every 1024 tokens of each sequence
DEC_MULTI_T = (4, 16)      # multi-token decode: tokens per sequence per call
# algorithmic bytes per token-head: q, k, v bf16 (768) + log_alpha fp32 (512) + beta (2) + out (256)
BYTES_PER_TOKEN_HEAD = 3 * D * 2 + D * 4 + 2 + D * 2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def prefill_bytes(tokens, heads, num_seqs, with_h0=False):
    return tokens * heads * BYTES_PER_TOKEN_HEAD + num_seqs * heads * D * D * 4 * (2 if with_h0 else 1)


def frontend_bytes(tokens, heads, d=128, width=4):
    """Front end, bf16 (d = dk = dv): raw q, k, v read and q, k, v written (2 B each),
    decay logits read and log_alpha written (4 B), beta logits and beta (2 B), plus the
    fp32 convolution taps."""
    per = 3 * d * 2 * 2 + d * 4 * 2 + 2 * 2
    return tokens * heads * per + 3 * heads * d * width * 4


# decode arithmetic per token-head (dk = dv = D): decay D*D multiplies, r = S^T k, y = S^T q and
# the rank-1 update D*D fused multiply-adds each (2 flop)
DECODE_FLOP_PER_TOKEN_HEAD = D * D + 3 * 2 * D * D


def decode_bytes(n, heads, tokens=1):
    # state read + write (fp32) once, + per token q, k, v, out bf16 + log_alpha fp32 + beta bf16
    return n * heads * (2 * D * D * 4 + tokens * (4 * D * 2 + D * 4 + 2))


def _multi_decode_entry(tm, t_m, world, hbm):
    """One multi-token decode line.  Steps of 2..16 tokens at d = 128 run the chunk form: its
    three state products are TF32 tensor-core work far below the tensor roof, so HBM is the
    bound; the fp32 CUDA-core flops of the token-by-token form are kept for comparison."""
    nbytes = decode_bytes(DEC_N, H, tm)
    flops = DEC_N * tm * H * DECODE_FLOP_PER_TOKEN_HEAD
    t_hbm = nbytes / (hbm * 1e9)
    return {"workload": f"kda_decode_N{DEC_N}_H{H}_d{D}_T{tm}", "tokens_per_seq": tm,
            "us_per_step": t_m * 1e6, "value": world * DEC_N * tm / t_m, "unit": UNIT,
            "achieved_gbs": nbytes / t_m / 1e9, "frac_hbm": t_hbm / t_m, "bound": "hbm", "frac": t_hbm / t_m,
            "token_loop_flops_per_launch": flops, "tensor_flops_per_launch": DEC_N * H * 6 * tm * D * D,
            "algorithmic_bytes_per_launch": nbytes,
            "kernels": ["decode_chunk_kernel" if tm > 1 else "decode_kernel"]}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU works."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_lines(out)


def parse_clock_lines(out):
    """Summarise nvidia-smi CSV samples: median SM clock under load, max clock,
    and every throttle reason seen active."""
    rows = []
    for line in out.strip().splitlines():
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), hw=parts[5],
                             hwt=parts[6], swt=parts[7], pcap=parts[8],
                             util=float(parts[9]) if parts[9] not in ("", "[N/A]") else 0.0))
        except ValueError:
            continue
    busy = [r for r in rows if r["util"] > 0] or rows
    if not busy:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    sms = sorted(r["sm"] for r in busy)
    reasons = set()
    for r in busy:
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                          ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
            if r[key].lower() == "active":
                reasons.add(name)
    return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(r["smax"] for r in busy),
            "reasons": sorted(reasons), "samples": len(busy)}


def source_digest():
    """Digest of the prefill kernel source; a stored ncu traffic figure is used
    only while it matches the kernel that is running."""
    import hashlib
    h = hashlib.sha256()
    for f in ("kda_chunk_tc.cu", "kda_chunk_common.cuh", "sm103_primitives.cuh"):
        with open(os.path.join(ROOT, "linear_attention_06_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel_digest):
    p = os.path.join(ROOT, "profiles", "ncu_traffic_chunk_tc_prefill.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_digest") != kernel_digest:
        return None
    return d.get("dram_bytes_per_launch_full_workload")


def oracle_sample(budget_s, threads=0):
    """Time the fp64 oracle on a bounded sample of the prefill workload: as many of
    its B sequences (all H heads each) as fit the time budget on the host cores."""
    import numpy as np
    from linear_attention_06_gb300 import workloads
    from oracle import kda_oracle
    cores = os.cpu_count() or 1
    used = kda_oracle.max_threads() if threads == 0 else threads

    def inputs(nseq):
        w = workloads.make_inputs(nseq * T, H, D, D, seed=1, num_seqs=nseq)   # same recipe
        return [np.ascontiguousarray(x.float().numpy().astype(np.float64))
                for x in (w.q, w.k, w.v, w.log_alpha, w.beta)]

    one = inputs(1)
    t0 = time.perf_counter()
    kda_oracle.prefill(*[a[:, :1].copy() for a in one], None, cu_seqlens=[0, T], num_threads=1)
    t1 = time.perf_counter() - t0                  # one (sequence, head) pair on one thread
    pairs = budget_s / max(t1, 1e-6) * max(1, min(used, B * H))
    nseq = int(max(1, min(B, pairs // H)))
    arr = one if nseq == 1 else inputs(nseq)
    cu = [i * T for i in range(nseq + 1)]

    def run():
        t0 = time.perf_counter()
        kda_oracle.prefill(*arr, None, cu_seqlens=cu, num_threads=used)
        return time.perf_counter() - t0

    return run, nseq, cores, used


def gpu_numa_node(dev_index):
    """NUMA node of the host memory nearest the GPU (its PCI function's node), or None."""
    import torch
    try:
        p = torch.cuda.get_device_properties(dev_index)
        bus = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            node = int(f.read().strip())
        return node if node >= 0 else None
    except (AttributeError, OSError, ValueError):
        return None


def node_cpus(node):
    """CPU ids of a NUMA node from sysfs ("0-3,8-11" ranges), or None."""
    try:
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            text = f.read().strip()
    except OSError:
        return None
    cpus = set()
    for part in text.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return cpus or None


class Ranks:
    """Process-group plumbing for N > 1: barrier and max over ranks.  Works with
    nccl (GPU tensors) or gloo (CPU tensors); a single process needs neither."""

    def __init__(self, backend=None, device=None):
        import torch.distributed as dist
        self.dist = dist
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.device = device
        if self.world > 1 and not dist.is_initialized():
            kw = {"device_id": device} if backend == "nccl" else {}
            dist.init_process_group(backend or "gloo", **kw)

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max(self, x):
        if self.world == 1:
            return x
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1 and self.dist.is_initialized():
            self.dist.destroy_process_group()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    budget = max(1.0, args.ref_step_budget)
    run, nseq, cores, used = oracle_sample(budget)
    for _ in range(args.warmup):
        run()
    t = sum(run() for _ in range(args.steps)) / args.steps
    value = nseq * T / t                           # tokens (all H heads each) per second
    sample = f"fp64 oracle, {nseq} of {B} sequences x {H} heads x {T} tokens per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": B, "seq_len": T, "heads": H,
                       "head_dim": D, "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch

    import linear_attention_06_gb300 as kda
    from linear_attention_06_gb300 import workloads

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ranks = Ranks("nccl", dev)
    world, rank = ranks.world, ranks.rank
    barrier, max_over_ranks = ranks.barrier, ranks.max

    stream = torch.cuda.current_stream()
    w = workloads.prefill_bf16(device=dev, seed=1 + rank)
    cu = w.cu_seqlens.to(dev)
    out = torch.empty_like(w.v)
    fin = torch.empty((B, H, D, D), dtype=torch.float32, device=dev)

    def prefill_step():
        kda.kda_prefill(w.q, w.k, w.v, w.log_alpha, w.beta, None, cu, out, fin, stream=stream)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        prefill_step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        prefill_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_prefill = max_over_ranks(ev0.elapsed_time(ev1) * 1e-3 / args.steps)
    prefill_launches = args.steps                 # one kernel launch per prefill step

    # ---- decode step (256 sequences x 32 heads), state updated in place
    dw = workloads.decode_inputs(device=dev, seed=2 + rank)
    S = dw.initial_state.clone()
    dout = torch.empty_like(dw.v)

    def decode_step():
        kda.kda_decode_step(dw.q, dw.k, dw.v, dw.log_alpha, dw.beta, S, dout, stream=stream)

    for _ in range(args.warmup):
        decode_step()
    torch.cuda.synchronize()
    barrier()
    ev0.record(stream)
    for _ in range(args.steps):
        decode_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_decode = max_over_ranks(ev0.elapsed_time(ev1) * 1e-3 / args.steps)

    # ---- the layer steps around the recurrence, on the same workload shapes
    layer = None
    if not args.no_layer:
        def timed(fn):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            barrier()
            ev0.record(stream)
            for _ in range(args.steps):
                fn()
            ev1.record(stream)
            torch.cuda.synchronize()
            barrier()
            return max_over_ranks(ev0.elapsed_time(ev1) * 1e-3 / args.steps)

        lx = workloads.make_layer_inputs(B * T, H, D, D, W=4, dtype=torch.bfloat16, seed=11 + rank,
                                         num_seqs=B, device=dev)
        fe_out = tuple(torch.empty_like(t) for t in (w.q, w.k, w.v, w.log_alpha, w.beta))
        t_fe = timed(lambda: kda.kda_frontend(lx.q_raw, lx.k_raw, lx.v_raw, lx.a_raw, lx.b_raw, lx.conv_q,
                                              lx.conv_k, lx.conv_v, num_seqs=B, out=fe_out, stream=stream))
        t_pg = timed(lambda: kda.kda_prefill_gated(w.q, w.k, w.v, w.log_alpha, w.beta, lx.g_raw, lx.norm_weight,
                                                   cu_seqlens=cu, out=out, final_state=fin, stream=stream))
        # the front end fused into the prefill: raw projections in, out and final states out
        t_pf = timed(lambda: kda.kda_prefill_frontend(lx.q_raw, lx.k_raw, lx.v_raw, lx.a_raw, lx.b_raw, lx.conv_q,
                                                      lx.conv_k, lx.conv_v, cu_seqlens=cu, out=out, final_state=fin,
                                                      stream=stream))
        gx = workloads.make_layer_inputs(DEC_N, H, D, D, dtype=torch.bfloat16, seed=12 + rank,
                                         cu_seqlens=list(range(DEC_N + 1)), device=dev)
        t_dg = timed(lambda: kda.kda_decode_step_gated(dw.q, dw.k, dw.v, dw.log_alpha, dw.beta, gx.g_raw,
                                                       gx.norm_weight, S, out=dout, stream=stream))
        layer = {"t_fe": t_fe, "t_pg": t_pg, "t_dg": t_dg, "t_pf": t_pf}

        # NEXT-1: the benchmark prefill also saving every sequence's state each CKPT_EVERY
        # tokens.  The checkpoint tables go to the device once (the binding would validate
        # and copy them on every call), and the call goes straight through the C ABI.
        import ctypes

        from linear_attention_06_gb300 import _lib
        L = _lib.lib()
        per_seq = T // CKPT_EVERY
        ck_cu_h = torch.arange(0, B * per_seq + 1, per_seq, dtype=torch.int32)
        ck_pos_h = torch.tensor([p for _ in range(B) for p in range(CKPT_EVERY, T + 1, CKPT_EVERY)],
                                dtype=torch.int32)
        cu_h = w.cu_seqlens.to(torch.int32).cpu()
        st = L.kda_check_checkpoints(ctypes.c_void_p(cu_h.data_ptr()), B, B * T,
                                     ctypes.c_void_p(ck_cu_h.data_ptr()), ctypes.c_void_p(ck_pos_h.data_ptr()))
        _lib._check("kda_check_checkpoints", st)
        ck_cu, ck_pos = ck_cu_h.to(dev), ck_pos_h.to(dev)
        ck_states = torch.empty((B * per_seq, H, D, D), dtype=torch.float32, device=dev)
        ck_shape = _lib.KdaShape(B, B * T, H, D, D, _lib.KDA_BF16)

        def ckpt_step():
            rc = L.kda_prefill_checkpointed(ctypes.byref(ck_shape), _lib._ptr(w.q), _lib._ptr(w.k), _lib._ptr(w.v),
                                            _lib._ptr(w.log_alpha), _lib._ptr(w.beta), None, _lib._ptr(cu),
                                            _lib._ptr(out), _lib._ptr(fin), _lib._ptr(ck_cu), _lib._ptr(ck_pos),
                                            _lib._ptr(ck_states), _lib._stream(stream))
            _lib._check("kda_prefill_checkpointed", rc)

        layer["t_ck"] = timed(ckpt_step)
        layer["n_ck"] = B * per_seq

        # NEXT-4: decode steps of several tokens per sequence (state read and written once)
        layer["multi"] = {}
        for tm in DEC_MULTI_T:
            mw = workloads.make_inputs(DEC_N * tm, H, D, D, dtype=torch.bfloat16, seed=13 + tm + rank,
                                       cu_seqlens=[tm * i for i in range(DEC_N + 1)], state_std=0.05, device=dev)
            ms_state = mw.initial_state.clone()
            m_out = torch.empty_like(mw.v)
            layer["multi"][tm] = timed(lambda: kda.kda_decode_step(mw.q, mw.k, mw.v, mw.log_alpha, mw.beta,
                                                                   ms_state, m_out, stream=stream))
            del mw, ms_state, m_out

        # the other prefill workloads: one 131072-token sequence (whole, and resumed from the
        # state after its first half), and 64 log-uniform lengths packed with per-sequence
        # initial states (load imbalance: the longest sequence sets the time)
        lw = workloads.long_prefill(device=dev, seed=3 + rank)
        Tl = lw.q.shape[0]
        l_out = torch.empty_like(lw.v)
        l_fin = torch.empty((1, H, D, D), dtype=torch.float32, device=dev)
        half = Tl // 2
        l_mid = torch.empty((1, H, D, D), dtype=torch.float32, device=dev)
        layer["t_long"] = timed(lambda: kda.kda_prefill(lw.q, lw.k, lw.v, lw.log_alpha, lw.beta, None, None,
                                                        l_out, l_fin, num_seqs=1, stream=stream))

        def resume_step():
            kda.kda_prefill(lw.q[:half], lw.k[:half], lw.v[:half], lw.log_alpha[:half], lw.beta[:half], None,
                            None, l_out[:half], l_mid, num_seqs=1, stream=stream)
            kda.kda_prefill(lw.q[half:], lw.k[half:], lw.v[half:], lw.log_alpha[half:], lw.beta[half:], l_mid,
                            None, l_out[half:], l_fin, num_seqs=1, stream=stream)

        layer["t_resume"] = timed(resume_step)
        # the same sequence through the split prefill (chunk-local kernel over all chunks of all
        # heads, then the state chain per head); its workspace is allocated once, outside the timing
        l_ws = torch.empty(kda.kda_prefill_split_workspace_size(Tl, 1, H), dtype=torch.uint8, device=dev)
        layer["t_long_split"] = timed(lambda: kda.kda_prefill_split(lw.q, lw.k, lw.v, lw.log_alpha, lw.beta, None,
                                                                    None, l_out, l_fin, num_seqs=1, workspace=l_ws,
                                                                    stream=stream))
        layer["long_split_ws"] = l_ws.numel()
        layer["long_tokens"] = Tl
        del lw, l_out, l_ws
        vw = workloads.varlen_prefill(device=dev, seed=4 + rank)
        v_cu = vw.cu_seqlens.to(dev)
        v_out = torch.empty_like(vw.v)
        v_fin = torch.empty_like(vw.initial_state)
        layer["t_varlen"] = timed(lambda: kda.kda_prefill(vw.q, vw.k, vw.v, vw.log_alpha, vw.beta, vw.initial_state,
                                                          v_cu, v_out, v_fin, stream=stream))
        layer["varlen_tokens"] = vw.q.shape[0]
        layer["varlen_seqs"] = v_cu.numel() - 1
        layer["varlen_longest"] = int((v_cu[1:] - v_cu[:-1]).max().item())
        del vw, v_out, v_fin
    clocks = sampler.stop()

    # ---- end to end through the public API with host buffers (pinned).  Every step copies
    # its inputs host->device, runs kda_prefill and copies out and the final states back;
    # copies in, compute and copies out run on three streams with two device buffer sets,
    # so step i's kernel overlaps step i+1's input copy and step i-1's output copy.
    e2e = None
    if not args.no_e2e:
        keys = ("q", "k", "v", "log_alpha", "beta")
        # the pinned host buffers are first touched by a thread on the GPU's NUMA node, so their
        # pages live in the host memory nearest the GPU; the affinity is restored afterwards
        numa = gpu_numa_node(dev.index if dev.index is not None else 0)
        cpus = node_cpus(numa) if numa is not None else None
        old_aff = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
        if cpus and old_aff is not None and cpus & old_aff:
            os.sched_setaffinity(0, cpus & old_aff)
        host = {k: getattr(w, k).cpu().pin_memory() for k in keys}
        hout = [torch.empty(out.shape, dtype=out.dtype).pin_memory().zero_() for _ in range(2)]
        hfin = [torch.empty(fin.shape, dtype=fin.dtype).pin_memory().zero_() for _ in range(2)]
        if old_aff is not None:
            os.sched_setaffinity(0, old_aff)
        dbuf = [{k: torch.empty_like(getattr(w, k)) for k in keys} for _ in range(2)]
        obuf = [(torch.empty_like(out), torch.empty_like(fin)) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = hout[0].numel() * hout[0].element_size() + hfin[0].numel() * hfin[0].element_size()
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()
        in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        in_free = [ev(), ev()]                    # compute has read buffer set b
        for b in range(2):
            in_free[b].record(stream)
            out_done[b].record(stream)

        def e2e_step(i):
            b = i & 1
            s_in.wait_event(in_free[b])
            with torch.cuda.stream(s_in):
                for k in keys:
                    dbuf[b][k].copy_(host[k], non_blocking=True)
            in_done[b].record(s_in)
            stream.wait_event(in_done[b])
            stream.wait_event(out_done[b])        # the previous use of this output set was copied out
            d = dbuf[b]
            kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], None, cu, obuf[b][0],
                            obuf[b][1], stream=stream)
            comp_done[b].record(stream)
            in_free[b].record(stream)
            s_out.wait_event(comp_done[b])
            with torch.cuda.stream(s_out):
                hout[b].copy_(obuf[b][0], non_blocking=True)
                hfin[b].copy_(obuf[b][1], non_blocking=True)
            out_done[b].record(s_out)

        for i in range(max(2, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        ev0.record(stream)
        s_in.wait_event(ev0)                      # no copy of the timed steps starts before ev0
        s_out.wait_event(ev0)
        for i in range(args.steps):
            e2e_step(i)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)                 # ev1 after the last copy out
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        t_e2e = max_over_ranks(ev0.elapsed_time(ev1) * 1e-3 / args.steps)

        # each leg alone (same pinned buffers, one stream at a time): the pipelined step can be
        # no faster than the slowest of the three.  Best of three trials: a host-side hiccup in
        # one trial would otherwise make the bound look slower than the pipelined step itself.
        def alone(s, fn, reps=5, trials=3):
            best = float("inf")
            with torch.cuda.stream(s):
                fn()
                torch.cuda.synchronize()
                for _ in range(trials):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(s)
                    for _ in range(reps):
                        fn()
                    b.record(s)
                    torch.cuda.synchronize()
                    best = min(best, a.elapsed_time(b) * 1e-3 / reps)
            return best

        def copy_in():
            for k in keys:
                dbuf[0][k].copy_(host[k], non_blocking=True)

        def copy_out():
            hout[0].copy_(obuf[0][0], non_blocking=True)
            hfin[0].copy_(obuf[0][1], non_blocking=True)

        t_in, t_out = alone(s_in, copy_in), alone(s_out, copy_out)
        bound = max(t_in, t_out, t_prefill)
        e2e = {"value": world * B * T / t_e2e, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3,
               "copy_in_ms": t_in * 1e3, "kernel_ms": t_prefill * 1e3, "copy_out_ms": t_out * 1e3,
               "h2d_gbs_alone": h2d / t_in / 1e9, "d2h_gbs_alone": d2h / t_out / 1e9,
               "slowest_leg_ms": bound * 1e3, "ms_over_slowest_leg": t_e2e / bound,
               "host_numa_node": numa,
               "pipelining": "copy-in / compute / copy-out on three streams, two buffer sets"}

    if rank != 0:
        ranks.close()
        return

    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    pbytes = prefill_bytes(B * T, H, B)
    achieved = pbytes / t_prefill / 1e9
    digest = source_digest()
    dbytes = decode_bytes(DEC_N, H)
    dec_gbs = dbytes / t_decode / 1e9
    line = {
        "metric": METRIC, "value": world * B * T / t_prefill, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_prefill * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world * B, "seq_len": T, "heads": H,
                   "head_dim": D, "chunk": 64, "initial_state": "zeros", "final_state": "returned",
                   "parallelism": f"replicas x{world}", "l2": "inputs larger than L2 (no flush)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": stored_traffic(digest),
                     "peak_source": f"{peak_kind} hbm_gbs", "kernel": "chunk_tc_kernel",
                     "algorithmic_bytes_per_launch": pbytes, "source_digest": digest},
        "decode": {"workload": f"kda_decode_N{DEC_N}_H{H}_d{D}", "us_per_step": t_decode * 1e6,
                   "achieved_gbs": dec_gbs, "peak_gbs": hbm, "frac": dec_gbs / hbm,
                   "algorithmic_bytes_per_launch": dbytes, "kernel": "decode_kernel"},
        "e2e": e2e, "gpu_launches": prefill_launches, "clocks": clocks,
    }
    if layer is not None:
        fbytes = frontend_bytes(B * T, H)
        gbytes = pbytes + B * T * H * D * 2                  # + the bf16 gate read once
        dgbytes = dbytes + DEC_N * H * D * 2
        line["layer"] = {
            "frontend": {"workload": f"kda_frontend_bf16_B{B}_H{H}_T{T}_d{D}_W4",
                         "us_per_step": layer["t_fe"] * 1e6, "achieved_gbs": fbytes / layer["t_fe"] / 1e9,
                         "peak_gbs": hbm, "frac": fbytes / layer["t_fe"] / 1e9 / hbm,
                         "algorithmic_bytes_per_launch": fbytes, "kernels": ["conv_kernel", "gate_kernel"]},
            "prefill_frontend": {"workload": WORKLOAD + "_frontend_W4",
                                 "ms_per_step": layer["t_pf"] * 1e3, "value": world * B * T / layer["t_pf"],
                                 "unit": UNIT, "achieved_gbs": pbytes / layer["t_pf"] / 1e9,
                                 "frac": pbytes / layer["t_pf"] / 1e9 / hbm, "algorithmic_bytes_per_launch": pbytes,
                                 "two_pass_ms": (layer["t_fe"] + t_prefill) * 1e3,
                                 "kernels": ["chunk_tc_kernel (front end in team P)"],
                                 "note": "kda_prefill_frontend: raw projections in (the same bytes as the prefill's "
                                         "inputs), the front end run on each chunk's tiles in shared memory; "
                                         "two_pass_ms = kda_frontend + kda_prefill"},
            "prefill_gated": {"workload": WORKLOAD + "_gated", "ms_per_step": layer["t_pg"] * 1e3,
                              "value": world * B * T / layer["t_pg"], "unit": UNIT,
                              "achieved_gbs": gbytes / layer["t_pg"] / 1e9,
                              "frac": gbytes / layer["t_pg"] / 1e9 / hbm,
                              "algorithmic_bytes_per_launch": gbytes, "kernels": ["chunk_tc_kernel", "gated_norm_bf16_128"]},
            "decode_gated": {"workload": f"kda_decode_N{DEC_N}_H{H}_d{D}_gated",
                             "us_per_step": layer["t_dg"] * 1e6, "achieved_gbs": dgbytes / layer["t_dg"] / 1e9,
                             "frac": dgbytes / layer["t_dg"] / 1e9 / hbm,
                             "algorithmic_bytes_per_launch": dgbytes, "kernels": ["decode_kernel (gate and norm in its store)"]},
        }
        ckbytes = pbytes + layer["n_ck"] * H * D * D * 4        # + every checkpoint state written once
        lt, nv = layer["long_tokens"], layer["varlen_seqs"]
        lbytes = prefill_bytes(lt, H, 1)
        vbytes = prefill_bytes(layer["varlen_tokens"], H, nv, with_h0=True)
        line["other_prefill_configs"] = {
            "long_prefill": {"workload": f"kda_prefill_bf16_B1_H{H}_T{lt}_d{D}", "ms_per_step": layer["t_long"] * 1e3,
                             "value": world * lt / layer["t_long"], "unit": UNIT,
                             "achieved_gbs": lbytes / layer["t_long"] / 1e9,
                             "frac": lbytes / layer["t_long"] / 1e9 / hbm, "algorithmic_bytes_per_launch": lbytes,
                             "note": f"{H} blocks (one per head) on {lt // 64} chunks each: one block per SM"},
            "long_prefill_split": {"workload": f"kda_prefill_bf16_B1_H{H}_T{lt}_d{D}_split",
                                   "ms_per_step": layer["t_long_split"] * 1e3,
                                   "value": world * lt / layer["t_long_split"], "unit": UNIT,
                                   "achieved_gbs": lbytes / layer["t_long_split"] / 1e9,
                                   "frac": lbytes / layer["t_long_split"] / 1e9 / hbm,
                                   "algorithmic_bytes_per_launch": lbytes,
                                   "workspace_bytes": layer["long_split_ws"],
                                   "kernels": ["chunk_local_kernel", "chunk_chain_kernel"],
                                   "note": "kda_prefill_split: the sequence in 8192-token segments; each segment's "
                                           "per-chunk records of every head (on the SMs the chains leave free, "
                                           "overlapping the previous segment's chains), then one state chain per "
                                           "head carrying the fp32 state on; bytes counted as for the fused kernel "
                                           "(the records' round trip through HBM is not in the algorithmic bytes)"},
            "long_prefill_resumed": {"workload": f"kda_prefill_bf16_B1_H{H}_T{lt}_d{D}_resume_at_{lt // 2}",
                                     "ms_per_step": layer["t_resume"] * 1e3,
                                     "value": world * lt / layer["t_resume"], "unit": UNIT,
                                     "note": "two calls: the first half, then the second half from its final state"},
            "varlen": {"workload": f"kda_prefill_bf16_varlen_N{nv}_H{H}_d{D}", "tokens": layer["varlen_tokens"],
                       "longest_sequence": layer["varlen_longest"], "ms_per_step": layer["t_varlen"] * 1e3,
                       "value": world * layer["varlen_tokens"] / layer["t_varlen"], "unit": UNIT,
                       "achieved_gbs": vbytes / layer["t_varlen"] / 1e9,
                       "frac": vbytes / layer["t_varlen"] / 1e9 / hbm, "algorithmic_bytes_per_launch": vbytes},
        }
        line["next"] = {
            "prefill_checkpointed": {"workload": WORKLOAD + f"_ckpt{CKPT_EVERY}", "checkpoints": layer["n_ck"],
                                     "ms_per_step": layer["t_ck"] * 1e3, "value": world * B * T / layer["t_ck"],
                                     "unit": UNIT, "achieved_gbs": ckbytes / layer["t_ck"] / 1e9,
                                     "frac": ckbytes / layer["t_ck"] / 1e9 / hbm,
                                     "algorithmic_bytes_per_launch": ckbytes, "kernels": ["chunk_tc_kernel"]},
            "decode_multi_token": [_multi_decode_entry(tm, t_m, world, hbm) for tm, t_m in layer["multi"].items()],
        }
    if world == 1 and not args.no_cpu_baseline:
        run, nseq, cores, used = oracle_sample(args.cpu_budget)
        t = run()
        line["cpu_baseline"] = {"value": nseq * T / t, "unit": UNIT, "cores": used,
                                "kind": "oracle",
                                "sample": f"fp64 oracle on {nseq} of {B} sequences x {H} heads x {T} tokens "
                                          f"({t:.1f} s, {cores} host cores)"}
    print(json.dumps(line), flush=True)
    ranks.close()


PROFILE_CASES = ("prefill", "decode_chunk_T16", "decode_chunk_T4", "split_T32768", "frontend", "prefill_gated")


def run_profile_case(name):
    """Three calls of one kernel family on its bench workload (or, for the split prefill, a
    32768-token sequence: inputs above L2, a few GB at most), for an ncu capture of one launch
    (-s 2 -c 1 after the two warm-up calls).  Prints one line."""
    import torch
    import linear_attention_06_gb300 as kda
    from linear_attention_06_gb300 import workloads
    dev = torch.device("cuda", 0)
    if name == "prefill":
        w = workloads.prefill_bf16(device=dev)
        out, fin = torch.empty_like(w.v), torch.empty((B, H, D, D), dtype=torch.float32, device=dev)
        cu = w.cu_seqlens.to(dev)
        call = lambda: kda.kda_prefill(w.q, w.k, w.v, w.log_alpha, w.beta, None, cu, out, fin)
    elif name.startswith("decode_chunk_T"):
        tm = int(name[len("decode_chunk_T"):])
        w = workloads.make_inputs(DEC_N * tm, H, D, D, dtype=torch.bfloat16, seed=13 + tm,
                                  cu_seqlens=[tm * i for i in range(DEC_N + 1)], state_std=0.05, device=dev)
        S, out = w.initial_state.clone(), torch.empty_like(w.v)
        call = lambda: kda.kda_decode_step(w.q, w.k, w.v, w.log_alpha, w.beta, S, out)
    elif name == "split_T32768":
        tl = 32768
        w = workloads.make_inputs(tl, H, D, D, dtype=torch.bfloat16, seed=3, cu_seqlens=[0, tl], device=dev)
        cu = torch.tensor([0, tl], dtype=torch.int32, device=dev)
        out, fin = torch.empty_like(w.v), torch.empty((1, H, D, D), dtype=torch.float32, device=dev)
        ws = torch.empty(kda.kda_prefill_split_workspace_size(tl, 1, H), dtype=torch.uint8, device=dev)
        call = lambda: kda.kda_prefill_split(w.q, w.k, w.v, w.log_alpha, w.beta, None, cu, out=out,
                                             final_state=fin, workspace=ws)
    elif name == "frontend":
        lx = workloads.make_layer_inputs(B * T, H, D, D, W=4, dtype=torch.bfloat16, seed=11, num_seqs=B, device=dev)
        w = workloads.prefill_bf16(device=dev)
        fe_out = tuple(torch.empty_like(t) for t in (w.q, w.k, w.v, w.log_alpha, w.beta))
        del w
        call = lambda: kda.kda_frontend(lx.q_raw, lx.k_raw, lx.v_raw, lx.a_raw, lx.b_raw, lx.conv_q, lx.conv_k,
                                        lx.conv_v, num_seqs=B, out=fe_out)
    elif name == "prefill_gated":
        w = workloads.prefill_bf16(device=dev)
        lx = workloads.make_layer_inputs(B * T, H, D, D, W=4, dtype=torch.bfloat16, seed=11, num_seqs=B, device=dev)
        out, fin = torch.empty_like(w.v), torch.empty((B, H, D, D), dtype=torch.float32, device=dev)
        cu = w.cu_seqlens.to(dev)
        call = lambda: kda.kda_prefill_gated(w.q, w.k, w.v, w.log_alpha, w.beta, lx.g_raw, lx.norm_weight,
                                             cu_seqlens=cu, out=out, final_state=fin)
    else:
        raise SystemExit(f"unknown profile case {name}")
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    print(f"profile case {name}: 3 calls", flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-layer", action="store_true", help="skip the front-end, gated-output, checkpointed-prefill and multi-token-decode timings")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-step-budget", type=float, default=4.0,
                    help="seconds of oracle work per step in --impl reference")
    ap.add_argument("--profile-case", choices=PROFILE_CASES,
                    help="only run three calls of one kernel family (for an ncu capture) and exit")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
