"""CPU tests of the benchmark's host logic: the multi-rank timing reduction
(world_size 2 over gloo), the clock-sample summary, and the reference arm's
JSON line (the fp64 oracle timed on host cores)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    r = bench.Ranks("gloo")
    r.barrier()
    mx = r.max(1.5 + rank)            # each rank "measured" a different step time
    q.put((rank, mx, r.world))
    r.close()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(res) == [(0, 2.5, 2), (1, 2.5, 2)]


def test_single_process_needs_no_process_group():
    r = bench.Ranks("gloo")
    assert r.world == 1 and r.max(3.0) == 3.0
    r.barrier()


def test_clock_summary():
    lines = "\n".join([
        "0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active, 99",
        "0, 1920, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active, 100",
        "0, 2070, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active, 0",
        "0, 1950, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active, 97",
    ])
    c = bench.parse_clock_lines(lines)
    assert c["sm_mhz"] == 1950 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3


def test_algorithmic_bytes():
    # 1538 bytes per token-head plus one fp32 state per (sequence, head)
    assert bench.BYTES_PER_TOKEN_HEAD == 1538
    assert bench.prefill_bytes(32768, 32, 4) == 32768 * 32 * 1538 + 4 * 32 * 128 * 128 * 4
    assert bench.decode_bytes(256, 32) == 256 * 32 * (2 * 65536 + 1024 + 512 + 2)


@pytest.mark.slow
def test_reference_arm_prints_one_json_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
           "--warmup", "3", "--ref-step-budget", "0.3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_multi_token_decode_roofs():
    import bench
    # one token: the plain decode kernel; the state traffic dominates, the line is HBM-bound
    e1 = bench._multi_decode_entry(1, 160e-6, 1, 6767.4)
    assert e1["bound"] == "hbm" and e1["frac"] == e1["frac_hbm"]
    assert e1["algorithmic_bytes_per_launch"] == bench.decode_bytes(bench.DEC_N, bench.H)
    assert e1["kernels"] == ["decode_kernel"]
    # several tokens: the chunk form; its state products (W S0, Q_g S0, Kb^T Delta: 6 T D^2 flop
    # per head) are tensor-core work, HBM stays the bound
    e16 = bench._multi_decode_entry(16, 500e-6, 1, 6767.4)
    assert e16["bound"] == "hbm" and e16["kernels"] == ["decode_chunk_kernel"]
    assert e16["tensor_flops_per_launch"] == bench.DEC_N * bench.H * 6 * 16 * bench.D * bench.D
    # the token-by-token flops for comparison: decay D^2 + three D^2 multiply-adds per token-head
    assert bench.DECODE_FLOP_PER_TOKEN_HEAD == 7 * bench.D * bench.D
    assert e16["token_loop_flops_per_launch"] == bench.DEC_N * 16 * bench.H * 7 * bench.D * bench.D
    nbytes = bench.decode_bytes(bench.DEC_N, bench.H, 16)
    assert abs(e16["frac"] - nbytes / (6767.4e9 * 500e-6)) < 1e-12
