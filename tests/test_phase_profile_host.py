"""Host-side checks of the prefill kernel's cycle-profile tool (no GPU)."""
import os
import re

from linear_attention_06_gb300 import phase_profile as pp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "linear_attention_06_gb300", "csrc", "kda_chunk_tc.cu")


def test_union_of_intervals():
    assert pp._union([]) == 0
    assert pp._union([(0, 5), (3, 8), (10, 12), (11, 11)]) == 10
    assert pp._union([(4, 6), (0, 10)]) == 10          # nested, unsorted


def test_chunk_arithmetic_matches_the_chunkwise_flop_count():
    # the products of one 64-token chunk at dk = dv = 128, written out from their shapes:
    # Gram 2*128*64*128, W' and U 2 * 2*128*64*64, Delta 2*128*64*128,
    # O 2*128*64*128 + 2*128*64*64, state 2*128*128*64
    C, d = 64, 128
    expect = (2 * 2 * C * C * d            # [A; P]: 128 rows (K-hat and Q-hat) x 64 x d
              + 2 * 2 * d * C * C          # W'^T and U^T
              + 2 * d * C * d              # Delta^T
              + 2 * d * C * d + 2 * d * C * C   # O^T
              + 2 * d * d * C)             # S^T update
    assert sum(g[3] for g in pp.GROUPS) == expect == 11534336


def test_trace_window_matches_the_kernel():
    src = open(SRC).read()
    m = re.search(r"kTraceChunks = (\d+), kTraceEvents = (\d+)", src)
    assert m, "trace window constants not found in the kernel source"
    assert tuple(int(v) for v in m.groups()) == (pp.TRACE_CHUNKS, pp.TRACE_EVENTS)
    assert "kda_debug_set_trace_first" in src
    # every window fits the benchmark's 128 chunks per sequence
    assert all(0 <= f and f + pp.TRACE_CHUNKS <= 128 for f in pp.TRACE_WINDOWS)
    # every issue event the tool reads is stamped in the kernel
    for _, issue, done, _ in pp.GROUPS:
        assert re.search(rf"KDA_TRACE\([^,]+, {issue}\);", src), issue
        assert done == issue + 1


def test_phase_slots_are_stamped_in_the_kernel():
    src = open(SRC).read()
    stamped = {int(v) for v in re.findall(r"KDA_PHASE\((\d+)\)", src)}
    assert set(pp.PHASES) <= stamped
