"""Host-side logic of bench.py (no GPU): the traffic figure it reads from the committed
ncu summary, the weak-scaling throughput, the algorithmic byte count of the decode
workload, and the parsing of the clock sampler's output (fed a canned nvidia-smi log)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import workloads as W  # noqa: E402


def test_traffic_comes_from_the_committed_profile():
    text = open(os.path.join(ROOT, "profiles", "index_score_kernel.decode.md")).read()
    line = [ln for ln in text.splitlines() if ln.startswith("dram_bytes_per_launch:")][0]
    assert bench.traffic_from_profile("decode") == float(line.split(":")[1])
    assert bench.traffic_from_profile("no_such_workload") is None


def test_weak_value_counts_every_rank():
    # 64 queries per rank, 2 ranks, 10 steps in 5 ms
    assert bench.weak_value(64, 2, 10, 5.0) == 64 * 2 * 10 / 0.005


def test_decode_index_bytes_are_the_visible_rows_plus_the_queries():
    wl = W.decode_batch()
    total, index, attn = bench.algorithmic_bytes(wl)
    rows = sum((int(p) + 1) // wl.ratio for p in wl.q_pos)
    per_query = wl.H * 128 * 2 + wl.H * 4 + wl.k * 4  # iq (bf16), w (fp32), sel (int32)
    assert index == rows * 256 + wl.Q * per_query
    assert total > index + attn  # the compressor's bytes come on top
    # every query attends to at most 512 selected rows and a 128-row window of 1 KiB
    assert attn <= wl.Q * ((512 + 128) * 1024 + 64 * 512 * 4 + 512 * 4 + 64)


class _FakeProc:
    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def test_clock_sampler_parsing():
    lines = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1300.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2055, 2070, 1100.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    c = bench.Clocks(0)
    c.proc = _FakeProc("\n".join(lines) + "\n")
    r = c.stop()
    assert r["sm_mhz"] == float(np.median([2070, 1980, 2055]))
    assert r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]
    assert r["samples"] == 3
    c2 = bench.Clocks(0)
    assert c2.stop() is None  # never started
