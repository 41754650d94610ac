"""The committed DRAM-traffic summary against the planner and the kernel
sources (CPU): the 256K rows are the 8192-token capture scaled by the ratio
of main (query row, key) pairs the planner counts for the two shapes (reads)
and by the token ratio (writes), and `bench.py` finds a current row for
the dominant kernel."""
import os
import re

import pytest

import bench
from branch_attention_speculative_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILE = os.path.join(ROOT, "profiles", "dram_traffic.md")


def _tables():
    small, full = {}, {}
    for line in open(PROFILE):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) == 4 and re.fullmatch(r"\d+", cells[1] or ""):
            small[cells[0]] = (int(cells[1]), int(cells[2]))
        if len(cells) == 6 and cells[1] == "eagle3_ttt_d7_256k":
            full[cells[0]] = (cells[2], int(cells[3]), int(cells[4]))
    return small, full


@pytest.fixture(scope="module")
def api():
    from branch_attention_speculative_gb300 import api as A, build as B
    B.build()
    return A


def test_scaled_rows_follow_the_planner(api):
    small, full = _tables()
    assert set(small) == set(full) == {"main_fwd", "main_bwd_kv", "main_bwd_dq"}
    wl = W.config(5)
    pairs_full = api.Plan.from_workload(wl).info()["main_pairs"]
    pairs_small = api.Plan.from_workload(bench.resize_workload(wl, 8192)).info()["main_pairs"]
    ratio = pairs_full / pairs_small
    for k, (rd, wr) in small.items():
        _, frd, fwr = full[k]
        assert abs(frd - rd * ratio) <= 1.0, k
        assert fwr == wr * (wl.tokens // 8192), k


def test_dominant_kernel_row_is_current():
    # the dK/dV kernel is the one bench.py reports traffic for
    t = bench.measured_traffic("main_bwd_kv", "eagle3_ttt_d7_256k")
    assert t is not None, "profiles/dram_traffic.md predates the dK/dV kernel source"
    _, full = _tables()
    _, rd, wr = full["main_bwd_kv"]
    assert t == rd + wr
