"""CPU tests of the split planner: its chunk rule is the library's (checked
by compiling the library's own host-callable rule into a small host
program), the rule's bounds, and the simulation's stated cost model."""
import math
import os
import shutil
import subprocess

import pytest

from speculative_decode_mla_paged_gb300 import tuning as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decode_mla_paged_gb300", "csrc")

NS = [1, 2, 127, 128, 255, 256, 257, 383, 1000, 5776, 23072, 92224, 185064]
SPLITS = [1, 2, 3, 7, 9, 14, 64, 255, 256]


def test_split_chunk_rule_bounds():
    for n in NS:
        for s in SPLITS:
            c, u = T.split_chunk(n, s), T.splits_used(n, s)
            assert c % 128 == 0 and c >= 256
            assert c >= -(-n // s)                       # S chunks cover the request
            assert c - 128 < max(-(-n // s), 256)        # and it is the smallest such multiple
            assert 1 <= u <= s and (u - 1) * c < n <= u * c
    assert T.splits_used(0, 8) == 0


def test_split_chunk_matches_the_library(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    prog = tmp_path / "chunks.cu"
    prog.write_text(
        '#include "va_internal.cuh"\n#include <cstdio>\n'
        "int main() {\n"
        f"  const long long ns[] = {{{', '.join(map(str, NS))}}};\n"
        f"  const int ss[] = {{{', '.join(map(str, SPLITS))}}};\n"
        "  for (long long n : ns) for (int s : ss)\n"
        '    std::printf("%lld %d %lld %lld\\n", n, s, (long long)va::split_chunk(n, s),'
        " (long long)va::splits_used(n, s));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "chunks"
    subprocess.run([nvcc, "-std=c++17", "-I", CSRC, "-I", os.path.join(ROOT, "include"), "-o", str(exe),
                    str(prog)], check=True, capture_output=True, timeout=300)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=60).stdout
    rows = [tuple(map(int, line.split())) for line in out.split("\n") if line.strip()]
    assert len(rows) == len(NS) * len(SPLITS)
    for n, s, c, u in rows:
        assert (c, u) == (T.split_chunk(n, s), T.splits_used(n, s)), (n, s)


def _combine_tiles(rows_splits):
    return rows_splits * 2048 * 2 / 6.8e12 / 2.5e-6


def test_one_unit_costs_its_tiles_plus_the_start_up():
    # T * H = 128 rows: the 2-CTA shape; one split: one unit of ceil(N / 128) tiles + 4
    est = T.simulate([1000], [16], 8, 1)
    assert est == pytest.approx(4 + math.ceil(1016 / 128) + _combine_tiles(16 * 8))


def test_units_beyond_the_resident_clusters_queue():
    # T * H = 256 rows: 36 four-CTA clusters at once.  A request of 36 * 256
    # keys at 36 splits is 36 units of two tiles (cost 6 each): one round;
    # two such requests take two rounds.
    one = T.simulate([9184], [32], 8, 36) - _combine_tiles(32 * 8 * 36)
    two = T.simulate([9184, 9184], [32, 32], 8, 36) - _combine_tiles(2 * 32 * 8 * 36)
    assert one == pytest.approx(6.0) and two == pytest.approx(12.0)


def test_plan_is_a_candidate_and_ranked_counts_are_distinct():
    prefix, drafts = [185000, 5000, 1200, 40000], [64, 16, 32, 16]
    cands = list(T._candidates(prefix, drafts))
    plan = T.plan_num_splits(prefix, drafts, 8)
    ranked = T.ranked_num_splits(prefix, drafts, 8, k=5)
    assert plan in cands and ranked[0] == plan
    assert len(ranked) == 5 == len(set(ranked)) and set(ranked) <= set(cands)
    costs = {s: T.simulate(prefix, drafts, 8, s) for s in cands}
    assert costs[plan] <= min(costs.values()) / 0.98 + 1e-9   # within the planner's 2 % hysteresis
