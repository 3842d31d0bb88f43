"""Host-side bookkeeping of bench.py: the algorithmic work it divides by, and the number of
library launches it claims per end-to-end step. No GPU."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _pairs_brute(B, Lq, Lk, causal, valid_lens):
    """Allowed (query, key) pairs counted one by one: key j is allowed for query i when
    j < valid length (and j <= i under the causal mask); a row with no allowed key counts
    all L_k keys, since the -1e9 fill gives it uniform weights over them."""
    total = 0
    for b in range(B):
        vl = Lk if valid_lens is None else max(0, min(valid_lens[b], Lk))
        for i in range(Lq):
            allowed = sum(1 for j in range(Lk) if j < vl and (not causal or j <= i))
            total += allowed if allowed > 0 else Lk
    return total


@pytest.mark.parametrize("B,Lq,Lk,causal,vl", [
    (2, 9, 9, True, None), (3, 7, 7, True, [7, 0, 3]), (2, 5, 11, False, [11, 4]), (1, 6, 6, False, None)])
def test_algorithmic_flops_match_brute_force_pair_counts(B, Lq, Lk, causal, vl):
    d, h = 128, 2
    proj, attn = bench.algorithmic_flops(B, Lq, Lk, d, h, causal, None if vl is None else np.array(vl))
    assert proj == 2.0 * d * d * (2 * B * Lq + 2 * B * Lk)       # Q, K, V and W_o projections
    assert attn == 4.0 * (d // h) * h * _pairs_brute(B, Lq, Lk, causal, vl)


def test_long_workload_work_is_the_quoted_figure():
    """B=4, L=8192, d_model 1024, h 16, causal: L (L + 1) / 2 pairs per head."""
    proj, attn = bench.algorithmic_flops(4, 8192, 8192, 1024, 16, True)
    assert attn == 4 * 64 * 16 * 4 * (8192 * 8193 // 2)
    assert round(attn / 1e9, 1) == 549.8 and round(proj / 1e9, 1) == 274.9


def test_host_pipeline_launch_count_follows_the_chunk_rule():
    """3 launches per chunk of sequences (4 chunks from 32 MiB of host input, else 2, never more
    than B), + 2 for the row-windowed ends of a self-attention call with L >= 256."""
    f = bench.host_pipeline_launches
    assert f(4, 8192, 8192, 1024, False, False) == 3 * 4 + 2    # long: 64 MB of input
    assert f(32, 128, 128, 512, False, False) == 3 * 2          # enc: 4 MB, L < 256
    assert f(32, 256, 256, 512, False, False) == 3 * 2 + 2      # dec: 8 MB, windowed ends
    assert f(16, 256, 320, 1024, True, False) == 3 * 2          # cross-attention: 18.9 MB
    assert f(1, 8192, 8192, 1024, False, False) == 3 + 2        # one sequence: one chunk
    assert f(3, 4096, 4096, 1024, False, False) == 3 * 2 + 2    # 25 MB: a small call, 2 chunks
    assert f(3, 8192, 8192, 1024, False, False) == 3 * 3 + 2    # 50 MB: up to 4 chunks, B = 3 of them


def test_clock_summary_takes_the_median_under_load(tmp_path):
    """The clock record's sm_mhz is the median over samples drawn while kernels ran (power at
    least half the peak seen and 150 W); idle samples between timed loops and unparsable
    fields do not count, and every active slowdown reason is reported."""
    import bench
    f = tmp_path / "clocks.csv"
    na = "Not Active"
    f.write_text("\n".join([
        f"0, 2070, 2070, 95.0, 0x0, {na}, {na}, {na}, {na}",           # idle
        f"0, 2070, 2070, 820.5, 0x4, {na}, {na}, {na}, Active",        # under load, power cap
        f"0, 1980, 2070, 900.0, 0x4, {na}, {na}, {na}, Active",
        f"0, 1500, 2070, 120.0, 0x0, {na}, {na}, {na}, {na}",          # idle, low clock
        f"0, [N/A], 2070, [N/A], 0x0, {na}, {na}, {na}, {na}",
    ]) + "\n")

    class _F:
        name = str(f)

        def flush(self):
            pass

    c = bench.ClockSampler(0)
    c.proc, c.file = object(), _F()
    s = c.summary()
    assert s["samples"] == 5 and s["samples_under_load"] == 2
    assert s["sm_mhz"] == 2025.0 and s["sm_mhz_min_under_load"] == 1980.0
    assert s["sm_max_mhz"] == 2070.0 and s["power_w_max"] == 900.0
    assert s["reasons"] == ["sw_power_cap"]


@pytest.mark.parametrize("workload", [bench.WORKLOAD, "long_d128"])
def test_committed_attention_profile_matches_the_sources(workload):
    """The bench reports the attention kernel's DRAM traffic from the committed ncu summary only while
    the kernel's sources (the kernel file and the shared headers) hash to the digest that summary was
    taken on; a source change without a new capture would turn the figure into null."""
    digest = bench.source_digest("attention_core", workload)
    traffic = bench.committed_traffic("attention_core", workload)
    assert traffic is not None, f"no committed profile for source digest {digest} ({workload})"
    assert traffic > 0
