"""Host-side accounting of bench.py (no GPU): the FLOP numerator of the
headline metric and the clock-record parsing that decides whether a run is
kept. The pair counts are checked against brute force over the masks (the
oracle's bottom-right mask for varlen), so a wrong closed form changes a
reported TFLOP/s figure and fails here.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle.attention as orc  # noqa: E402


def _brute_pairs(lengths, causal):
    tot = 0
    for L in lengths:
        for i in range(L):
            for j in range(L):
                tot += (j <= i) if causal else 1
    return tot


def test_pair_count_matches_brute_force():
    rng = np.random.default_rng(5)
    for causal in (False, True):
        for _ in range(20):
            lengths = rng.integers(0, 40, size=rng.integers(1, 6)).tolist()
            assert bench.pair_count(lengths, causal) == _brute_pairs(lengths, causal)
    assert bench.pair_count([], True) == 0


def test_var_pair_count_matches_the_bottom_right_mask():
    rng = np.random.default_rng(6)
    cases = [([0], [5]), ([5], [0]), ([3], [3]), ([7], [2]), ([2], [7]), ([1], [1])]
    for _ in range(30):
        n = int(rng.integers(1, 5))
        cases.append((rng.integers(0, 50, size=n).tolist(), rng.integers(0, 50, size=n).tolist()))
    for ql, kl in cases:
        want_causal = sum(int(orc.lower_right_visible(a, b).sum()) for a, b in zip(ql, kl))
        want_full = sum(a * b for a, b in zip(ql, kl))
        assert bench.var_pair_count(ql, kl, True) == want_causal, (ql, kl)
        assert bench.var_pair_count(ql, kl, False) == want_full, (ql, kl)
    # equal lengths: the self-attention count
    assert bench.var_pair_count([9, 4], [9, 4], True) == bench.pair_count([9, 4], True)


def test_attn_flops_counts_two_and_five_matmuls():
    lengths = [3, 10, 0, 7]
    pairs = bench.pair_count(lengths, False)
    assert bench.attn_flops(lengths, 4, 128, False, "fwd") == 4 * 128 * 4 * pairs
    assert bench.attn_flops(lengths, 4, 128, False, "bwd") == 10 * 128 * 4 * pairs
    cp = bench.pair_count(lengths, True)
    assert bench.attn_flops(lengths, 2, 64, True, "bwd") == 10 * 64 * 2 * cp


def test_clock_summary_flags_throttle_reasons():
    s = bench.ClockSampler(0)
    s.lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 1400.0, 0x4, Not Active, Active, Not Active, Active",
        "garbled line",
    ]
    out = s.summary()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2055.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    empty = bench.ClockSampler(0)
    assert empty.summary()["reasons"] == ["unsampled"]


def test_tc_peak_follows_the_clock_record():
    peaks = {"bf16_tflops": 1971.6, "bf16_tflops_sustained": 1718.0, "hbm_gbs": 6790.3}
    burst = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 4}
    capped = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 4}
    low = {"sm_mhz": 1455.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 40}
    assert bench.choose_tc_peak(peaks, burst)[:2] == (1971.6, "bf16_tflops")
    assert bench.choose_tc_peak(peaks, capped)[:2] == (1718.0, "bf16_tflops_sustained")
    assert bench.choose_tc_peak(peaks, low)[:2] == (1718.0, "bf16_tflops_sustained")
    # the headline kernel of the first bench line, recomputed: 864.1 TFLOP/s at burst clocks
    peak, _, _ = bench.choose_tc_peak(peaks, burst)
    assert abs(864.118 / peak - 0.438) < 1e-3


def test_attainable_roofline_of_the_sparse_gem_step():
    # GEM-like s=0.9 (105,061 tokens, 4 heads, d 128): 24 L d bytes per sequence and head
    lengths = [105061]
    nbytes = bench.attn_bytes(lengths, 4, 128, "fwd_bwd")
    assert nbytes == 24 * 128 * 4 * 105061
    assert bench.attn_bytes([3, 5], 2, 64, "fwd") + bench.attn_bytes([3, 5], 2, 64, "bwd") == \
        bench.attn_bytes([3, 5], 2, 64, "fwd_bwd")
    # HBM-bound: AI x bandwidth below the tensor peak
    att = bench.attainable(1.0e11, nbytes, 1971.6, 6790.3)
    assert abs(att - 1.0e11 / nbytes * 6790.3 / 1e3) < 1e-9 and att < 1971.6
    # compute-bound: capped at the tensor peak
    assert bench.attainable(1.0e15, 1.0e9, 1971.6, 6790.3) == 1971.6


def test_gpus_flag_must_match_the_launched_ranks(monkeypatch):
    import pytest
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    with pytest.raises(SystemExit):
        bench.dist_setup(2)
