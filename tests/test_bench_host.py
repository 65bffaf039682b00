"""Host-side arithmetic of bench.py (no GPU): acceptance along the block."""

import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
torch = pytest.importorskip("torch")
import bench  # noqa: E402


def test_acceptance_rates_from_histogram():
    G = 4
    # tau = accepted drafts + 1: 2 cycles accepted nothing, 1 accepted one,
    # 1 accepted all three drafts
    r = bench.acceptance_rates([0, 2, 1, 0, 1], G)
    assert r["tau_mean"] == pytest.approx((2 * 1 + 1 * 2 + 1 * 4) / 4)
    # position 1 accepted in 2 of 4 cycles, position 2 and 3 in 1 of 4
    assert r["accept_rate_by_position"] == [0.5, 0.25, 0.25]
    assert r["accept_rate_given_previous"] == [0.5, 0.5, 1.0]


def test_acceptance_rates_all_rejected():
    r = bench.acceptance_rates([0, 5, 0, 0], 3)
    assert r["tau_mean"] == 1.0
    assert r["accept_rate_by_position"] == [0.0, 0.0]
    assert r["accept_rate_given_previous"] == [0.0, None]


def test_attention_ring_bytes_counts_the_visible_window():
    dims = dict(bench.DIMS_FULL)
    # 5 layers x 32 requests x 8 KV heads x 4096 keys x 128 dims x (K, V) x 2 bytes
    assert bench.attention_ring_bytes(dims, 32, 8192) == 5 * 32 * 8 * 4096 * 128 * 2 * 2
    assert bench.attention_ring_bytes(dims, 1, 100) == 5 * 8 * 100 * 128 * 2 * 2
