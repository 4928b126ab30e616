"""The host-only legs of bench.py: the oracle's decode and quantize timings on bounded samples."""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_oracle_decode_timing_on_a_bounded_sample():
    r = bench.time_oracle(W.ALL["tiny"](), 0.2)
    assert r["value"] > 0 and r["cores"] == 1 and r["kind"] == "oracle" and "repetitions" in r["sample"]


def test_oracle_quantize_timing_on_a_bounded_sample():
    wl = W.ALL["llama7b"]()
    r = bench.time_oracle_quantize(wl, 0.3)
    assert r["value"] > 0 and r["unit"] == "GB/s" and r["cores"] == 1 and r["kind"] == "oracle"
    assert "of 8193 tokens x 32 KV heads" in r["sample"]
