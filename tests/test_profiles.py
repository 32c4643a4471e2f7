"""The DRAM-traffic record the bench's roofline line reports belongs to the indexer as it
is built now: its source hash matches the one the counters were taken with, and its
figures are consistent (read + write = the launch's traffic; the ratio to the
algorithmic bytes, which are the bench's own formula for the DeepSeek-V3.2 decode
shape: k^I + scores + q and w per launch)."""
import json
import os

import bench

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_indexer_traffic_record_matches_the_current_kernel():
    rec = json.load(open(os.path.join(ROOT, "profiles", "indexer_traffic.json")))
    assert rec["source_sha256"] == bench.indexer_source_sha256(), \
        "the indexer changed since its DRAM traffic was captured: re-take the counters"
    assert rec["bytes_per_launch_full_shape"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    alg = bench.B * bench.L * 128 + bench.B * bench.L * 4 + bench.B * (64 * 128 + 64 * 4)
    assert rec["algorithmic_bytes"] == alg
    assert abs(rec["traffic_over_algorithmic"] - rec["bytes_per_launch_full_shape"] / alg) < 1e-4
    assert 1.0 <= rec["traffic_over_algorithmic"] < 1.1   # k^I is read once
    assert "--clock-control none" in rec["command"]
