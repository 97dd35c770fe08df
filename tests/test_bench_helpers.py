"""bench.py's pure helpers (no GPU): launch statistics, the whole-job throughput,
and the rule that a recorded DRAM capture counts only for the sources it was
taken on."""
import json
import re

import numpy as np

import bench


def test_launch_stats_are_microseconds_of_the_per_launch_times():
    per_ms = [0.1 + 0.001 * i for i in range(101)]  # 100 .. 200 us
    st = bench.launch_stats(per_ms)
    assert st["n"] == 101
    assert abs(st["median"] - 150.0) < 1e-9
    assert abs(st["p10"] - 110.0) < 1e-9 and abs(st["p90"] - 190.0) < 1e-9
    assert abs(st["mean"] - 1e3 * float(np.mean(per_ms))) < 1e-9


def test_weak_scaling_counts_every_rank_bytes():
    # 529.5 MB per rank per step, 20 steps in 2.16 ms on 1 and on 4 ranks
    one = bench.weak_scaling_gbs(529_530_880, 1, 20, 2.16)
    four = bench.weak_scaling_gbs(529_530_880, 4, 20, 2.16)
    assert abs(one - 529_530_880 * 20 / 2.16e-3 / 1e9) < 1e-6
    assert abs(four - 4 * one) < 1e-6


def test_kernel_hash_is_a_stable_hex_digest():
    h = bench.kernel_hash()
    assert re.fullmatch(r"[0-9a-f]{16}", h)
    assert h == bench.kernel_hash()


def test_recorded_traffic_only_for_the_same_sources(tmp_path):
    path = tmp_path / "capture.json"
    assert bench.recorded_traffic(str(path), "abc") is None  # no capture
    path.write_text(json.dumps({"kernel_hash": "abc", "dram_bytes_per_launch": 543_000_000}))
    assert bench.recorded_traffic(str(path), "abc") == 543_000_000
    assert bench.recorded_traffic(str(path), "abd") is None  # other kernel sources
