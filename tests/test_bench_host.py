"""Host-side pieces of bench.py that need no GPU: the all-cores oracle
baseline (concurrent oracle runs over chunk-aligned shards)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402


def _bf16_bits(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)   # truncation is enough for a sample


def test_sharded_oracle_round_trips_every_shard():
    bits = _bf16_bits(5 * 1024 + 300, 0)                  # ragged: the last shard is short
    cb, _ = oracle.calibrate(bits, "bf16")
    sec = bench.time_oracle_sharded(bits, "bf16", 1024, cb, threads=3)
    assert sec > 0


def test_sharded_oracle_more_threads_than_chunks():
    bits = _bf16_bits(2 * 1024, 1)
    cb, _ = oracle.calibrate(bits, "bf16")
    assert bench.time_oracle_sharded(bits, "bf16", 1024, cb, threads=16) > 0


def test_host_threads_positive():
    assert bench.host_threads() >= 1
