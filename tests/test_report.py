"""Exponent statistics report: its arithmetic pinned by closed forms and by
the oracle (escape counts and compressed sizes of real encodes).  CPU only."""
import math

import numpy as np
import pytest

import oracle
from lossless_bf16_kv_gb300.report import exponent_stats


def _cb(hist):
    return list(oracle.top16(np.asarray(hist, np.uint64)))


def test_uniform_histograms_have_log2_entropy():
    for k in (1, 2, 16, 256):
        h = np.zeros(256, np.int64)
        h[:k] = 1000
        s = exponent_stats(h, _cb(h))
        assert s["entropy_bits"] == pytest.approx(math.log2(k), abs=1e-12)
        assert s["distinct_exponents"] == k
        assert s["topk_coverage"][1] == pytest.approx(1 / k)


def test_two_point_entropy():
    h = np.zeros(256, np.int64)
    h[120], h[121] = 3, 1
    s = exponent_stats(h, _cb(h))
    assert s["entropy_bits"] == pytest.approx(-(0.75 * math.log2(0.75) + 0.25 * math.log2(0.25)))
    assert s["topk_coverage"][1] == 0.75 and s["topk_coverage"][2] == 1.0


@pytest.mark.parametrize("fmt,chunk", [("bf16", 1024), ("bf16", 64), ("e5m2", 1024)])
def test_escapes_and_ratio_match_the_oracle(fmt, chunk):
    rng = np.random.default_rng(11)
    n = 50001
    if fmt == "bf16":
        x = ((rng.standard_normal(n).astype(np.float32) * 4).view(np.uint32) >> 16).astype(np.uint16)
    else:
        x = rng.integers(0, 256, n, dtype=np.uint8)
    cal = x[: n // 3]
    cb, _ = oracle.calibrate(cal, fmt)
    hist = oracle.histogram(x, fmt)
    s = exponent_stats(hist, list(cb), fmt, chunk)
    ref = oracle.encode(x, chunk, cb, fmt)
    assert s["n_escapes"] == ref["n_escapes"]
    assert s["compression_ratio"] == pytest.approx(
        n * (2 if fmt == "bf16" else 1) / oracle.compressed_bytes(n, chunk, ref["n_escapes"], fmt))
    # An ideal entropy coder of the exponents never does worse than 4-bit codes
    # without escapes.
    if s["n_escapes"] == 0:
        assert s["entropy_coded_ratio"] >= s["compression_ratio"] * 0.999
    cover = [s["topk_coverage"][k] for k in (1, 2, 4, 8, 16)]
    assert cover == sorted(cover) and cover[-1] <= 1.0
