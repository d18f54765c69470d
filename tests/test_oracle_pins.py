"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each test checks it against a
hand-worked fixture (tests/golden/), a closed form, a library routine (numpy
bincount / lexsort), IEEE-style float semantics of the bit patterns, or an
invariant the pages state (bitwise round trip: "SplitZip: Ultra-Fast Lossless
KV Compression for Disaggregated LLM Serving", section Codec API; ratio bounds
from 4-bit codes and, for E5M2, "up to 1.14x", section FAQ).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_kv_gb300 import synth
from tests.golden_io import STREAM_FIXTURES, fixture_streams, int_array, load


def _bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return t.contiguous().view(torch.uint8).numpy().reshape(-1)


def _exp_numpy(u: np.ndarray, fmt: str) -> np.ndarray:
    # Exponent field by library bit ops, for cross-checks (not the oracle's code).
    if fmt == "bf16":
        return ((u.astype(np.uint32) >> 7) & 0xFF).astype(np.int64)
    return ((u.astype(np.uint32) >> 2) & 0x1F).astype(np.int64)


# ----------------------------------------------------------------- fixtures

@pytest.mark.parametrize("name", STREAM_FIXTURES)
def test_golden_encode_streams(name):
    fx = fixture_streams(load(name))
    s = oracle.encode(fx["input"], fx["chunk"], fx["codebook"], fmt=fx["fmt"])
    np.testing.assert_array_equal(s["codes"], fx["codes"])
    np.testing.assert_array_equal(s["signman"], fx["signman"])
    np.testing.assert_array_equal(s["esc_pos"], fx["esc_pos"])
    np.testing.assert_array_equal(s["esc_val"], fx["esc_val"])
    np.testing.assert_array_equal(s["chunk_off"], fx["chunk_off"])
    assert s["n_escapes"] == fx["esc_pos"].size
    n = fx["input"].size
    assert oracle.compressed_bytes(n, fx["chunk"], s["n_escapes"], fx["fmt"]) == \
        fx["compressed_bytes"]


@pytest.mark.parametrize("name", STREAM_FIXTURES)
def test_golden_decode_streams(name):
    fx = fixture_streams(load(name))
    y = oracle.decode(fx, fx["input"].size, fx["chunk"], fx["codebook"], fmt=fx["fmt"])
    np.testing.assert_array_equal(y, fx["input"])


def test_golden_top16_tie_rule():
    fx = load("top16_tie_rule.txt")
    hist = np.zeros(int(fx["nbins"][0]), np.uint64)
    for tok in fx["nonzero"]:
        b, c = tok.split(":")
        hist[int(b)] = int(c)
    np.testing.assert_array_equal(oracle.top16(hist), int_array(fx["codebook"], np.uint8))


# ------------------------------------------------- exhaustive bit patterns

def test_all_bf16_patterns_self_calibrated():
    # Every exponent occurs 2 * 128 = 256 times among the 65536 patterns: all
    # bins tie, so the codebook is exponents 0..15 and covers 16/256 of them.
    x = _bits(synth.all_bf16_patterns())
    cb, cov = oracle.calibrate(x, "bf16")
    np.testing.assert_array_equal(cb, np.arange(16, dtype=np.uint8))
    assert cov == pytest.approx(16 / 256, abs=0)
    for chunk in (8, 1024, 65536):
        s = oracle.encode(x, chunk, cb, "bf16")
        assert s["n_escapes"] == 65536 - 16 * 256
        np.testing.assert_array_equal(oracle.decode(s, x.size, chunk, cb, "bf16"), x)


def test_all_bf16_patterns_kv_codebook():
    # A codebook of 16 distinct exponents covers exactly 16 * 256 patterns.
    cal = _bits(synth.kv_cache(1, 256, seed=1))
    cb, _ = oracle.calibrate(cal, "bf16")
    assert len(set(cb.tolist())) == 16
    x = _bits(synth.all_bf16_patterns())
    s = oracle.encode(x, 1024, cb, "bf16")
    assert s["n_escapes"] == 65536 - 16 * 256
    np.testing.assert_array_equal(oracle.decode(s, x.size, 1024, cb, "bf16"), x)


def test_all_e5m2_patterns():
    # 32 exponents x (2 signs x 4 mantissas) = 8 patterns each: all tie.
    x = _bits(synth.all_e5m2_patterns())
    cb, cov = oracle.calibrate(x, "e5m2")
    np.testing.assert_array_equal(cb, np.arange(16, dtype=np.uint8))
    assert cov == 0.5
    for chunk in (8, 16, 1024):
        s = oracle.encode(x, chunk, cb, "e5m2")
        assert s["n_escapes"] == 256 - 16 * 8
        np.testing.assert_array_equal(oracle.decode(s, x.size, chunk, cb, "e5m2"), x)


# --------------------------------------------- library-routine cross-checks

@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_histogram_matches_bincount(fmt):
    x = _bits(synth.kv_cache(2, 512, seed=3, dtype=torch.bfloat16 if fmt == "bf16"
                             else torch.float8_e5m2))
    nb = 256 if fmt == "bf16" else 32
    ref = np.bincount(_exp_numpy(x, fmt), minlength=nb).astype(np.uint64)
    np.testing.assert_array_equal(oracle.histogram(x, fmt), ref)


@pytest.mark.parametrize("seed", range(6))
def test_top16_matches_lexsort(seed):
    rng = np.random.default_rng(seed)
    nb = 256 if seed % 2 == 0 else 32
    hist = rng.integers(0, 6, nb).astype(np.uint64)  # many ties on purpose
    order = np.lexsort((np.arange(nb), -hist.astype(np.int64)))  # count desc, bin asc
    np.testing.assert_array_equal(oracle.top16(hist), order[:16].astype(np.uint8))


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_escapes_match_membership(fmt):
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    x = _bits(synth.kv_cache(1, 3000, seed=5, dtype=dt))  # n = 6,144,000
    cb, cov = oracle.calibrate(_bits(synth.kv_cache(1, 300, seed=6, dtype=dt)), fmt)
    chunk = 1000
    s = oracle.encode(x, chunk, cb, fmt)
    e = _exp_numpy(x, fmt)
    miss = ~np.isin(e, cb.astype(np.int64))
    # E = n - sum over codebook exponents of the histogram.
    hist = np.bincount(e, minlength=256 if fmt == "bf16" else 32)
    assert s["n_escapes"] == x.size - int(hist[cb.astype(np.int64)].sum())
    assert s["n_escapes"] == int(miss.sum())
    # Escapes are exactly the missed elements, in element order, chunk-local.
    idx = np.flatnonzero(miss)
    np.testing.assert_array_equal(s["esc_pos"], (idx % chunk).astype(np.uint16))
    np.testing.assert_array_equal(s["esc_val"], e[idx].astype(np.uint8))
    per_chunk = np.bincount(idx // chunk, minlength=-(-x.size // chunk))
    np.testing.assert_array_equal(s["chunk_off"],
                                  np.concatenate([[0], np.cumsum(per_chunk)]).astype(np.uint32))
    np.testing.assert_array_equal(oracle.decode(s, x.size, chunk, cb, fmt), x)


# ------------------------------------------------------ value semantics

def _bf16_value(sign, exponent, mantissa):
    # IEEE-style meaning of BF16 fields (bias 127, 7 fraction bits).
    if exponent == 255:
        return math.nan if mantissa else (-math.inf if sign else math.inf)
    if exponent == 0:
        mag = math.ldexp(mantissa / 128.0, -126)
    else:
        mag = math.ldexp(1.0 + mantissa / 128.0, exponent - 127)
    return -mag if sign else mag


def test_streams_carry_bf16_values():
    """Reading the streams as sign/mantissa byte + code -> exponent gives back
    each element's float value (checked through float arithmetic, not bits)."""
    t = synth.student_t_scaled_bf16((4096,), seed=9, u_lo=-6, u_hi=6)
    x = _bits(t)
    vals = t.float().numpy()
    cb, _ = oracle.calibrate(_bits(synth.normal_bf16((4096,), seed=1)), "bf16")
    chunk = 64
    s = oracle.encode(x, chunk, cb, "bf16")
    esc = {}
    for c in range(len(s["chunk_off"]) - 1):
        for j in range(s["chunk_off"][c], s["chunk_off"][c + 1]):
            esc[c * chunk + int(s["esc_pos"][j])] = int(s["esc_val"][j])
    for i in range(x.size):
        nib = (s["codes"][i // 2] >> (4 * (i % 2))) & 0xF
        exponent = esc.get(i, int(cb[nib]))
        sm = int(s["signman"][i])
        v = _bf16_value(sm >> 7, exponent, sm & 0x7F)
        if math.isnan(vals[i]):
            assert math.isnan(v)
        else:
            assert v == float(vals[i]), i
            assert math.copysign(1.0, v) == math.copysign(1.0, float(vals[i]))


# ---------------------------------------------------- closed forms / bounds

@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
@pytest.mark.parametrize("n,chunk", [(1, 8), (2, 8), (3, 8), (7, 8), (8, 8), (9, 8),
                                     (1023, 1024), (1024, 1024), (1025, 1024),
                                     (5000, 65536), (70001, 24)])
def test_sizes_and_roundtrip_edges(fmt, n, chunk):
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    x = _bits(synth.kv_cache(1, 1 + n // 2048, seed=n, dtype=dt))[:n].copy()
    cb, _ = oracle.calibrate(x, fmt)
    s = oracle.encode(x, chunk, cb, fmt)
    assert s["codes"].size == (n + 1) // 2
    assert s["signman"].size == (n if fmt == "bf16" else (3 * n + 7) // 8)
    C = -(-n // chunk)
    assert s["chunk_off"].size == C + 1 and s["chunk_off"][C] == s["n_escapes"]
    # compressed_bytes equals the byte count of the arrays actually produced.
    total = (s["codes"].nbytes + s["signman"].nbytes + s["esc_pos"].nbytes
             + s["esc_val"].nbytes + s["chunk_off"].nbytes)
    assert oracle.compressed_bytes(n, chunk, s["n_escapes"], fmt) == total
    np.testing.assert_array_equal(oracle.decode(s, n, chunk, cb, fmt), x)


def test_all_escape_input():
    # Every element's exponent outside the codebook: E = n, all codes 0.
    x = np.full(1000, 0x7F80, np.uint16)  # +inf, exponent 255
    cb = np.arange(16, dtype=np.uint8)
    s = oracle.encode(x, 256, cb, "bf16")
    assert s["n_escapes"] == 1000
    assert not s["codes"].any()
    np.testing.assert_array_equal(s["chunk_off"], [0, 256, 512, 768, 1000])
    np.testing.assert_array_equal(oracle.decode(s, 1000, 256, cb, "bf16"), x)


@pytest.mark.parametrize("fmt,bound", [("bf16", 4 / 3), ("e5m2", 8 / 7)])
def test_ratio_bounds(fmt, bound):
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    elem = 2 if fmt == "bf16" else 1
    x = _bits(synth.kv_cache(1, 4096, seed=11, dtype=dt))
    cb, _ = oracle.calibrate(x, fmt)
    s = oracle.encode(x, 1024, cb, fmt)
    ratio = elem * x.size / oracle.compressed_bytes(x.size, 1024, s["n_escapes"], fmt)
    assert ratio <= bound
    # Zero escapes: only the 4(C+1) metadata bytes keep the ratio below the bound.
    z = np.full(1 << 20, 0x3C if fmt == "e5m2" else 0x3F80,
                np.uint8 if fmt == "e5m2" else np.uint16)
    cbz, cov = oracle.calibrate(z, fmt)
    assert cov == 1.0
    sz = oracle.encode(z, 1024, cbz, fmt)
    assert sz["n_escapes"] == 0
    bz = oracle.compressed_bytes(z.size, 1024, 0, fmt)
    assert elem * z.size / bz == pytest.approx(bound * (1 - 4 * 1025 / bz), rel=1e-12)


def test_escape_capacity_overflow():
    x = _bits(synth.student_t_scaled_bf16((20000,), seed=4))
    cb, _ = oracle.calibrate(_bits(synth.normal_bf16((4096,), seed=1)), "bf16")
    full = oracle.encode(x, 1024, cb, "bf16")
    E = full["n_escapes"]
    assert E > 100
    part = oracle.encode(x, 1024, cb, "bf16", esc_capacity=100)
    assert part["n_escapes"] == E  # the count still reports the need
    np.testing.assert_array_equal(part["esc_pos"], full["esc_pos"][:100])
    np.testing.assert_array_equal(part["esc_val"], full["esc_val"][:100])
    for k in ("codes", "signman", "chunk_off"):
        np.testing.assert_array_equal(part[k], full[k])


def test_codec_api_example_round_trip():
    # README section Codec API: randn(1024, 4096) BF16, calibrated on itself,
    # chunk 1024, decodes bitwise to the input.
    x = _bits(synth.normal_bf16((1024, 4096), seed=0))
    cb, cov = oracle.calibrate(x, "bf16")
    assert 0.99 < cov <= 1.0
    s = oracle.encode(x, 1024, cb, "bf16")
    np.testing.assert_array_equal(oracle.decode(s, x.size, 1024, cb, "bf16"), x)
