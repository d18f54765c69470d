"""Portable payload (include/splitzip_transfer.h): the oracle's container
writer and reader, checked against the layout rules and the per-slice codec,
and the library's host-side parser and size bound checked against payloads
the oracle wrote.  CPU only: no compute call of the library is made."""
import struct

import numpy as np
import pytest

import oracle
from oracle import payload as op
from lossless_bf16_kv_gb300 import splitzip as sz


def _data(fmt, n, seed):
    rng = np.random.default_rng(seed)
    if fmt == "bf16":
        # Normal values (BF16 bit patterns by truncation) plus a few arbitrary patterns.
        v = (rng.standard_normal(n).astype(np.float32) * 3.0).view(np.uint32) >> 16
        x = v.astype(np.uint16)
        k = max(1, n // 97)
        x[rng.integers(0, n, k)] = rng.integers(0, 1 << 16, k, dtype=np.uint16)
    else:
        x = rng.integers(0, 256, n, dtype=np.uint8)
        x[: n // 2] = (x[: n // 2] & 0x83) | (15 << 2)  # half with one exponent
    return x


def _codebook(x, fmt):
    return [int(c) for c in oracle.calibrate(x, fmt)[0]]


CASES = [("bf16", 5000, 256, 1024), ("bf16", 4096, 1024, 1024), ("bf16", 70001, 64, 16384),
         ("e5m2", 9999, 512, 2048), ("e5m2", 1, 8, 16)]


@pytest.mark.parametrize("fmt,n,chunk,se", CASES)
def test_oracle_payload_round_trips(fmt, n, chunk, se):
    x = _data(fmt, n, n)
    buf = op.write(x, fmt, chunk, se, _codebook(x, fmt))
    assert np.array_equal(op.decode(buf), x)


@pytest.mark.parametrize("fmt,n,chunk,se", CASES)
def test_oracle_payload_layout(fmt, n, chunk, se):
    """Header fields are the inputs; every region starts on 16 bytes, lies in
    order without overlap and has the size of its stream; each slice holds
    exactly the oracle's encoding of that slice."""
    x = _data(fmt, n, n + 1)
    cb = _codebook(x, fmt)
    buf = op.write(x, fmt, chunk, se, cb)
    head, slices = op.read(buf)
    S = -(-n // se)
    assert buf[:8] == b"SPLITZIP" and struct.unpack_from("<II", buf, 8) == (1, 0 if fmt == "bf16" else 1)
    assert (head["n"], head["slice_elems"], head["num_slices"], head["chunk_size"]) == (n, se, S, chunk)
    assert head["total_bytes"] == len(buf) and len(buf) % 16 == 0
    prev_end = 64 + 48 * S
    for i, s in enumerate(slices):
        m = min(se, n - i * se)
        ref = oracle.encode(x[i * se: i * se + m], chunk, np.asarray(cb, np.uint8), fmt)
        assert s["n"] == m and s["n_escapes"] == ref["n_escapes"]
        for name in ("codes", "signman", "chunk_off", "esc_pos", "esc_val"):
            assert np.array_equal(s[name], ref[name]), name
        assert s["off_dense"] % 16 == 0 and s["off_dense"] >= prev_end
        sizes = [(m + 1) // 2, m if fmt == "bf16" else (3 * m + 7) // 8, 4 * (-(-m // chunk) + 1)]
        prev_end = s["off_dense"] + sum((v + 15) // 16 * 16 for v in sizes)
    for s in slices:
        assert s["off_escapes"] % 16 == 0 and s["off_escapes"] >= prev_end
        prev_end = s["off_escapes"] + (3 * s["n_escapes"] + 15) // 16 * 16
    assert prev_end == len(buf)
    assert head["n_escapes"] == sum(s["n_escapes"] for s in slices)


def test_per_slice_codebooks():
    x = np.concatenate([_data("bf16", 3000, 5), (_data("bf16", 3000, 6) & 0x807F) | (100 << 7)])
    cbs = [_codebook(x[:3072], "bf16"), _codebook(x[3072:], "bf16")]
    buf = op.write(x, "bf16", 256, 3072, cbs)
    _, slices = op.read(buf)
    assert [s["codebook"] for s in slices] == cbs
    assert np.array_equal(op.decode(buf), x)


def _torch_buf(buf: bytes):
    import torch
    return torch.frombuffer(bytearray(buf), dtype=torch.uint8)


@pytest.mark.parametrize("fmt,n,chunk,se", CASES)
def test_library_parses_oracle_payloads(fmt, n, chunk, se):
    x = _data(fmt, n, n + 2)
    buf = op.write(x, fmt, chunk, se, _codebook(x, fmt))
    info, slices = sz.splitzip_payload_parse(_torch_buf(buf))
    head, ref = op.read(buf)
    for k in ("n", "slice_elems", "num_slices", "chunk_size", "n_escapes", "total_bytes"):
        assert info[k] == head[k], k
    assert info["fmt"] == fmt and info["version"] == 1
    for s, r in zip(slices, ref):
        for k in ("n", "n_escapes", "off_dense", "off_escapes", "codebook"):
            assert s[k] == r[k], k
    # The size bound is exact for one slice and an upper bound otherwise.
    bound = sz.splitzip_payload_bytes_bound(n, chunk, se, head["n_escapes"], fmt)
    assert bound >= len(buf)
    if head["num_slices"] == 1:
        assert bound == len(buf)


def _corruptions(buf: bytes):
    b = bytearray(buf)
    yield "magic", b[:0] + b"SPLITZAP" + b[8:]
    yield "version", b[:8] + struct.pack("<I", 2) + b[12:]
    yield "format", b[:12] + struct.pack("<I", 7) + b[16:]
    n = struct.unpack_from("<Q", b, 16)[0]
    yield "n", b[:16] + struct.pack("<Q", n + 1) + b[24:]
    yield "chunk", b[:36] + struct.pack("<I", 12) + b[40:]
    tot = struct.unpack_from("<Q", b, 48)[0]
    yield "total", b[:48] + struct.pack("<Q", tot + 16) + b[56:]
    e = struct.unpack_from("<Q", b, 64 + 8)[0]
    yield "escapes", b[:72] + struct.pack("<Q", e + 1) + b[80:]
    d = struct.unpack_from("<Q", b, 64 + 16)[0]
    yield "dense offset", b[:80] + struct.pack("<Q", d + 16) + b[88:]
    cb = bytearray(b[96:112])
    cb[1] = cb[0]
    yield "duplicate codebook entry", b[:96] + cb + b[112:]
    yield "truncated", b[: len(b) - 16]


def test_library_rejects_malformed_payloads():
    x = _data("bf16", 5000, 9)
    buf = op.write(x, "bf16", 256, 2048, _codebook(x, "bf16"))
    sz.splitzip_payload_parse(_torch_buf(buf))  # the intact payload parses
    for what, bad in _corruptions(buf):
        with pytest.raises(sz.SplitZipError):
            sz.splitzip_payload_parse(_torch_buf(bytes(bad)), len(bad))
        assert what


@pytest.mark.parametrize("name", ["payload_bf16_two_slices.txt", "payload_e5m2_two_slices.txt"])
def test_hand_worked_payload(name):
    """A payload derived by hand from the format spec (tests/golden/): the
    oracle writes exactly its bytes and decodes them back, and the library's
    parser and size bound agree."""
    from tests.golden_io import hex_array, int_array, load
    fx = load(name)
    fmt = fx["format"][0]
    rows = sorted((int(k.split("@")[1]), v) for k, v in fx.items() if k.startswith("payload@"))
    assert [off for off, _ in rows] == list(range(0, 16 * len(rows), 16))
    ref = bytes(int(t, 16) for _, v in rows for t in v)
    x = hex_array(fx["input_hex"], np.uint16 if fmt == "bf16" else np.uint8)
    cb = [int(c) for c in fx["codebook"]]
    chunk, se = int(fx["chunk"][0]), int(fx["slice_elems"][0])
    assert len(ref) == int(fx["total_bytes"][0])
    assert op.write(x, fmt, chunk, se, cb) == ref
    assert np.array_equal(op.decode(ref), x)
    info, slices = sz.splitzip_payload_parse(_torch_buf(ref))
    assert (info["fmt"], info["version"], info["n"], info["slice_elems"], info["chunk_size"]) == \
        (fmt, 1, len(x), se, chunk)
    assert info["num_slices"] == 2 and info["n_escapes"] == int(fx["n_escapes"][0])
    assert info["total_bytes"] == len(ref)
    assert [s["n"] for s in slices] == [int(v) for v in fx["slice_n"]]
    assert [s["n_escapes"] for s in slices] == [int(v) for v in fx["slice_escapes"]]
    assert [s["off_dense"] for s in slices] == [int(v) for v in fx["slice_off_dense"]]
    assert [s["off_escapes"] for s in slices] == [int(v) for v in fx["slice_off_escapes"]]
    assert all(list(s["codebook"]) == cb for s in slices)
    assert sz.splitzip_payload_bytes_bound(len(x), chunk, se, info["n_escapes"], fmt) == len(ref)
    assert int_array(fx["slice_n"], np.uint64).sum() == len(x)


def _per_slice_input(fmt):
    """Two slices whose exponent counts are fixed by construction, so each
    slice's top-16 codebook (count descending, ties to the smaller exponent)
    is known by hand.  Slice 0 (208 elements): exponent b + k appears 20 - k
    times (k < 16) and eight other exponents once each.  Slice 1 (204
    elements, the ragged last slice): exponents t + 2..t + 15 appear 7..20
    times, t and t + 1 six times each (a tie), and two more exponents three
    times in all.  Signs, mantissas and the order within a slice are random."""
    rng = np.random.default_rng(17)
    if fmt == "bf16":
        b, t, rare0, rare1 = 100, 120, list(range(50, 58)), [200, 200, 5]
    else:
        b, t, rare0, rare1 = 0, 16, list(range(16, 24)), [0, 0, 1]
    e0 = [b + k for k in range(16) for _ in range(20 - k)] + rare0
    counts1 = [6, 6] + list(range(7, 21))
    e1 = [t + k for k in range(16) for _ in range(counts1[k])] + rare1
    cb0 = [b + k for k in range(16)]
    cb1 = [t + k for k in range(15, 1, -1)] + [t, t + 1]
    parts = []
    for e in (e0, e1):
        e = rng.permutation(np.asarray(e, np.uint32))
        if fmt == "bf16":
            sm = rng.integers(0, 1 << 16, e.size, dtype=np.uint32) & 0x807F
            parts.append((sm | (e << 7)).astype(np.uint16))
        else:
            sm = rng.integers(0, 256, e.size, dtype=np.uint32) & 0x83
            parts.append((sm | (e << 2)).astype(np.uint8))
    return np.concatenate(parts), [cb0, cb1], [8, 3]


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_per_slice_calibrated_payload_codebooks(fmt):
    """The oracle's per-slice calibrated payload: every slice carries the
    top-16 of its own exponents (worked out by hand above), its escapes are
    exactly the elements outside that codebook, and the rest of the payload
    is the pinned writer's with those codebooks."""
    x, cbs, escapes = _per_slice_input(fmt)
    assert x.size == 412
    buf = op.write_calibrated(x, fmt, 8, 208)
    head, slices = op.read(buf)
    assert [s["codebook"] for s in slices] == cbs
    assert [s["n_escapes"] for s in slices] == escapes and head["n_escapes"] == 11
    assert buf == op.write(x, fmt, 8, 208, cbs)
    assert np.array_equal(op.decode(buf), x)
    # One codebook for the whole tensor would not be either slice's.
    whole = [int(c) for c in oracle.calibrate(x, fmt)[0]]
    assert whole not in cbs
