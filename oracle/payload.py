"""Oracle of the portable SplitZip payload (TEST INFRASTRUCTURE, NOT PRODUCT CODE).

Only the test suite and the benchmark's CPU arms use this module.  It shares
nothing with the CUDA library: it writes and reads the payload container with
``struct`` and numpy, one region after another, and encodes / decodes each
slice with the plain C oracle of this package.

The container has no counterpart on the pages beyond their roadmap item for
integration-facing codebook and payload metadata ("SplitZip: Ultra-Fast
Lossless KV Compression for Disaggregated LLM Serving", README section
Roadmap); its layout is the library's own definition, restated here:

  header (64 bytes, little-endian): b"SPLITZIP", version u32 = 1, format u32
      (0 = BF16, 1 = E5M2), n u64, slice_elems u64, num_slices u32,
      chunk_size u32, total escapes u64, total bytes u64, 8 zero bytes;
  slice table: per slice n u64, escapes u64, dense offset u64, escape offset
      u64, 16 codebook bytes (48 bytes);
  dense regions in slice order (codes, signman, chunk_off, each starting on a
      16-byte boundary, zero padding), then escape regions in slice order
      (esc_pos as uint16, esc_val as uint8, zero padding to 16 bytes).
Each slice is an independently encoded tensor of ``slice_elems`` elements
(the last one shorter).
"""
from __future__ import annotations

import struct

import numpy as np

from . import calibrate as _calibrate
from . import decode as _decode
from . import encode as _encode

MAGIC = b"SPLITZIP"
VERSION = 1
FORMAT_CODE = {"bf16": 0, "e5m2": 1}
HEADER = struct.Struct("<8sIIQQIIQQ8x")   # 64 bytes
ENTRY = struct.Struct("<QQQQ16s")         # 48 bytes


def _pad16(v: int) -> int:
    return (v + 15) // 16 * 16


def _slices(n: int, slice_elems: int):
    return [(s0, min(slice_elems, n - s0)) for s0 in range(0, n, slice_elems)]


def write(x, fmt: str, chunk: int, slice_elems: int, codebooks) -> bytes:
    """The payload of x (a flat array of uint16 BF16 or uint8 E5M2 bit
    patterns) cut into slices of slice_elems elements.  codebooks: one shared
    codebook (16 ints) or one per slice."""
    x = np.ascontiguousarray(x).reshape(-1)
    n = x.size
    parts = _slices(n, slice_elems)
    cbs = [list(codebooks)] * len(parts) if np.ndim(codebooks) == 1 else [list(c) for c in codebooks]
    assert len(cbs) == len(parts), "one codebook, or one per slice"
    encoded = [_encode(x[s0:s0 + m], chunk, np.asarray(cb, np.uint8), fmt)
               for (s0, m), cb in zip(parts, cbs)]

    dense = []
    for st in encoded:
        region = bytearray()
        for name in ("codes", "signman", "chunk_off"):
            region += np.ascontiguousarray(st[name]).tobytes()
            region += bytes(_pad16(len(region)) - len(region))
        dense.append(bytes(region))
    escapes = []
    for st in encoded:
        region = (np.asarray(st["esc_pos"], np.uint16).tobytes() +
                  np.asarray(st["esc_val"], np.uint8).tobytes())
        escapes.append(region + bytes(_pad16(len(region)) - len(region)))

    table_end = HEADER.size + ENTRY.size * len(parts)
    off = _pad16(table_end)
    dense_off = []
    for region in dense:
        dense_off.append(off)
        off += len(region)
    esc_off = []
    for region in escapes:
        esc_off.append(off)
        off += len(region)
    total = off
    n_esc = [int(st["n_escapes"]) for st in encoded]

    out = bytearray(HEADER.pack(MAGIC, VERSION, FORMAT_CODE[fmt], n, slice_elems, len(parts),
                                chunk, sum(n_esc), total))
    for (s0, m), e, d, q, cb in zip(parts, n_esc, dense_off, esc_off, cbs):
        out += ENTRY.pack(m, e, d, q, bytes(cb))
    out += bytes(_pad16(table_end) - table_end)
    for region in dense + escapes:
        out += region
    assert len(out) == total
    return bytes(out)


def write_calibrated(x, fmt: str, chunk: int, slice_elems: int) -> bytes:
    """The payload of x with a codebook of its own for every slice: each slice
    is calibrated on its own exponents (the top-16 of that slice, the pages'
    calibration step applied per KV-cache layer instead of once offline) and
    then encoded with that codebook."""
    x = np.ascontiguousarray(x).reshape(-1)
    cbs = [[int(c) for c in _calibrate(x[s0:s0 + m], fmt)[0]]
           for s0, m in _slices(x.size, slice_elems)]
    return write(x, fmt, chunk, slice_elems, cbs)


def read(buf: bytes):
    """(header dict, list of per-slice stream dicts) of a payload."""
    magic, version, fcode, n, se, S, chunk, esc, total = HEADER.unpack_from(buf, 0)
    if magic != MAGIC or version != VERSION or total > len(buf):
        raise ValueError("not a version-1 SplitZip payload")
    fmt = {v: k for k, v in FORMAT_CODE.items()}[fcode]
    head = {"fmt": fmt, "n": n, "slice_elems": se, "num_slices": S, "chunk_size": chunk,
            "n_escapes": esc, "total_bytes": total}
    slices = []
    for i in range(S):
        m, e, d, q, cb = ENTRY.unpack_from(buf, HEADER.size + ENTRY.size * i)
        n_codes = (m + 1) // 2
        n_sm = m if fmt == "bf16" else (3 * m + 7) // 8
        n_off = -(-m // chunk) + 1
        p = d
        codes = np.frombuffer(buf, np.uint8, n_codes, p)
        p = _pad16(p + n_codes)
        signman = np.frombuffer(buf, np.uint8, n_sm, p)
        p = _pad16(p + n_sm)
        chunk_off = np.frombuffer(buf, np.uint32, n_off, p)
        esc_pos = np.frombuffer(buf, np.uint16, e, q)
        esc_val = np.frombuffer(buf, np.uint8, e, q + 2 * e)
        slices.append({"n": m, "n_escapes": e, "off_dense": d, "off_escapes": q,
                       "codebook": list(cb), "codes": codes, "signman": signman,
                       "chunk_off": chunk_off, "esc_pos": esc_pos, "esc_val": esc_val})
    return head, slices


def decode(buf: bytes) -> np.ndarray:
    """The tensor a payload holds, decoded slice by slice with the oracle."""
    head, slices = read(buf)
    parts = [_decode(s, s["n"], head["chunk_size"], np.asarray(s["codebook"], np.uint8),
                     head["fmt"]) for s in slices]
    return np.concatenate(parts)
