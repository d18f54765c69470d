"""C-ABI library: it builds, loads without a GPU and exports every function
include/*.h declares; its pure host functions agree with the oracle's closed
forms.  No compute call is made here."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from lossless_bf16_kv_gb300 import _build
from lossless_bf16_kv_gb300 import splitzip as sz

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in ("splitzip.h", "splitzip_testing.h", "splitzip_transfer.h"):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(splitzip_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    _build.build_library()
    return ctypes.CDLL(_build.LIBPATH)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("splitzip_calibrate", "splitzip_encode", "splitzip_decode",
                 "splitzip_compressed_bytes", "splitzip_calibrate_e5m2", "splitzip_encode_e5m2",
                 "splitzip_decode_e5m2", "splitzip_compressed_bytes_e5m2"):
        assert must in names


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_binds_every_declared_function(lib):
    bound = sz.library()
    for name in declared_functions():
        assert getattr(bound, name).argtypes is not None, name


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_compressed_bytes_matches_oracle(fmt, lib):
    rng = np.random.default_rng(7)
    for _ in range(300):
        n = int(rng.integers(1, 1 << 32))
        chunk = 8 * int(rng.integers(1, 8193))
        E = int(rng.integers(0, n + 1))
        assert sz.splitzip_compressed_bytes(n, chunk, E, fmt) == \
            oracle.compressed_bytes(n, chunk, E, fmt)


def test_stream_sizes(lib):
    for n in (1, 2, 3, 8, 9, 1000, 2**31, 2**32 - 1):
        assert sz.library().splitzip_codes_bytes(n) == (n + 1) // 2
        assert sz.splitzip_signman_bytes(n, "bf16") == n
        assert sz.splitzip_signman_bytes(n, "e5m2") == (3 * n + 7) // 8
        assert sz.splitzip_num_chunks(n, 1024) == -(-n // 1024)
    # 4 KiB header, a uint32 escape count per block of 64 tiles and per
    # superblock of 4096 tiles for the largest element count (fixed size),
    # then per 8192-element tile: an 8-byte look-back word, a 4-byte escape
    # count, 32 uint16 segment counts and 256 uint16 escape entries; each
    # array rounded up to 256 bytes.
    sums = 4 * (2**19 // 64 + 2**19 // 4096)
    def expect(n):
        t = -(-n // 8192)
        a = lambda v: -(-v // 256) * 256
        return 4096 + sums + a(8 * t) + a(4 * t) + a(64 * t) + a(512 * t)
    for n in (1, 8192, 8193, 10**6, 2**31, 2**32 - 1):
        assert sz.splitzip_workspace_bytes(n) == expect(n)
    assert sz.splitzip_workspace_bytes(2**31) == 4096 + 33280 + 588 * 2**18


def test_chunk_division_multiplier():
    """The kernels divide x < 2^17 by the chunk d (8 <= d <= 65536, d % 8 == 0)
    as (x * ceil(2^33 / d)) >> 33; check it against integer division."""
    x = np.arange(1 << 17, dtype=np.uint64)
    for d in list(range(8, 4097, 8)) + [8 * k for k in (1021, 4093, 8191, 8192)] + [65528, 65536]:
        m = np.uint64(((1 << 33) + d - 1) // d)
        np.testing.assert_array_equal((x * m) >> np.uint64(33), x // np.uint64(d))


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(sz, "LIBPATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(sz, "_lib", None)
    with pytest.raises(ImportError):
        sz.library()
