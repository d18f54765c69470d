"""Plain CPU oracle of the SplitZip codec -- TEST INFRASTRUCTURE.

Only the tests, the smoke check (``__graft_entry__.smoke``) and the benchmark's
CPU-baseline / reference arm may import this package.  The product path (the
CUDA library and its Python binding) never does, and must not.

The arithmetic lives in ``splitzip_oracle.c``: single-threaded loops over the
elements, written from the method's description ("SplitZip: Ultra-Fast Lossless
KV Compression for Disaggregated LLM Serving", sections Abstract, Highlights,
Codec API and FAQ; the arXiv abstract on the paper index page).  This module
only compiles that file with gcc and marshals numpy arrays through ctypes.  It
shares no code with the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "splitzip_oracle.c")
_LIBPATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u64p = ctypes.POINTER(ctypes.c_uint64)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (plain C99, -O2)."""
    if (not force and os.path.exists(_LIBPATH)
            and os.path.getmtime(_LIBPATH) >= os.path.getmtime(_SRC)):
        return _LIBPATH
    tmp = _LIBPATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-Wall",
                    "-Werror", "-o", tmp, _SRC], check=True)
    os.replace(tmp, _LIBPATH)
    return _LIBPATH


def _bind(lib):
    u64, u32, i32, dbl = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int,
                          ctypes.c_double)
    lib.oracle_histogram_bf16.argtypes = [_u16p, u64, _u64p]
    lib.oracle_histogram_bf16.restype = None
    lib.oracle_histogram_e5m2.argtypes = [_u8p, u64, _u64p]
    lib.oracle_histogram_e5m2.restype = None
    lib.oracle_top16.argtypes = [_u64p, i32, _u8p]
    lib.oracle_top16.restype = i32
    lib.oracle_calibrate_bf16.argtypes = [_u16p, u64, _u8p]
    lib.oracle_calibrate_bf16.restype = dbl
    lib.oracle_calibrate_e5m2.argtypes = [_u8p, u64, _u8p]
    lib.oracle_calibrate_e5m2.restype = dbl
    enc = [u64, u32, _u8p, _u8p, _u8p, _u16p, _u8p, u64, _u32p]
    lib.oracle_encode_bf16.argtypes = [_u16p] + enc
    lib.oracle_encode_bf16.restype = u64
    lib.oracle_encode_e5m2.argtypes = [_u8p] + enc
    lib.oracle_encode_e5m2.restype = u64
    dec = [_u8p, _u8p, _u16p, _u8p, _u32p, u64, u32, _u8p, u64]
    lib.oracle_decode_bf16.argtypes = dec + [_u16p]
    lib.oracle_decode_bf16.restype = i32
    lib.oracle_decode_e5m2.argtypes = dec + [_u8p]
    lib.oracle_decode_e5m2.restype = i32
    lib.oracle_compressed_bytes_bf16.argtypes = [u64, u32, u64]
    lib.oracle_compressed_bytes_bf16.restype = u64
    lib.oracle_compressed_bytes_e5m2.argtypes = [u64, u32, u64]
    lib.oracle_compressed_bytes_e5m2.restype = u64
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


_override = threading.local()


def _active():
    lib = getattr(_override, "lib", None)
    return lib if lib is not None else _load()


class use_library:
    """Context manager: route this thread's oracle calls to another build of the
    oracle source (the mutation tests plant mistakes in a copy of the C file
    and check that the pins catch them)."""

    def __init__(self, so_path: str):
        self.lib = _bind(ctypes.CDLL(so_path))

    def __enter__(self):
        self.prev = getattr(_override, "lib", None)
        _override.lib = self.lib
        return self

    def __exit__(self, *exc):
        _override.lib = self.prev
        return False


def compile_variant(src_text: str, out_dir: str) -> str:
    """Compile C source text (a modified copy of the oracle) into out_dir."""
    src = os.path.join(out_dir, "variant.c")
    so = os.path.join(out_dir, "libvariant.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-o", so, src], check=True)
    return so


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as(x, dtype) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x).reshape(-1))
    if a.dtype != dtype:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def _dtype_info(fmt: str):
    if fmt == "bf16":
        return np.uint16, ctypes.c_uint16, 256
    if fmt == "e5m2":
        return np.uint8, ctypes.c_uint8, 32
    raise ValueError(f"unknown format {fmt!r}")


def signman_bytes(n: int, fmt: str) -> int:
    """Length of the sign+mantissa stream: n bytes (BF16) or ceil(3n/8) (E5M2)."""
    return n if fmt == "bf16" else (3 * n + 7) // 8


def histogram(x, fmt: str = "bf16") -> np.ndarray:
    """Exponent histogram (256 bins for BF16, 32 for E5M2)."""
    dt, ct, nb = _dtype_info(fmt)
    a = _as(x, dt)
    h = np.zeros(nb, np.uint64)
    fn = _active().oracle_histogram_bf16 if fmt == "bf16" else _active().oracle_histogram_e5m2
    fn(_ptr(a, ct), a.size, _ptr(h, ctypes.c_uint64))
    return h


def top16(hist) -> np.ndarray:
    """Top-16 codebook of a histogram (count descending, ties to the smaller exponent)."""
    h = np.ascontiguousarray(np.asarray(hist, dtype=np.uint64))
    cb = np.zeros(16, np.uint8)
    rc = _active().oracle_top16(_ptr(h, ctypes.c_uint64), h.size, _ptr(cb, ctypes.c_uint8))
    if rc != 0:
        raise ValueError("histogram needs 16..256 bins")
    return cb


def calibrate(x, fmt: str = "bf16"):
    """Returns (codebook uint8[16], coverage float)."""
    dt, ct, _ = _dtype_info(fmt)
    a = _as(x, dt)
    cb = np.zeros(16, np.uint8)
    fn = _active().oracle_calibrate_bf16 if fmt == "bf16" else _active().oracle_calibrate_e5m2
    cov = fn(_ptr(a, ct), a.size, _ptr(cb, ctypes.c_uint8))
    return cb, float(cov)


def encode(x, chunk: int, cb, fmt: str = "bf16", esc_capacity: int | None = None):
    """Encode; returns a dict of numpy streams plus ``n_escapes`` (E needed).

    With ``esc_capacity`` None the escape arrays are sized to fit (a second
    pass runs if a first guess was too small); otherwise exactly that many
    entries are allocated and only the first ``esc_capacity`` are stored.
    """
    dt, ct, _ = _dtype_info(fmt)
    a = _as(x, dt)
    n = a.size
    nchunks = -(-n // chunk)
    fn = _active().oracle_encode_bf16 if fmt == "bf16" else _active().oracle_encode_e5m2
    cap = esc_capacity if esc_capacity is not None else n // 64 + 1024
    while True:
        codes = np.zeros((n + 1) // 2, np.uint8)
        sm = np.zeros(signman_bytes(n, fmt), np.uint8)
        esc_pos = np.zeros(cap, np.uint16)
        esc_val = np.zeros(cap, np.uint8)
        chunk_off = np.zeros(nchunks + 1, np.uint32)
        cbv = np.ascontiguousarray(np.asarray(cb, dtype=np.uint8))
        E = fn(_ptr(a, ct), n, chunk, _ptr(cbv, ctypes.c_uint8), _ptr(codes, ctypes.c_uint8),
               _ptr(sm, ctypes.c_uint8), _ptr(esc_pos, ctypes.c_uint16),
               _ptr(esc_val, ctypes.c_uint8), cap, _ptr(chunk_off, ctypes.c_uint32))
        if esc_capacity is not None or E <= cap:
            break
        cap = int(E)
    if esc_capacity is None:
        esc_pos, esc_val = esc_pos[:E].copy(), esc_val[:E].copy()
    return {"codes": codes, "signman": sm, "esc_pos": esc_pos, "esc_val": esc_val,
            "chunk_off": chunk_off, "n_escapes": int(E)}


def decode(streams: dict, n: int, chunk: int, cb, fmt: str = "bf16") -> np.ndarray:
    """Decode streams back to the raw bit patterns (uint16 for BF16, uint8 for E5M2)."""
    dt, ct, _ = _dtype_info(fmt)
    y = np.zeros(n, dt)
    codes = np.ascontiguousarray(streams["codes"], dtype=np.uint8)
    sm = np.ascontiguousarray(streams["signman"], dtype=np.uint8)
    esc_pos = np.ascontiguousarray(streams["esc_pos"], dtype=np.uint16)
    esc_val = np.ascontiguousarray(streams["esc_val"], dtype=np.uint8)
    chunk_off = np.ascontiguousarray(streams["chunk_off"], dtype=np.uint32)
    cbv = np.ascontiguousarray(np.asarray(cb, dtype=np.uint8))
    assert codes.size >= (n + 1) // 2 and sm.size >= signman_bytes(n, fmt)
    assert chunk_off.size == -(-n // chunk) + 1
    fn = _active().oracle_decode_bf16 if fmt == "bf16" else _active().oracle_decode_e5m2
    rc = fn(_ptr(codes, ctypes.c_uint8), _ptr(sm, ctypes.c_uint8), _ptr(esc_pos, ctypes.c_uint16),
            _ptr(esc_val, ctypes.c_uint8), _ptr(chunk_off, ctypes.c_uint32), n, chunk,
            _ptr(cbv, ctypes.c_uint8), min(esc_pos.size, esc_val.size), _ptr(y, ct))
    if rc != 0:
        raise ValueError("malformed escape metadata")
    return y


def compressed_bytes(n: int, chunk: int, n_escapes: int, fmt: str = "bf16") -> int:
    fn = (_active().oracle_compressed_bytes_bf16 if fmt == "bf16"
          else _active().oracle_compressed_bytes_e5m2)
    return int(fn(n, chunk, n_escapes))
