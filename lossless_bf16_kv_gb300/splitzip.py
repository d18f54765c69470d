"""Thin Python binding of the SplitZip C ABI (include/splitzip.h).

Argument marshalling only: PyTorch supplies device memory and streams, and
every step of the codec runs in the library's CUDA kernels.  The binding fails
loudly if the library is missing; there is no CPU fallback.

Low level: ``splitzip_*`` functions with the C names, taking torch tensors.
High level: ``ChunkLocalSplitZipGPU``, shaped like the codec API the pages
describe ("SplitZip: Ultra-Fast Lossless KV Compression for Disaggregated LLM
Serving", README section Codec API: ``calibrate(x) -> coverage``,
``encode(x) -> encoded`` with ``.compressed_bytes``, ``decode(encoded)``).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIBPATH = os.path.join(_PKG, "_lib", "libsplitzip.so")

(OK, ERR_INVALID_ARG, ERR_ESCAPE_OVERFLOW, ERR_TIMEOUT, ERR_CUDA, ERR_WORKSPACE,
 ERR_TOO_LARGE) = range(7)
STATUS_NAMES = {OK: "OK", ERR_INVALID_ARG: "INVALID_ARG", ERR_ESCAPE_OVERFLOW: "ESCAPE_OVERFLOW",
                ERR_TIMEOUT: "TIMEOUT", ERR_CUDA: "CUDA", ERR_WORKSPACE: "WORKSPACE",
                ERR_TOO_LARGE: "TOO_LARGE"}
MAX_CHUNK = 65536
MAX_ELEMENTS = 0xFFFFFFFF
TEST_STALL_FIRST_TILE = 0x1
TEST_PIPELINED = 0x2


class SplitZipError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class Codebook(ctypes.Structure):
    _fields_ = [("exp", ctypes.c_uint8 * 16)]


class Streams(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("signman", ctypes.c_void_p),
                ("esc_pos", ctypes.c_void_p), ("esc_val", ctypes.c_void_p),
                ("chunk_off", ctypes.c_void_p), ("esc_capacity", ctypes.c_uint64)]


class PayloadInfo(ctypes.Structure):
    _fields_ = [("version", ctypes.c_uint32), ("format", ctypes.c_uint32),
                ("n", ctypes.c_uint64), ("slice_elems", ctypes.c_uint64),
                ("num_slices", ctypes.c_uint32), ("chunk_size", ctypes.c_uint32),
                ("n_escapes", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64)]


class SliceEntry(ctypes.Structure):
    _fields_ = [("n", ctypes.c_uint64), ("n_escapes", ctypes.c_uint64),
                ("off_dense", ctypes.c_uint64), ("off_escapes", ctypes.c_uint64),
                ("cb", Codebook)]


FORMATS = {"bf16": 0, "e5m2": 1}


class EncodeTestOpts(ctypes.Structure):
    _fields_ = [("spin_limit", ctypes.c_uint32), ("flags", ctypes.c_uint32)]


_lib = None


def library() -> ctypes.CDLL:
    """The loaded libsplitzip.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBPATH):
        raise ImportError(f"{LIBPATH} is missing: build it first "
                          "(python -m lossless_bf16_kv_gb300._build)")
    lib = ctypes.CDLL(LIBPATH)
    vp, u64, u32, i32, st = (ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int,
                             ctypes.c_int)
    cbp, sp = ctypes.POINTER(Codebook), ctypes.POINTER(Streams)
    sig = {
        "splitzip_workspace_bytes": (ctypes.c_size_t, [u64, u32]),
        "splitzip_workspace_init": (st, [vp, ctypes.c_size_t, vp]),
        "splitzip_codes_bytes": (u64, [u64]),
        "splitzip_signman_bytes": (u64, [u64]),
        "splitzip_signman_bytes_e5m2": (u64, [u64]),
        "splitzip_num_chunks": (u64, [u64, u32]),
        "splitzip_compressed_bytes": (u64, [u64, u32, u64]),
        "splitzip_compressed_bytes_e5m2": (u64, [u64, u32, u64]),
        "splitzip_calibrate": (st, [vp, u64, cbp, ctypes.POINTER(ctypes.c_double), vp, vp]),
        "splitzip_calibrate_e5m2": (st, [vp, u64, cbp, ctypes.POINTER(ctypes.c_double), vp, vp]),
        "splitzip_calibrate_async": (st, [vp, u64, vp, vp, vp, vp]),
        "splitzip_calibrate_async_e5m2": (st, [vp, u64, vp, vp, vp, vp]),
        "splitzip_histogram": (st, [vp, u64, vp, vp, vp]),
        "splitzip_histogram_e5m2": (st, [vp, u64, vp, vp, vp]),
        "splitzip_encode": (st, [vp, u64, u32, cbp, sp, vp, vp]),
        "splitzip_encode_e5m2": (st, [vp, u64, u32, cbp, sp, vp, vp]),
        "splitzip_encode_test": (st, [vp, u64, u32, cbp, sp, vp, vp, i32,
                                      ctypes.POINTER(EncodeTestOpts)]),
        "splitzip_encode_status": (st, [vp, vp, ctypes.POINTER(u64)]),
        "splitzip_decode": (st, [sp, u64, u32, cbp, vp, vp]),
        "splitzip_decode_e5m2": (st, [sp, u64, u32, cbp, vp, vp]),
        "splitzip_encode_devcb": (st, [vp, u64, u32, vp, sp, vp, vp]),
        "splitzip_encode_devcb_e5m2": (st, [vp, u64, u32, vp, sp, vp, vp]),
        "splitzip_decode_devcb": (st, [sp, u64, u32, vp, vp, vp]),
        "splitzip_decode_devcb_e5m2": (st, [sp, u64, u32, vp, vp, vp]),
        "splitzip_encode_noalloc": (st, [vp, u64, u32, cbp, sp, vp, vp]),
        "splitzip_version": (i32, []),
        "splitzip_payload_bytes_bound": (u64, [u32, u64, u32, u64, u64]),
        "splitzip_payload_parse": (st, [vp, u64, ctypes.POINTER(PayloadInfo),
                                        ctypes.POINTER(SliceEntry), u32]),
        "splitzip_transfer_scratch_bytes": (ctypes.c_size_t, [u32, u64, u32]),
        "splitzip_encode_to_host": (st, [vp, u64, u32, u32, cbp, u32, u64, vp, u64,
                                         ctypes.POINTER(u64), vp, ctypes.c_size_t, vp, vp, vp]),
        "splitzip_encode_to_host_events": (st, [vp, u64, u32, u32, cbp, u32, u64, vp, u64,
                                                ctypes.POINTER(u64), vp, ctypes.c_size_t,
                                                vp, vp, vp, ctypes.POINTER(vp), u32]),
        "splitzip_decode_from_host": (st, [vp, u64, vp, u64, vp, ctypes.c_size_t, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != OK:
        raise SplitZipError(status, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, what: str) -> ctypes.c_void_p:
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _fmt_of(x: torch.Tensor, fmt: str | None) -> str:
    if fmt is not None:
        return fmt
    if x.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        return "bf16"
    if x.dtype in (torch.float8_e5m2, torch.uint8):
        return "e5m2"
    raise TypeError(f"unsupported dtype {x.dtype}")


_ELEM = {"bf16": 2, "e5m2": 1}


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def _need(t: torch.Tensor, nbytes: int, what: str):
    """The C ABI takes plain pointers: check here that t holds nbytes."""
    if _nbytes(t) < nbytes:
        raise SplitZipError(ERR_INVALID_ARG, f"{what} holds {_nbytes(t)} bytes, {nbytes} needed")


def _elements(x: torch.Tensor, fmt: str, what: str = "x") -> int:
    """Element count of x in the format's element width (2 bytes BF16, 1 E5M2)."""
    if fmt not in _ELEM:
        raise ValueError(f"unknown format {fmt!r}")
    if x.element_size() != _ELEM[fmt]:
        raise SplitZipError(ERR_INVALID_ARG,
                            f"{what} has {x.element_size()}-byte elements, {fmt} needs {_ELEM[fmt]}")
    return x.numel()


def _need_streams(s: dict, n: int, chunk: int, fmt: str):
    _need(s["codes"], splitzip_codes_bytes(n), "codes")
    _need(s["signman"], splitzip_signman_bytes(n, fmt), "signman")
    _need(s["chunk_off"], 4 * (splitzip_num_chunks(n, chunk) + 1), "chunk_off")


def _codebook(cb) -> Codebook:
    c = Codebook()
    vals = [int(v) for v in (cb.tolist() if hasattr(cb, "tolist") else cb)]
    if len(vals) != 16:
        raise ValueError("a codebook has 16 entries")
    for k, v in enumerate(vals):
        c.exp[k] = v
    return c


def _streams(s: dict) -> Streams:
    out = Streams()
    out.codes = _dev(s["codes"], "codes")
    out.signman = _dev(s["signman"], "signman")
    out.chunk_off = _dev(s["chunk_off"], "chunk_off")
    cap = s["esc_pos"].numel()
    out.esc_capacity = min(cap, s["esc_val"].numel())
    out.esc_pos = _dev(s["esc_pos"], "esc_pos") if cap else None
    out.esc_val = _dev(s["esc_val"], "esc_val") if cap else None
    return out


# ------------------------------------------------------------ sizes (host)

def splitzip_workspace_bytes(n: int, chunk: int = 1024) -> int:
    return int(library().splitzip_workspace_bytes(n, chunk))


def splitzip_num_chunks(n: int, chunk: int) -> int:
    return int(library().splitzip_num_chunks(n, chunk))


def splitzip_codes_bytes(n: int) -> int:
    return int(library().splitzip_codes_bytes(n))


def splitzip_signman_bytes(n: int, fmt: str = "bf16") -> int:
    lib = library()
    return int(lib.splitzip_signman_bytes(n) if fmt == "bf16" else lib.splitzip_signman_bytes_e5m2(n))


def splitzip_compressed_bytes(n: int, chunk: int, n_escapes: int, fmt: str = "bf16") -> int:
    lib = library()
    fn = lib.splitzip_compressed_bytes if fmt == "bf16" else lib.splitzip_compressed_bytes_e5m2
    return int(fn(n, chunk, n_escapes))


def alloc_workspace(n: int, device="cuda") -> torch.Tensor:
    """Zero-filled workspace for n elements (zeroed once; reusable after)."""
    return torch.zeros(splitzip_workspace_bytes(n), dtype=torch.uint8, device=device)


def alloc_streams(n: int, chunk: int, fmt: str = "bf16", esc_capacity: int | None = None,
                  device="cuda") -> dict:
    """Empty stream buffers for n elements (esc_capacity defaults to n // 32 + 1024)."""
    cap = n // 32 + 1024 if esc_capacity is None else esc_capacity
    return {
        "codes": torch.empty(splitzip_codes_bytes(n), dtype=torch.uint8, device=device),
        "signman": torch.empty(splitzip_signman_bytes(n, fmt), dtype=torch.uint8, device=device),
        "esc_pos": torch.empty(cap, dtype=torch.int16, device=device),
        "esc_val": torch.empty(cap, dtype=torch.uint8, device=device),
        "chunk_off": torch.empty(splitzip_num_chunks(n, chunk) + 1, dtype=torch.int32, device=device),
    }


# ----------------------------------------------------------- entry points

def splitzip_calibrate(x: torch.Tensor, workspace: torch.Tensor, fmt: str | None = None,
                       stream=None):
    """Codebook (list of 16 ints) and coverage of x; synchronises the stream."""
    fmt = _fmt_of(x, fmt)
    n = _elements(x, fmt)
    _need(workspace, splitzip_workspace_bytes(n), "workspace")
    cb, cov = Codebook(), ctypes.c_double()
    fn = library().splitzip_calibrate if fmt == "bf16" else library().splitzip_calibrate_e5m2
    _check(fn(_dev(x, "x"), n, ctypes.byref(cb), ctypes.byref(cov),
              _dev(workspace, "workspace"), _stream(stream)), "splitzip_calibrate")
    return list(cb.exp), cov.value


def splitzip_calibrate_async(x: torch.Tensor, cb_out: torch.Tensor, covered_out: torch.Tensor,
                             workspace: torch.Tensor, fmt: str | None = None, stream=None):
    """Device-side calibration: cb_out (16 uint8) and covered_out (1 int64) on the GPU."""
    fmt = _fmt_of(x, fmt)
    n = _elements(x, fmt)
    _need(workspace, splitzip_workspace_bytes(n), "workspace")
    _need(cb_out, 16, "cb_out")
    _need(covered_out, 8, "covered_out")
    fn = (library().splitzip_calibrate_async if fmt == "bf16"
          else library().splitzip_calibrate_async_e5m2)
    _check(fn(_dev(x, "x"), n, _dev(cb_out, "cb_out"), _dev(covered_out, "covered_out"),
              _dev(workspace, "workspace"), _stream(stream)), "splitzip_calibrate_async")


def splitzip_histogram(x: torch.Tensor, workspace: torch.Tensor, fmt: str | None = None,
                       stream=None, out: torch.Tensor | None = None) -> torch.Tensor:
    """Exponent histogram of x on the GPU: int64 tensor of 256 (BF16) / 32 (E5M2)
    counts; asynchronous."""
    fmt = _fmt_of(x, fmt)
    n = _elements(x, fmt)
    _need(workspace, splitzip_workspace_bytes(n), "workspace")
    if out is None:
        out = torch.empty(256 if fmt == "bf16" else 32, dtype=torch.int64, device=x.device)
    _need(out, 8 * (256 if fmt == "bf16" else 32), "out")
    fn = library().splitzip_histogram if fmt == "bf16" else library().splitzip_histogram_e5m2
    _check(fn(_dev(x, "x"), n, _dev(out, "out"), _dev(workspace, "workspace"),
              _stream(stream)), "splitzip_histogram")
    return out


def splitzip_encode(x: torch.Tensor, chunk: int, codebook, streams: dict,
                    workspace: torch.Tensor, fmt: str | None = None, stream=None):
    """Enqueue one encode of x into `streams` (see alloc_streams); asynchronous."""
    fmt = _fmt_of(x, fmt)
    n = _elements(x, fmt)
    fn = library().splitzip_encode if fmt == "bf16" else library().splitzip_encode_e5m2
    if n and chunk > 0:
        _need_streams(streams, n, chunk, fmt)
        _need(workspace, splitzip_workspace_bytes(n, chunk), "workspace")
    s = _streams(streams)
    _check(fn(_dev(x, "x"), n, chunk, ctypes.byref(_codebook(codebook)),
              ctypes.byref(s), _dev(workspace, "workspace"), _stream(stream)), "splitzip_encode")


def splitzip_encode_test(x, chunk, codebook, streams, workspace, fmt=None, stream=None,
                         spin_limit=0, flags=0):
    """splitzip_encode with the test controls of include/splitzip_testing.h."""
    fmt = _fmt_of(x, fmt)
    n = _elements(x, fmt)
    if n and chunk > 0:
        _need_streams(streams, n, chunk, fmt)
        _need(workspace, splitzip_workspace_bytes(n, chunk), "workspace")
    s, o = _streams(streams), EncodeTestOpts(spin_limit, flags)
    _check(library().splitzip_encode_test(
        _dev(x, "x"), n, chunk, ctypes.byref(_codebook(codebook)), ctypes.byref(s),
        _dev(workspace, "workspace"), _stream(stream), int(fmt == "e5m2"), ctypes.byref(o)),
        "splitzip_encode_test")


def splitzip_encode_status(workspace: torch.Tensor, stream=None):
    """(status, E) of the last finished encode on this workspace; synchronises."""
    e = ctypes.c_uint64()
    st = library().splitzip_encode_status(_dev(workspace, "workspace"), _stream(stream),
                                          ctypes.byref(e))
    return int(st), int(e.value)


def splitzip_decode(streams: dict, n: int, chunk: int, codebook, y: torch.Tensor,
                    fmt: str = "bf16", stream=None, n_escapes: int | None = None):
    """Enqueue one decode of `streams` into y (n elements); asynchronous.

    n_escapes bounds the escape entries the kernel may read (default: the
    capacity of the escape buffers)."""
    if n > 0 and chunk > 0:
        _need_streams(streams, n, chunk, fmt)
        _need(y, n * _ELEM[fmt], "y")
    s = _streams(streams)
    if n_escapes is not None:
        s.esc_capacity = min(s.esc_capacity, n_escapes)
    fn = library().splitzip_decode if fmt == "bf16" else library().splitzip_decode_e5m2
    _check(fn(ctypes.byref(s), n, chunk, ctypes.byref(_codebook(codebook)), _dev(y, "y"),
              _stream(stream)), "splitzip_decode")


def _devcb(cb: torch.Tensor) -> ctypes.c_void_p:
    """A device codebook: 16 uint8 on the GPU, 4-byte aligned (as
    splitzip_calibrate_async writes it)."""
    if cb.dtype != torch.uint8 or cb.numel() < 16:
        raise SplitZipError(ERR_INVALID_ARG, "a device codebook is 16 uint8 values")
    return _dev(cb, "codebook")


def splitzip_encode_devcb(x: torch.Tensor, chunk: int, cb_dev: torch.Tensor, streams: dict,
                          workspace: torch.Tensor, fmt: str | None = None, stream=None):
    """splitzip_encode with the codebook read from device memory (cb_dev, e.g.
    the output of splitzip_calibrate_async); asynchronous.  An invalid device
    codebook is reported by splitzip_encode_status as ERR_INVALID_ARG."""
    fmt = _fmt_of(x, fmt)
    n = _elements(x, fmt)
    fn = library().splitzip_encode_devcb if fmt == "bf16" else library().splitzip_encode_devcb_e5m2
    if n and chunk > 0:
        _need_streams(streams, n, chunk, fmt)
        _need(workspace, splitzip_workspace_bytes(n, chunk), "workspace")
    s = _streams(streams)
    _check(fn(_dev(x, "x"), n, chunk, _devcb(cb_dev), ctypes.byref(s),
              _dev(workspace, "workspace"), _stream(stream)), "splitzip_encode_devcb")


def splitzip_decode_devcb(streams: dict, n: int, chunk: int, cb_dev: torch.Tensor,
                          y: torch.Tensor, fmt: str = "bf16", stream=None,
                          n_escapes: int | None = None):
    """splitzip_decode with the codebook read from device memory; asynchronous."""
    if n > 0 and chunk > 0:
        _need_streams(streams, n, chunk, fmt)
        _need(y, n * _ELEM[fmt], "y")
    s = _streams(streams)
    if n_escapes is not None:
        s.esc_capacity = min(s.esc_capacity, n_escapes)
    fn = library().splitzip_decode_devcb if fmt == "bf16" else library().splitzip_decode_devcb_e5m2
    _check(fn(ctypes.byref(s), n, chunk, _devcb(cb_dev), _dev(y, "y"), _stream(stream)),
           "splitzip_decode_devcb")


def splitzip_version() -> int:
    return int(library().splitzip_version())


# --------------------------------------------------- payloads and transfers

def _ptr(t: torch.Tensor, what: str) -> ctypes.c_void_p:
    """Pointer of a contiguous tensor on the GPU or in host memory."""
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def splitzip_payload_bytes_bound(n: int, chunk: int, slice_elems: int, n_escapes: int,
                                 fmt: str = "bf16") -> int:
    return int(library().splitzip_payload_bytes_bound(FORMATS[fmt], n, chunk, slice_elems,
                                                      n_escapes))


def splitzip_payload_parse(payload: torch.Tensor, nbytes: int | None = None):
    """(info dict, list of slice dicts) of a host payload; raises if malformed."""
    if payload.is_cuda or payload.dtype != torch.uint8:
        raise ValueError("a payload is a host uint8 tensor")
    nbytes = payload.numel() if nbytes is None else nbytes
    info = PayloadInfo()
    _check(library().splitzip_payload_parse(_ptr(payload, "payload"), nbytes, ctypes.byref(info),
                                            None, 0), "splitzip_payload_parse")
    entries = (SliceEntry * info.num_slices)()
    _check(library().splitzip_payload_parse(_ptr(payload, "payload"), nbytes, ctypes.byref(info),
                                            entries, info.num_slices), "splitzip_payload_parse")
    d = {k: int(getattr(info, k)) for k, _ in PayloadInfo._fields_}
    d["fmt"] = {v: k for k, v in FORMATS.items()}[d["format"]]
    sl = [{"n": int(e.n), "n_escapes": int(e.n_escapes), "off_dense": int(e.off_dense),
           "off_escapes": int(e.off_escapes), "codebook": list(e.cb.exp)} for e in entries]
    return d, sl


def splitzip_transfer_scratch_bytes(slice_elems: int, chunk: int, fmt: str = "bf16") -> int:
    return int(library().splitzip_transfer_scratch_bytes(FORMATS[fmt], slice_elems, chunk))


def alloc_transfer_scratch(slice_elems: int, chunk: int, fmt: str = "bf16",
                           device="cuda") -> torch.Tensor:
    return torch.empty(splitzip_transfer_scratch_bytes(slice_elems, chunk, fmt),
                       dtype=torch.uint8, device=device)


def _cbs(codebooks) -> tuple:
    """A shared codebook (16 ints), one codebook per slice, or None (every
    slice calibrated on the device)."""
    if codebooks is None:
        return None, 0
    seq = codebooks.tolist() if hasattr(codebooks, "tolist") else list(codebooks)
    if len(seq) == 16 and all(isinstance(v, int) for v in seq):
        seq = [seq]
    arr = (Codebook * len(seq))()
    for i, cb in enumerate(seq):
        arr[i] = _codebook(cb)
    return arr, len(seq)


def _three_streams(streams):
    if streams is None:
        raise ValueError("three distinct CUDA streams are needed (compute, h2d, d2h)")
    return [ctypes.c_void_p(s.cuda_stream) for s in streams]


def _events(ready_events):
    """A C array of the events' cudaEvent_t handles (None for no events)."""
    if not ready_events:
        return None, 0
    arr = (ctypes.c_void_p * len(ready_events))()
    for i, ev in enumerate(ready_events):
        h = ev.cuda_event
        if not h:   # a torch event is created lazily, on its first record
            raise ValueError(f"ready event {i} has not been recorded")
        arr[i] = h
    return arr, len(ready_events)


def splitzip_encode_to_host(x: torch.Tensor, chunk: int, codebooks, slice_elems: int,
                            payload: torch.Tensor, scratch: torch.Tensor, streams,
                            fmt: str | None = None, ready_events=None):
    """Encode x (GPU or pinned host tensor) slice by slice into the host uint8
    tensor `payload`.  Returns (status, payload bytes); status is OK or
    ERR_ESCAPE_OVERFLOW (payload too small: the bytes needed are returned).
    codebooks: one shared codebook, one per slice, or None to calibrate every
    slice on the device just before it is encoded.
    ready_events: None, or one torch.cuda.Event per slice, each already
    recorded on the producing stream; slice i is read only after the work of
    that record completes (a tensor still being produced)."""
    fmt = _fmt_of(x, fmt)
    n = _elements(x, fmt)
    arr, k = _cbs(codebooks)
    evs, ne = _events(ready_events)
    nbytes = ctypes.c_uint64()
    sc, sh, sd = _three_streams(streams)
    st = library().splitzip_encode_to_host_events(
        _ptr(x, "x"), n, FORMATS[fmt], chunk, arr, k, slice_elems, _ptr(payload, "payload"),
        _nbytes(payload), ctypes.byref(nbytes), _dev(scratch, "scratch"), _nbytes(scratch),
        sc, sh, sd, evs, ne)
    if st not in (OK, ERR_ESCAPE_OVERFLOW):
        _check(st, "splitzip_encode_to_host")
    return int(st), int(nbytes.value)


def splitzip_decode_from_host(payload: torch.Tensor, nbytes: int, y: torch.Tensor,
                              scratch: torch.Tensor, streams):
    """Decode a host payload into y (GPU or pinned host tensor); synchronous."""
    _need(payload, nbytes, "payload")
    if not payload.is_cuda:
        # The library checks y's element count against the payload; its element
        # width (which the payload's format fixes) only the tensor knows.
        info = PayloadInfo()
        if library().splitzip_payload_parse(_ptr(payload, "payload"), nbytes,
                                            ctypes.byref(info), None, 0) == OK:
            _elements(y, {v: k for k, v in FORMATS.items()}[int(info.format)], "y")
    sc, sh, sd = _three_streams(streams)
    _check(library().splitzip_decode_from_host(
        _ptr(payload, "payload"), nbytes, _ptr(y, "y"), y.numel(), _dev(scratch, "scratch"),
        _nbytes(scratch), sc, sh, sd), "splitzip_decode_from_host")


def encode_to_host(x: torch.Tensor, chunk: int, codebooks, slice_elems: int, scratch, streams,
                   fmt: str | None = None, payload: torch.Tensor | None = None,
                   ready_events=None):
    """splitzip_encode_to_host into a pinned payload, grown once if too small.
    Returns (payload tensor, payload bytes)."""
    fmt = _fmt_of(x, fmt)
    n = x.numel()
    if payload is None:
        cap = splitzip_payload_bytes_bound(n, chunk, slice_elems, n // 128 + 4096, fmt)
        payload = torch.empty(cap, dtype=torch.uint8).pin_memory()
    st, nbytes = splitzip_encode_to_host(x, chunk, codebooks, slice_elems, payload, scratch,
                                         streams, fmt, ready_events)
    if st == ERR_ESCAPE_OVERFLOW:
        payload = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        st, nbytes = splitzip_encode_to_host(x, chunk, codebooks, slice_elems, payload, scratch,
                                             streams, fmt, ready_events)
        _check(st, "splitzip_encode_to_host")
    return payload, nbytes


# ------------------------------------------------------------- codec object

@dataclass
class Encoded:
    """One encoded tensor: device streams plus what decode needs to restore it."""
    fmt: str
    shape: tuple
    dtype: torch.dtype
    n: int
    chunk: int
    codebook: list
    streams: dict
    n_escapes: int

    @property
    def compressed_bytes(self) -> int:
        """Compressed size from the library's closed form (codebook not counted)."""
        return splitzip_compressed_bytes(self.n, self.chunk, self.n_escapes, self.fmt)

    @property
    def ratio(self) -> float:
        return self.n * (2 if self.fmt == "bf16" else 1) / self.compressed_bytes


class ChunkLocalSplitZipGPU:
    """Stateful codec with a calibrated codebook, as in the pages' Codec API:
    ``coverage = codec.calibrate(x)``, ``enc = codec.encode(x)``,
    ``y = codec.decode(enc)``, ``enc.compressed_bytes``."""

    def __init__(self, device="cuda", chunk_size: int = 1024, fmt: str = "bf16"):
        if fmt not in ("bf16", "e5m2"):
            raise ValueError("fmt is 'bf16' or 'e5m2'")
        self.device = torch.device(device)
        self.chunk_size = int(chunk_size)
        self.fmt = fmt
        self.codebook = None
        self._ws = None

    def _workspace(self, n: int) -> torch.Tensor:
        need = splitzip_workspace_bytes(n, self.chunk_size)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def _flat(self, x: torch.Tensor) -> torch.Tensor:
        want = torch.bfloat16 if self.fmt == "bf16" else torch.float8_e5m2
        if x.dtype != want:
            raise TypeError(f"expected {want}, got {x.dtype}")
        return x.reshape(-1) if x.is_contiguous() else x.contiguous().reshape(-1)

    def calibrate(self, x: torch.Tensor) -> float:
        flat = self._flat(x)
        self.codebook, coverage = splitzip_calibrate(flat, self._workspace(flat.numel()),
                                                     self.fmt)
        return coverage

    def encode(self, x: torch.Tensor, esc_capacity: int | None = None, stream=None) -> Encoded:
        """Encodes x and synchronises once to read E; retries with the exact
        escape capacity if the first guess overflowed."""
        if self.codebook is None:
            raise RuntimeError("calibrate() first")
        flat = self._flat(x)
        n = flat.numel()
        ws = self._workspace(n)
        streams = alloc_streams(n, self.chunk_size, self.fmt, esc_capacity, self.device)
        splitzip_encode(flat, self.chunk_size, self.codebook, streams, ws, self.fmt, stream)
        status, E = splitzip_encode_status(ws, stream)
        if status == ERR_ESCAPE_OVERFLOW:
            streams = alloc_streams(n, self.chunk_size, self.fmt, E, self.device)
            splitzip_encode(flat, self.chunk_size, self.codebook, streams, ws, self.fmt, stream)
            status, E = splitzip_encode_status(ws, stream)
        _check(status, "encode")
        streams["esc_pos"] = streams["esc_pos"][:E]
        streams["esc_val"] = streams["esc_val"][:E]
        return Encoded(self.fmt, tuple(x.shape), x.dtype, n, self.chunk_size,
                       list(self.codebook), streams, E)

    def decode(self, enc: Encoded, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty(enc.shape, dtype=enc.dtype, device=self.device)
        splitzip_decode(enc.streams, enc.n, enc.chunk, enc.codebook, out.view(-1), enc.fmt,
                        stream, enc.n_escapes)
        return out
