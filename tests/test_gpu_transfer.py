"""Pipelined transfers through host payloads (include/splitzip_transfer.h),
on the GPU through the C ABI: every payload byte equals the oracle's payload
of the same slices, and decoding it gives back the input bit for bit, with
input and output on the device or in pinned host memory."""
import numpy as np
import pytest
import torch

import oracle
from oracle import payload as op
from lossless_bf16_kv_gb300 import splitzip as sz
from lossless_bf16_kv_gb300 import synth

from .gpu_helpers import ensure_library, host_bits

pytestmark = pytest.mark.gpu


def _kv(fmt, n, seed):
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    layers = max(1, -(-n // (2 * 256 * 1024)))
    return synth.kv_cache(layers, 256, seed=seed, device="cuda", dtype=dt).reshape(-1)[:n].clone()


def _streams():
    return [torch.cuda.Stream() for _ in range(3)]


def _check_roundtrip(x, fmt, chunk, se, cbs, where):
    ensure_library()
    bits = host_bits(x)
    scratch = sz.alloc_transfer_scratch(se, chunk, fmt)
    streams = _streams()
    src = x if where == "device" else x.cpu().pin_memory()
    payload, nbytes = sz.encode_to_host(src, chunk, cbs, se, scratch, streams, fmt)
    ref = op.write(bits, fmt, chunk, se, cbs)
    assert nbytes == len(ref)
    assert payload[:nbytes].numpy().tobytes() == ref
    y = torch.empty_like(x)
    sz.splitzip_decode_from_host(payload, nbytes, y, scratch, streams)
    assert np.array_equal(host_bits(y), bits)
    yh = torch.empty(x.shape, dtype=x.dtype).pin_memory()
    sz.splitzip_decode_from_host(payload, nbytes, yh, scratch, streams)
    assert np.array_equal(host_bits(yh), bits)


@pytest.mark.parametrize("where", ["device", "host"])
@pytest.mark.parametrize("fmt,n,chunk,se", [
    ("bf16", (1 << 20) + 3 * 1024 + 5, 1024, 1 << 18),   # five slices, the last ragged
    ("bf16", 300000, 256, 65536),
    ("bf16", 1000, 8, 1024),                              # one slice
    ("e5m2", (1 << 20) + 77, 1024, 1 << 17),
    ("e5m2", 50000, 64, 4096),
])
def test_transfer_matches_oracle(fmt, n, chunk, se, where):
    x = _kv(fmt, n, seed=n % 97)
    cal = _kv(fmt, min(n, 1 << 18), seed=1)
    cb = [int(c) for c in oracle.calibrate(host_bits(cal), fmt)[0]]
    _check_roundtrip(x, fmt, chunk, se, cb, where)


def test_per_slice_codebooks():
    fmt, se, chunk = "bf16", 1 << 17, 1024
    x = _kv(fmt, 5 * se - 100, seed=3)
    bits = host_bits(x)
    cbs = [[int(c) for c in oracle.calibrate(bits[i:i + se], fmt)[0]] for i in range(0, x.numel(), se)]
    _check_roundtrip(x, fmt, chunk, se, cbs, "device")


def test_many_escapes():
    """Student-t values spread over 2^40 of scale: most exponents escape an
    N(0,1) codebook, so escape regions dominate the payload."""
    ensure_library()
    x = synth.student_t_scaled_bf16((512, 1000), seed=4, device="cuda").reshape(-1)
    cb = [int(c) for c in oracle.calibrate(host_bits(synth.normal_bf16((256, 1024), 1, "cuda")), "bf16")[0]]
    _check_roundtrip(x, "bf16", 1024, 1 << 16, cb, "device")


def test_small_payload_reports_the_size_needed():
    ensure_library()
    fmt, chunk, se = "bf16", 1024, 1 << 16
    x = synth.student_t_scaled_bf16((256, 1024), seed=5, device="cuda").reshape(-1)
    cb = [int(c) for c in oracle.calibrate(host_bits(synth.normal_bf16((256, 1024), 1, "cuda")), "bf16")[0]]
    ref = op.write(host_bits(x), fmt, chunk, se, cb)
    head, _ = op.read(ref)
    dense_end = min(s["off_escapes"] for s in op.read(ref)[1])
    scratch, streams = sz.alloc_transfer_scratch(se, chunk, fmt), _streams()
    small = torch.empty(dense_end + 16, dtype=torch.uint8).pin_memory()
    st, need = sz.splitzip_encode_to_host(x, chunk, cb, se, small, scratch, streams, fmt)
    assert st == sz.ERR_ESCAPE_OVERFLOW and need == len(ref) == head["total_bytes"]
    payload, nbytes = sz.encode_to_host(x, chunk, cb, se, scratch, streams, fmt, payload=small)
    assert payload[:nbytes].numpy().tobytes() == ref


def test_decode_checks_its_arguments():
    ensure_library()
    fmt, chunk, se = "bf16", 1024, 1 << 16
    x = _kv(fmt, 100000, seed=6)
    cb = [int(c) for c in oracle.calibrate(host_bits(x), fmt)[0]]
    scratch, streams = sz.alloc_transfer_scratch(se, chunk, fmt), _streams()
    payload, nbytes = sz.encode_to_host(x, chunk, cb, se, scratch, streams, fmt)
    y = torch.empty(x.numel() - 1, dtype=x.dtype, device="cuda")
    with pytest.raises(sz.SplitZipError):
        sz.splitzip_decode_from_host(payload, nbytes, y, scratch, streams)   # wrong n
    bad = payload.clone()
    bad[0] = ord("X")
    with pytest.raises(sz.SplitZipError):
        sz.splitzip_decode_from_host(bad, nbytes, torch.empty_like(x), scratch, streams)
    with pytest.raises(sz.SplitZipError):
        sz.splitzip_decode_from_host(payload, nbytes, torch.empty_like(x), scratch[:1024], streams)


def test_encode_checks_its_arguments():
    """Rejected on the host before any work is enqueued."""
    ensure_library()
    fmt, chunk, se = "bf16", 1024, 1 << 16
    x = _kv(fmt, 100000, seed=7)
    cb = [int(c) for c in oracle.calibrate(host_bits(x), fmt)[0]]
    scratch, streams = sz.alloc_transfer_scratch(se, chunk, fmt), _streams()
    payload = torch.empty(sz.splitzip_payload_bytes_bound(x.numel(), chunk, se, x.numel(), fmt),
                          dtype=torch.uint8).pin_memory()
    bad_calls = [
        dict(slice_elems=se + 8),                        # not a multiple of the chunk size
        dict(slice_elems=512),                           # smaller than a chunk
        dict(codebooks=[cb, cb, cb]),                    # two slices: neither one codebook nor one each
        dict(codebooks=[cb[0]] * 16),                    # repeated exponents
        dict(streams=[streams[0], streams[0], streams[2]]),  # streams must differ
        dict(scratch=scratch[: scratch.numel() // 2]),  # scratch too small
    ]
    for bad in bad_calls:
        kw = dict(slice_elems=se, codebooks=cb, streams=streams, scratch=scratch)
        kw.update(bad)
        with pytest.raises(sz.SplitZipError) as err:
            sz.splitzip_encode_to_host(x, chunk, kw["codebooks"], kw["slice_elems"], payload,
                                       kw["scratch"], kw["streams"], fmt)
        assert err.value.status == sz.ERR_INVALID_ARG, bad


def test_payload_must_be_host_memory():
    ensure_library()
    fmt, chunk, se = "bf16", 1024, 1 << 16
    x = _kv(fmt, 100000, seed=8)
    cb = [int(c) for c in oracle.calibrate(host_bits(x), fmt)[0]]
    scratch, streams = sz.alloc_transfer_scratch(se, chunk, fmt), _streams()
    payload, nbytes = sz.encode_to_host(x, chunk, cb, se, scratch, streams, fmt)
    on_device = payload.cuda()
    with pytest.raises(sz.SplitZipError) as err:
        sz.splitzip_encode_to_host(x, chunk, cb, se, on_device, scratch, streams, fmt)
    assert err.value.status == sz.ERR_INVALID_ARG
    with pytest.raises(sz.SplitZipError) as err:
        sz.splitzip_decode_from_host(on_device, nbytes, torch.empty_like(x), scratch, streams)
    assert err.value.status == sz.ERR_INVALID_ARG


@pytest.mark.parametrize("where", ["device", "host"])
@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_encode_waits_for_each_slice_to_be_produced(fmt, where):
    """A producer on its own stream writes the tensor slice by slice, each slice
    after a spin of several milliseconds, and records one event per slice; the
    encode call is issued at once.  Every slice must be read only after its
    event: the payload equals the oracle's payload of the produced data, not of
    the zeros the buffer held when the call was made."""
    ensure_library()
    chunk, se = 1024, 1 << 17
    src = _kv(fmt, 4 * se + 3 * chunk + 9, seed=11)     # five slices, the last ragged
    n = src.numel()
    cb = [int(c) for c in oracle.calibrate(host_bits(src), fmt)[0]]
    x = (torch.zeros_like(src) if where == "device"
         else torch.zeros(src.shape, dtype=src.dtype).pin_memory())
    scratch, streams = sz.alloc_transfer_scratch(se, chunk, fmt), _streams()
    torch.cuda.synchronize()
    producer = torch.cuda.Stream()
    events = []
    with torch.cuda.stream(producer):
        for lo in range(0, n, se):
            torch.cuda._sleep(10_000_000)                # about 5 ms at 2 GHz
            x[lo:lo + se].copy_(src[lo:lo + se], non_blocking=True)
            events.append(torch.cuda.Event())
            events[-1].record(producer)
    payload, nbytes = sz.encode_to_host(x, chunk, cb, se, scratch, streams, fmt,
                                        ready_events=events)
    bits = host_bits(src)
    assert payload[:nbytes].numpy().tobytes() == op.write(bits, fmt, chunk, se, cb)
    y = torch.empty_like(src)
    sz.splitzip_decode_from_host(payload, nbytes, y, scratch, streams)
    assert np.array_equal(host_bits(y), bits)


def test_ready_events_are_checked():
    """One event per slice or none: other counts, and events never recorded,
    are rejected before any work is enqueued."""
    ensure_library()
    fmt, chunk, se = "bf16", 1024, 1 << 16
    x = _kv(fmt, 3 * se, seed=12)
    cb = [int(c) for c in oracle.calibrate(host_bits(x), fmt)[0]]
    scratch, streams = sz.alloc_transfer_scratch(se, chunk, fmt), _streams()
    payload = torch.empty(sz.splitzip_payload_bytes_bound(x.numel(), chunk, se, x.numel(), fmt),
                          dtype=torch.uint8).pin_memory()
    events = [torch.cuda.Event() for _ in range(4)]
    for ev in events:
        ev.record()
    for evs in (events[:2], events):                     # three slices
        with pytest.raises(sz.SplitZipError) as err:
            sz.splitzip_encode_to_host(x, chunk, cb, se, payload, scratch, streams, fmt,
                                       ready_events=evs)
        assert err.value.status == sz.ERR_INVALID_ARG
    with pytest.raises(ValueError):
        sz.splitzip_encode_to_host(x, chunk, cb, se, payload, scratch, streams, fmt,
                                   ready_events=[torch.cuda.Event()] * 3)
    st, nbytes = sz.splitzip_encode_to_host(x, chunk, cb, se, payload, scratch, streams, fmt,
                                            ready_events=events[:3])
    assert st == sz.OK
    assert payload[:nbytes].numpy().tobytes() == op.write(host_bits(x), fmt, chunk, se, cb)
