"""Error paths through the C ABI on a GPU: argument checks, escape overflow,
and the bounded look-back wait made to run out on purpose (no fault, trap or
hang: the kernel gives up after a short poll limit and reports a status)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_kv_gb300 import splitzip as sz
from lossless_bf16_kv_gb300 import synth
from tests.gpu_helpers import (assert_streams_equal, ensure_library, gpu_calibrate, gpu_encode,
                               host_bits)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(n=100_000, fmt="bf16"):
    ensure_library()
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    x = synth.student_t_scaled_bf16((n,), seed=1, device=DEV).float().to(dt)
    cb, _ = gpu_calibrate(synth.kv_cache(1, 16, seed=1, device=DEV, dtype=dt))
    return x, cb


def test_invalid_arguments_are_rejected():
    x, cb = _setup()
    n = x.numel()
    ws = sz.alloc_workspace(n, DEV)
    st = sz.alloc_streams(n, 1024, esc_capacity=n)
    lib = sz.library()
    s = sz._streams(st)
    good_cb = sz._codebook(cb)
    stream = sz._stream(None)
    xp = ctypes.c_void_p(x.data_ptr())
    wp = ctypes.c_void_p(ws.data_ptr())
    inv = sz.ERR_INVALID_ARG
    assert lib.splitzip_encode(xp, n, 1000 + 4, ctypes.byref(good_cb), ctypes.byref(s), wp, stream) == inv
    assert lib.splitzip_encode(xp, n, 65544, ctypes.byref(good_cb), ctypes.byref(s), wp, stream) == inv
    assert lib.splitzip_encode(xp, 0, 1024, ctypes.byref(good_cb), ctypes.byref(s), wp, stream) == inv
    assert lib.splitzip_encode(xp, 1 << 32, 1024, ctypes.byref(good_cb), ctypes.byref(s), wp, stream) == inv
    assert lib.splitzip_encode(None, n, 1024, ctypes.byref(good_cb), ctypes.byref(s), wp, stream) == inv
    assert lib.splitzip_encode(ctypes.c_void_p(x.data_ptr() + 2), n - 8, 1024,
                               ctypes.byref(good_cb), ctypes.byref(s), wp, stream) == inv
    dup = sz._codebook([5] * 16)
    assert lib.splitzip_encode(xp, n, 1024, ctypes.byref(dup), ctypes.byref(s), wp, stream) == inv
    big = sz._codebook(list(range(20, 36)))  # >= 32: not an E5M2 exponent
    assert lib.splitzip_encode_e5m2(xp, n, 1024, ctypes.byref(big), ctypes.byref(s), wp, stream) == inv
    y = torch.empty_like(x)
    assert lib.splitzip_decode(ctypes.byref(s), n, 12, ctypes.byref(good_cb),
                               ctypes.c_void_p(y.data_ptr()), stream) == inv
    assert lib.splitzip_decode(ctypes.byref(s), n, 1024, ctypes.byref(good_cb),
                               ctypes.c_void_p(y.data_ptr() + 8), stream) == inv
    # Nothing was enqueued: a valid call still works afterwards.
    sz.splitzip_encode(x, 1024, cb, st, ws)
    assert sz.splitzip_encode_status(ws)[0] == sz.OK


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_escape_overflow(fmt):
    x, cb = _setup(fmt=fmt)
    xb = host_bits(x)
    ref = oracle.encode(xb, 1024, np.asarray(cb, np.uint8), fmt)
    E = ref["n_escapes"]
    assert E > 200
    gpu, status, E_gpu, _ = gpu_encode(x, 1024, cb, esc_capacity=100)
    assert status == sz.ERR_ESCAPE_OVERFLOW
    assert E_gpu == E
    np.testing.assert_array_equal(gpu["codes"], ref["codes"])
    np.testing.assert_array_equal(gpu["signman"], ref["signman"])
    np.testing.assert_array_equal(gpu["chunk_off"], ref["chunk_off"])
    np.testing.assert_array_equal(gpu["esc_pos"], ref["esc_pos"][:100])
    np.testing.assert_array_equal(gpu["esc_val"], ref["esc_val"][:100])
    # The next encode on the same workspace reports OK again.
    again, status, _, _ = gpu_encode(x, 1024, cb, esc_capacity=E)
    assert status == sz.OK
    assert_streams_equal(again, ref, "after overflow")


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_lookback_wait_gives_up(fmt):
    """The single-launch pipeline's first tile never publishes its prefix;
    its successor polls 2000 times, records TIMEOUT and returns.  The context
    stays usable and the next call on the workspace is correct.  (The default
    three-launch encode has no waits to run out.)"""
    engine = "pipelined"
    n = 40_000
    x, cb = _setup(n=n, fmt=fmt)
    ws = sz.alloc_workspace(n, DEV)
    st = sz.alloc_streams(n, 1024, fmt, esc_capacity=n)
    flags = sz.TEST_STALL_FIRST_TILE | (sz.TEST_PIPELINED if engine == "pipelined" else 0)
    sz.splitzip_encode_test(x, 1024, cb, st, ws, fmt, spin_limit=2000, flags=flags)
    status, _ = sz.splitzip_encode_status(ws)
    assert status == sz.ERR_TIMEOUT
    # Same workspace, normal call: correct again.
    ref = oracle.encode(host_bits(x), 1024, np.asarray(cb, np.uint8), fmt)
    gpu, status, _, _ = gpu_encode(x, 1024, cb, esc_capacity=n, ws=ws, engine=engine)
    assert status == sz.OK
    assert_streams_equal(gpu, ref, "after timeout")


def test_codec_object_api():
    """The pages' Codec API shape: calibrate -> coverage, encode -> encoded with
    compressed_bytes, decode -> bitwise-identical tensor."""
    x = synth.normal_bf16((1024, 4096), seed=0, device=DEV)
    codec = sz.ChunkLocalSplitZipGPU(device=DEV, chunk_size=1024)
    coverage = codec.calibrate(x)
    assert 0.99 < coverage <= 1.0
    enc = codec.encode(x, esc_capacity=1)  # forces the overflow retry path
    y = codec.decode(enc)
    assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    ref = oracle.encode(host_bits(x), 1024, np.asarray(codec.codebook, np.uint8))
    assert enc.n_escapes == ref["n_escapes"]
    assert enc.compressed_bytes == oracle.compressed_bytes(x.numel(), 1024, ref["n_escapes"])
    assert enc.ratio <= 4 / 3


def test_binding_rejects_undersized_buffers():
    """The C ABI takes plain pointers, so the Python binding checks every buffer
    against n (and the element width against the format) before anything is
    enqueued."""
    ensure_library()
    n, chunk = 100_000, 1024
    x = torch.ones(n, dtype=torch.bfloat16, device="cuda")
    cb = list(range(120, 136))
    ws = sz.alloc_workspace(n, x.device)
    st = sz.alloc_streams(n, chunk, "bf16", device=x.device)
    small = {k: (v[: v.numel() // 2] if k in ("codes", "signman", "chunk_off") else v)
             for k, v in st.items()}
    bad_calls = [
        lambda: sz.splitzip_encode(x, chunk, cb, small, ws, "bf16"),
        lambda: sz.splitzip_encode(x, chunk, cb, st, ws[:4096], "bf16"),
        lambda: sz.splitzip_encode(x.view(torch.uint8), chunk, cb, st, ws, "bf16"),
        lambda: sz.splitzip_decode(st, n, chunk, cb, torch.empty(n - 1, dtype=x.dtype,
                                                                 device=x.device), "bf16"),
        lambda: sz.splitzip_decode(small, n, chunk, cb, torch.empty_like(x), "bf16"),
        lambda: sz.splitzip_calibrate(x, ws[:4096], "bf16"),
        lambda: sz.splitzip_histogram(x, ws, "bf16", out=torch.empty(8, dtype=torch.int64,
                                                                     device=x.device)),
    ]
    for i, call in enumerate(bad_calls):
        with pytest.raises(sz.SplitZipError) as err:
            call()
        assert err.value.status == sz.ERR_INVALID_ARG, i
