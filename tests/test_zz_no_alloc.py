"""The no-allocation BF16 encode (splitzip_encode_noalloc).

It exists for callers that cannot allocate device memory when they encode --
for instance a KV-transfer hook inside a serving engine whose memory pool
already owns the GPU, or a plugin that is handed only its input and output
buffers -- so its scratch lives in a fixed array inside the library instead of
a caller workspace.  Here it is called through the C ABI and checked against
the regular entry point (splitzip_encode with a workspace): the streams must be
identical byte for byte (the codec is exact integer work), on two calls in a
row, the second of which starts from the array exactly as the first left it.

This file is collected last on purpose, so that a run that stops at the first
failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

from lossless_bf16_kv_gb300 import splitzip as sz
from lossless_bf16_kv_gb300 import synth
from tests.gpu_helpers import ensure_library, gpu_calibrate, gpu_encode

pytestmark = pytest.mark.gpu
DEV = "cuda"
KEYS = ("codes", "signman", "chunk_off", "esc_pos", "esc_val")


def _noalloc(x: torch.Tensor, chunk: int, cb, esc_capacity: int):
    lib = sz.library()
    n = x.numel()
    st = sz.alloc_streams(n, chunk, "bf16", esc_capacity, DEV)
    status_dev = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    rc = lib.splitzip_encode_noalloc(ctypes.c_void_p(x.data_ptr()), n, chunk,
                                     ctypes.byref(sz._codebook(cb)),
                                     ctypes.byref(sz._streams(st)),
                                     ctypes.c_void_p(status_dev.data_ptr()), sz._stream(None))
    assert rc == sz.OK
    torch.cuda.synchronize()
    E = int(st["chunk_off"][-1].item())
    stored = min(E, esc_capacity)
    host = {"codes": st["codes"].cpu().numpy(), "signman": st["signman"].cpu().numpy(),
            "chunk_off": st["chunk_off"].cpu().numpy().view(np.uint32),
            "esc_pos": st["esc_pos"][:stored].cpu().numpy().view(np.uint16),
            "esc_val": st["esc_val"][:stored].cpu().numpy()}
    return host, int(status_dev.item()), E


def test_noalloc_encode_matches_encode_twice():
    ensure_library()
    cb, _ = gpu_calibrate(synth.kv_cache(1, 256, seed=1, device=DEV))
    inputs = [synth.kv_cache(1, 2048, seed=0, device=DEV).reshape(-1)[:3_000_017],
              synth.kv_cache(1, 700, seed=4, device=DEV).reshape(-1)[:1_000_003]]
    for call, x in enumerate(inputs):  # two calls in a row, different sizes
        ref, status, E, _ = gpu_encode(x, 1024, cb, esc_capacity=x.numel())
        assert status == sz.OK
        got, bits, E_got = _noalloc(x, 1024, cb, esc_capacity=x.numel())
        assert bits == 0, f"call {call}: status bits {bits}"
        assert E_got == E
        for k in KEYS:
            np.testing.assert_array_equal(got[k], ref[k], err_msg=f"call {call}: {k}")


def test_noalloc_reports_overflow_and_size_limit():
    ensure_library()
    cb, _ = gpu_calibrate(synth.kv_cache(1, 256, seed=1, device=DEV))
    x = synth.kv_cache(1, 512, seed=2, device=DEV).reshape(-1)
    ref, _, E, _ = gpu_encode(x, 1024, cb, esc_capacity=x.numel())
    assert E > 10
    got, bits, E_got = _noalloc(x, 1024, cb, esc_capacity=10)
    assert bits == 1 and E_got == E
    for k in ("codes", "signman", "chunk_off"):
        np.testing.assert_array_equal(got[k], ref[k])
    np.testing.assert_array_equal(got["esc_pos"], ref["esc_pos"][:10])
    # Above the fixed scratch size: rejected before anything is enqueued.
    lib = sz.library()
    st = sz.alloc_streams(1024, 1024, "bf16", 16, DEV)
    rc = lib.splitzip_encode_noalloc(ctypes.c_void_p(x.data_ptr()), (1 << 31) + 1, 1024,
                                     ctypes.byref(sz._codebook(cb)),
                                     ctypes.byref(sz._streams(st)), None, sz._stream(None))
    assert rc == sz.ERR_TOO_LARGE
