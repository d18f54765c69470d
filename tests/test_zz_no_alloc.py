"""The no-allocation BF16 encode (splitzip_encode_noalloc).

It exists for callers that cannot allocate device memory when they encode --
for instance a KV-transfer hook inside a serving engine whose memory pool
already owns the GPU, or a plugin that is handed only its input and output
buffers -- so its scratch lives in a fixed array inside the library instead of
a caller workspace.  Here it is called through the C ABI and checked against
the regular entry point (splitzip_encode with a workspace): the streams must be
identical byte for byte (the codec is exact integer work), on two calls in a
row, the second of which starts from the array exactly as the first left it.

The streams are also compared directly with the oracle's (several chunk
sizes, ragged element counts), and across a device reset, after which the
library's fixed array lives in a new context and its address is looked up
again.

This file is collected last on purpose, so that a run that stops at the first
failure has run every other test before it.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_kv_gb300 import splitzip as sz
from lossless_bf16_kv_gb300 import synth
from tests.gpu_helpers import assert_streams_equal, ensure_library, gpu_calibrate, gpu_encode, host_bits

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


@pytest.mark.parametrize("n,chunk", [(1_000_003, 8), (2_500_001, 1000), (777_777, 4096),
                                     (3 * 65536 + 5, 65536), (5, 8)])
def test_noalloc_encode_matches_oracle(n, chunk):
    """The no-allocation encode's streams equal the oracle's, at chunk sizes
    other than 1024 and element counts that end in a partial chunk and tile."""
    ensure_library()
    cal = synth.kv_cache(1, 256, seed=1, device=DEV)
    cb, _ = oracle.calibrate(host_bits(cal), "bf16")
    x = synth.kv_cache(1, -(-n // 2048), seed=n % 31, device=DEV).reshape(-1)[:n].contiguous()
    ref = oracle.encode(host_bits(x), chunk, cb, "bf16")
    got, bits, E = _noalloc(x, chunk, cb, esc_capacity=n)
    assert bits == 0
    got["n_escapes"] = E
    assert_streams_equal(got, ref, f"noalloc n={n} chunk={chunk}")


def test_noalloc_encode_after_device_reset(tmp_path):
    """A plain C program encodes, resets the device (a new context, in which
    the library's fixed array may sit elsewhere) and encodes again: both
    calls succeed and both equal the oracle's streams.  It runs in a process of
    its own, so this process's context is untouched."""
    from tests.test_c_program import compile_program
    ensure_library()
    n, chunk = 1_500_007, 1024
    x = synth.kv_cache(1, 800, seed=9, device="cpu").reshape(-1)[:n]
    cal = synth.kv_cache(1, 128, seed=1, device="cpu").reshape(-1)
    xb = synth.raw_bits(x).numpy().view(np.uint16)
    cb, _ = oracle.calibrate(synth.raw_bits(cal).numpy().view(np.uint16), "bf16")
    xb.tofile(tmp_path / "x.bin")
    cb.tofile(tmp_path / "cb.bin")
    exe = compile_program(tmp_path, os.path.join(os.path.dirname(__file__), "c_noalloc_reset.c"))
    prefix = str(tmp_path / "out")
    r = subprocess.run([exe, str(tmp_path / "x.bin"), str(tmp_path / "cb.bin"), str(chunk), prefix],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    fields = dict(kv.split("=") for kv in r.stdout.split())
    ref = oracle.encode(xb, chunk, cb, "bf16")
    for rnd in (0, 1):
        assert int(fields[f"status{rnd}"]) == 0
        assert int(fields[f"E{rnd}"]) == ref["n_escapes"]
        for name, dtype in (("codes", np.uint8), ("signman", np.uint8), ("esc_pos", np.uint16),
                            ("esc_val", np.uint8), ("chunk_off", np.uint32)):
            got = np.fromfile(f"{prefix}.{rnd}.{name}", dtype)
            assert np.array_equal(got, ref[name]), f"round {rnd}: {name} differs"
