"""Shared helpers of the GPU tests: run the CUDA path through the C ABI and
compare every stream with the oracle's, byte for byte."""
import numpy as np
import torch

import oracle
from lossless_bf16_kv_gb300 import _build
from lossless_bf16_kv_gb300 import splitzip as sz

_built = False


def ensure_library():
    global _built
    if not _built:
        _build.build_library()
        sz.library()
        _built = True


def host_bits(x: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a BF16 / E5M2 tensor as a flat numpy array."""
    x = x.contiguous().reshape(-1)
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).cpu().numpy().view(np.uint16)
    return x.view(torch.uint8).cpu().numpy()


def fmt_of(x: torch.Tensor) -> str:
    return "bf16" if x.dtype == torch.bfloat16 else "e5m2"


def gpu_calibrate(x: torch.Tensor):
    ensure_library()
    flat = x.reshape(-1)
    ws = sz.alloc_workspace(flat.numel(), flat.device)
    return sz.splitzip_calibrate(flat, ws, fmt_of(x))


def gpu_encode(x: torch.Tensor, chunk: int, cb, esc_capacity=None, ws=None, engine="multi"):
    """Encode on the GPU; returns (host streams dict, status, E, device streams).

    engine "multi" is splitzip_encode (three launches); "pipelined" is the
    single-launch pipeline behind splitzip_encode_noalloc, reached through the
    test entry point."""
    ensure_library()
    flat = x.reshape(-1)
    n = flat.numel()
    fmt = fmt_of(x)
    if ws is None:
        ws = sz.alloc_workspace(n, flat.device)
    st = sz.alloc_streams(n, chunk, fmt, esc_capacity, flat.device)
    if engine == "pipelined":
        sz.splitzip_encode_test(flat, chunk, cb, st, ws, fmt, flags=sz.TEST_PIPELINED)
    else:
        sz.splitzip_encode(flat, chunk, cb, st, ws, fmt)
    status, E = sz.splitzip_encode_status(ws)
    stored = min(E, st["esc_pos"].numel())
    host = {
        "codes": st["codes"].cpu().numpy(),
        "signman": st["signman"].cpu().numpy(),
        "esc_pos": st["esc_pos"][:stored].cpu().numpy().view(np.uint16),
        "esc_val": st["esc_val"][:stored].cpu().numpy(),
        "chunk_off": st["chunk_off"].cpu().numpy().view(np.uint32),
        "n_escapes": E,
    }
    return host, status, E, st


def gpu_decode(streams: dict, n: int, chunk: int, cb, like: torch.Tensor, n_escapes=None):
    ensure_library()
    y = torch.empty(n, dtype=like.dtype, device=like.device)
    sz.splitzip_decode(streams, n, chunk, cb, y, fmt_of(like), n_escapes=n_escapes)
    torch.cuda.synchronize()
    return y


def device_streams(host: dict, device="cuda") -> dict:
    """Upload numpy streams (e.g. the oracle's) as device tensors."""
    return {
        "codes": torch.from_numpy(np.ascontiguousarray(host["codes"])).to(device),
        "signman": torch.from_numpy(np.ascontiguousarray(host["signman"])).to(device),
        "esc_pos": torch.from_numpy(np.ascontiguousarray(host["esc_pos"]).view(np.int16)).to(device),
        "esc_val": torch.from_numpy(np.ascontiguousarray(host["esc_val"])).to(device),
        "chunk_off": torch.from_numpy(np.ascontiguousarray(host["chunk_off"]).view(np.int32)).to(device),
    }


def assert_streams_equal(gpu: dict, ref: dict, what=""):
    assert gpu["n_escapes"] == ref["n_escapes"], f"{what}: E {gpu['n_escapes']} != {ref['n_escapes']}"
    for k in ("codes", "signman", "chunk_off", "esc_pos", "esc_val"):
        a, b = gpu[k], ref[k]
        assert a.shape == b.shape, f"{what}: {k} shape {a.shape} != {b.shape}"
        if not np.array_equal(a, b):
            bad = np.flatnonzero(a != b)
            raise AssertionError(f"{what}: {k} differs at {bad.size} places, first {bad[:8]} "
                                 f"gpu={a[bad[:8]]} oracle={b[bad[:8]]}")


def check_roundtrip(x: torch.Tensor, chunk: int, cb, what=""):
    """Full parity check of one tensor: streams byte-identical to the oracle's,
    GPU decode bit-exact, and both cross-decodes bit-exact."""
    fmt = fmt_of(x)
    xb = host_bits(x)
    ref = oracle.encode(xb, chunk, np.asarray(cb, np.uint8), fmt)
    gpu, status, E, dev = gpu_encode(x, chunk, cb, esc_capacity=ref["n_escapes"] + 16)
    assert status == sz.OK, f"{what}: status {status}"
    assert_streams_equal(gpu, ref, what)
    y = gpu_decode(dev, xb.size, chunk, cb, x, n_escapes=E)
    assert np.array_equal(host_bits(y), xb), f"{what}: GPU decode not bit-exact"
    # oracle streams -> GPU decode
    y2 = gpu_decode(device_streams(ref), xb.size, chunk, cb, x, n_escapes=ref["n_escapes"])
    assert np.array_equal(host_bits(y2), xb), f"{what}: GPU decode of oracle streams"
    # GPU streams -> oracle decode
    y3 = oracle.decode(gpu, xb.size, chunk, np.asarray(cb, np.uint8), fmt)
    assert np.array_equal(y3, xb), f"{what}: oracle decode of GPU streams"
    return ref["n_escapes"]
