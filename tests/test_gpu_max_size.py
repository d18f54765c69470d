"""The largest tensor the format allows (n = 2^32 - 1 elements, chunk_off is
uint32) on the GPU through the C ABI: a bit-exact round trip, and every stream
byte-identical to the oracle's in chunk-aligned windows at the start, in the
middle and at the ragged end (the oracle encodes windows of whole chunks on
its own: positions are chunk-local and offsets are differences)."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_kv_gb300 import splitzip as sz

from .gpu_helpers import ensure_library, host_bits

pytestmark = pytest.mark.gpu

N = (1 << 32) - 1


def _big(fmt: str) -> torch.Tensor:
    g = torch.Generator(device="cuda").manual_seed(123)
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    x = torch.empty(N, dtype=dt, device="cuda")
    step = 1 << 28
    for s in range(0, N, step):
        m = min(step, N - s)
        v = torch.randn(m, generator=g, device="cuda") * 3
        v[torch.rand(m, generator=g, device="cuda") < 0.002] *= 1000  # rare exponents
        x[s:s + m] = v.to(dt)
    return x


def _windows(chunk: int):
    C = -(-N // chunk)
    return [(0, 3), (C // 2, 2), (C - 3, 3)]  # (first chunk, chunks)


@pytest.mark.parametrize("fmt,chunk", [("bf16", 1024), ("bf16", 65536), ("e5m2", 1024)])
def test_max_size(fmt, chunk):
    ensure_library()
    x = _big(fmt)
    sample = x[: 1 << 24]
    ws = sz.alloc_workspace(N, x.device)
    cb, _ = sz.splitzip_calibrate(sample, ws, fmt)
    st = sz.alloc_streams(N, chunk, fmt, N // 64, x.device)
    sz.splitzip_encode(x, chunk, cb, st, ws, fmt)
    status, E = sz.splitzip_encode_status(ws)
    assert status == sz.OK, status
    chunk_off = st["chunk_off"]
    assert int(chunk_off[-1].item()) & 0xFFFFFFFF == E
    y = torch.empty_like(x)
    sz.splitzip_decode(st, N, chunk, cb, y, fmt, n_escapes=E)
    torch.cuda.synchronize()
    same = torch.equal(x.view(torch.uint8) if fmt == "e5m2" else x.view(torch.int16),
                       y.view(torch.uint8) if fmt == "e5m2" else y.view(torch.int16))
    assert same, "round trip not bit-exact"
    del y
    cbv = np.asarray(cb, np.uint8)
    offs = chunk_off.cpu().numpy().view(np.uint32).astype(np.int64)
    for c0, k in _windows(chunk):
        e0, e1 = c0 * chunk, min(N, (c0 + k) * chunk)
        ref = oracle.encode(host_bits(x[e0:e1]), chunk, cbv, fmt)
        assert np.array_equal(offs[c0:c0 + k + 1] - offs[c0], ref["chunk_off"].astype(np.int64))
        q0, q1 = int(offs[c0]), int(offs[min(c0 + k, len(offs) - 1)])
        assert np.array_equal(st["esc_pos"][q0:q1].cpu().numpy().view(np.uint16), ref["esc_pos"])
        assert np.array_equal(st["esc_val"][q0:q1].cpu().numpy(), ref["esc_val"])
        assert np.array_equal(st["codes"][e0 // 2:(e1 + 1) // 2].cpu().numpy(), ref["codes"])
        if fmt == "bf16":
            sm = st["signman"][e0:e1].cpu().numpy()
        else:
            sm = st["signman"][e0 * 3 // 8:(3 * e1 + 7) // 8].cpu().numpy()
        assert np.array_equal(sm, ref["signman"])
