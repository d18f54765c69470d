"""Encode and decode captured in a CUDA graph: the library's calls only enqueue
kernels on the caller's stream (no allocation, no synchronisation, a
self-resetting workspace), so one capture can be replayed on new data.  Each
replay's streams must equal the oracle's and its decode must be bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_kv_gb300 import splitzip as sz
from lossless_bf16_kv_gb300 import synth

from tests.gpu_helpers import assert_streams_equal, ensure_library, gpu_calibrate, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_encode_decode_replayed_from_a_cuda_graph(fmt):
    ensure_library()
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    chunk = 1000
    inputs = [synth.kv_cache(1, 512, seed=s, device=DEV, dtype=dt).reshape(-1)[:700_001].clone()
              for s in (5, 6, 7)]
    n = inputs[0].numel()
    cb, _ = gpu_calibrate(synth.kv_cache(1, 64, seed=1, device=DEV, dtype=dt))
    x = inputs[0].clone()                 # the captured input buffer, refilled in place
    y = torch.empty_like(x)
    ws = sz.alloc_workspace(n, DEV)
    st = sz.alloc_streams(n, chunk, fmt, esc_capacity=n, device=DEV)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):         # warm-up outside the capture
        for _ in range(2):
            sz.splitzip_encode(x, chunk, cb, st, ws, fmt)
            sz.splitzip_decode(st, n, chunk, cb, y, fmt)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sz.splitzip_encode(x, chunk, cb, st, ws, fmt)
        sz.splitzip_decode(st, n, chunk, cb, y, fmt)

    for src in reversed(inputs):          # a different tensor each replay
        x.copy_(src)
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        xb = host_bits(src)
        ref = oracle.encode(xb, chunk, np.asarray(cb, np.uint8), fmt)
        status, E = sz.splitzip_encode_status(ws)
        assert status == sz.OK and E == ref["n_escapes"]
        got = {k: v.cpu().numpy() for k, v in st.items()}
        got["n_escapes"] = E
        got["chunk_off"] = got["chunk_off"].view(np.uint32)
        got["esc_pos"] = got["esc_pos"][:E].view(np.uint16)
        got["esc_val"] = got["esc_val"][:E]
        assert_streams_equal(got, ref, f"{fmt} graph replay")
        assert np.array_equal(host_bits(y), xb), f"{fmt} graph replay: decode not bit-exact"
