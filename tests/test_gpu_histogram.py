"""Exponent histograms on the GPU (splitzip_histogram, through the C ABI)
equal the oracle's counts exactly; the statistics report built on them agrees
with real encodes."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_kv_gb300 import report
from lossless_bf16_kv_gb300 import splitzip as sz
from lossless_bf16_kv_gb300 import synth

from .gpu_helpers import ensure_library, host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [1, 7, 8, 9, 15, 17, 4099, 1000003, (1 << 22) + 5])
@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_histogram_matches_oracle(fmt, n):
    ensure_library()
    g = torch.Generator(device="cuda").manual_seed(n)
    if fmt == "bf16":
        x = (torch.randn(n, generator=g, device="cuda") * 7).to(torch.bfloat16)
    else:
        x = torch.randint(0, 256, (n,), generator=g, device="cuda", dtype=torch.uint8).view(torch.float8_e5m2)
    ws = sz.alloc_workspace(n, x.device)
    h = sz.splitzip_histogram(x, ws, fmt)
    h2 = sz.splitzip_histogram(x, ws, fmt)  # the workspace is left ready for the next call
    torch.cuda.synchronize()
    ref = oracle.histogram(host_bits(x), fmt).astype(np.int64)
    assert np.array_equal(h.cpu().numpy(), ref)
    assert np.array_equal(h2.cpu().numpy(), ref)


def test_histogram_of_every_bit_pattern():
    ensure_library()
    x = synth.all_bf16_patterns().cuda()
    ws = sz.alloc_workspace(x.numel(), x.device)
    h = sz.splitzip_histogram(x, ws, "bf16").cpu().numpy()
    assert (h == 256).all()
    y = synth.all_e5m2_patterns().cuda()
    h = sz.splitzip_histogram(y, ws, "e5m2").cpu().numpy()
    assert (h == 8).all()


@pytest.mark.parametrize("name", ["n01_1024x4096", "kv_layer_32k", "escape_stress_t15_u4"])
def test_report_agrees_with_encode(name):
    ensure_library()
    w = synth.WORKLOADS[name]
    (r,) = report.run([name])
    x = w.make("cuda").reshape(-1)
    cal = w.make_calib("cuda").reshape(-1)
    ws = sz.alloc_workspace(max(x.numel(), cal.numel()), x.device)
    cb, _ = sz.splitzip_calibrate(cal, ws, w.fmt)
    st = sz.alloc_streams(x.numel(), w.chunk, w.fmt, x.numel(), x.device)
    sz.splitzip_encode(x, w.chunk, cb, st, ws, w.fmt)
    status, E = sz.splitzip_encode_status(ws)
    assert status == sz.OK and r["codebook"] == list(cb)
    assert r["n_escapes"] == E
    assert r["compression_ratio"] == pytest.approx(
        x.numel() * x.element_size() / sz.splitzip_compressed_bytes(x.numel(), w.chunk, E, w.fmt))
