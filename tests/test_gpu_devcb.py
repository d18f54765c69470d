"""Codebooks that stay on the device: splitzip_calibrate_async's outputs, the
encode and decode that read their codebook from device memory
(splitzip_encode_devcb / splitzip_decode_devcb), and transfers that calibrate
every slice (KV-cache layer) on the device before encoding it.  All through
the C ABI, against the oracle: codebooks and covered counts equal, streams
byte-identical, decodes bit-exact, payloads equal byte for byte."""
import numpy as np
import pytest
import torch

import oracle
from oracle import payload as op
from lossless_bf16_kv_gb300 import splitzip as sz
from lossless_bf16_kv_gb300 import synth

from .gpu_helpers import assert_streams_equal, ensure_library, fmt_of, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"
E5 = torch.float8_e5m2


def _calibrate_async(x: torch.Tensor):
    """(device codebook tensor, covered count) from splitzip_calibrate_async."""
    ensure_library()
    flat = x.reshape(-1)
    ws = sz.alloc_workspace(flat.numel(), flat.device)
    cb = torch.full((16,), 0xEE, dtype=torch.uint8, device=DEV)
    cov = torch.full((1,), -1, dtype=torch.int64, device=DEV)
    sz.splitzip_calibrate_async(flat, cb, cov, ws, fmt_of(x))
    torch.cuda.synchronize()
    return cb, int(cov.item())


def _oracle_calibration(bits: np.ndarray, fmt: str):
    """The oracle's codebook and the exact count of elements it covers."""
    cb, _ = oracle.calibrate(bits, fmt)
    covered = int(oracle.histogram(bits, fmt)[cb.astype(np.int64)].sum())
    return cb, covered


# The calibration samples of the five workloads (configs 1-5: the N(0,1)
# sample of configs 1 and 4, the single-layer KV sample, the prefill sample,
# the E5M2 prefill sample), every bit pattern, and ragged or escape-heavy cases.
CAL_INPUTS = {
    "n01_seed1": lambda: synth.normal_bf16((1024, 4096), seed=1, device=DEV),
    "kv_layer_seed1": lambda: synth.kv_cache(1, 32768, seed=1, device=DEV, squeeze_single=True),
    "prefill_sample_bf16": lambda: synth.kv_cache(64, 1024, seed=1, device=DEV),
    "prefill_sample_e5m2": lambda: synth.kv_cache(64, 1024, seed=1, device=DEV, dtype=E5),
    "all_bf16": lambda: synth.all_bf16_patterns().to(DEV),
    "all_e5m2": lambda: synth.all_e5m2_patterns().to(DEV),
    "ragged_e5m2": lambda: synth.kv_cache(1, 300, seed=7, device=DEV, dtype=E5).reshape(-1)[:614_397],
    "t15_odd": lambda: synth.student_t_scaled_bf16((100_001,), seed=2, device=DEV),
    "three": lambda: synth.normal_bf16((3,), seed=5, device=DEV),
}


@pytest.mark.parametrize("name", sorted(CAL_INPUTS))
def test_calibrate_async_matches_oracle(name):
    x = CAL_INPUTS[name]()
    cb_dev, covered = _calibrate_async(x)
    ref_cb, ref_covered = _oracle_calibration(host_bits(x), fmt_of(x))
    np.testing.assert_array_equal(cb_dev.cpu().numpy(), ref_cb)
    assert covered == ref_covered


def _device_streams_to_host(st: dict, E: int) -> dict:
    return {"codes": st["codes"].cpu().numpy(), "signman": st["signman"].cpu().numpy(),
            "chunk_off": st["chunk_off"].cpu().numpy().view(np.uint32),
            "esc_pos": st["esc_pos"][:E].cpu().numpy().view(np.uint16),
            "esc_val": st["esc_val"][:E].cpu().numpy(), "n_escapes": E}


CASES = [  # (format, elements, chunk, calibration sample, input seed)
    ("bf16", 3_000_017, 1024, "kv", 0),
    ("bf16", 1_048_576, 8, "kv", 3),
    ("bf16", 777_777, 4096, "n01", 4),
    ("bf16", 200_003, 65536, "t15", 5),
    ("e5m2", 3_000_011, 1024, "kv", 0),
    ("e5m2", 500_000, 1000, "kv", 6),
    ("e5m2", 65_541, 8, "kv", 7),
]


def _inputs(fmt, n, sample, seed):
    dt = torch.bfloat16 if fmt == "bf16" else E5
    tokens = -(-n // (2 * 8 * 128))
    x = synth.kv_cache(1, tokens, seed=seed, device=DEV, dtype=dt).reshape(-1)[:n].clone()
    if sample == "n01":
        cal = synth.normal_bf16((256, 1024), seed=1, device=DEV)
    elif sample == "t15":
        x = synth.student_t_scaled_bf16((n,), seed=seed, u_lo=-4.0, u_hi=4.0, device=DEV)
        cal = synth.normal_bf16((256, 1024), seed=1, device=DEV)
    else:
        cal = synth.kv_cache(1, 1024, seed=1, device=DEV, dtype=dt)
    return x, cal


@pytest.mark.parametrize("fmt,n,chunk,sample,seed", CASES)
def test_devcb_encode_and_decode_match_oracle(fmt, n, chunk, sample, seed):
    """Calibrate on the device, encode with that device codebook, decode with
    it: streams equal the oracle's encode with the oracle's codebook of the same
    sample, and the decode (of the GPU streams and of the oracle's) is
    bit-exact.  No host round trip between the calls."""
    ensure_library()
    x, cal = _inputs(fmt, n, sample, seed)
    ws = sz.alloc_workspace(max(n, cal.numel()), x.device)
    cb_dev = torch.empty(16, dtype=torch.uint8, device=DEV)
    cov = torch.empty(1, dtype=torch.int64, device=DEV)
    st = sz.alloc_streams(n, chunk, fmt, n, DEV)
    sz.splitzip_calibrate_async(cal.reshape(-1), cb_dev, cov, ws, fmt)
    sz.splitzip_encode_devcb(x, chunk, cb_dev, st, ws, fmt)
    y = torch.empty_like(x)
    sz.splitzip_decode_devcb(st, n, chunk, cb_dev, y, fmt)
    status, E = sz.splitzip_encode_status(ws)
    assert status == sz.OK
    bits = host_bits(x)
    ref_cb, _ = oracle.calibrate(host_bits(cal), fmt)
    np.testing.assert_array_equal(cb_dev.cpu().numpy(), ref_cb)
    ref = oracle.encode(bits, chunk, ref_cb, fmt)
    assert_streams_equal(_device_streams_to_host(st, E), ref, f"{fmt} n={n} chunk={chunk}")
    assert np.array_equal(host_bits(y), bits)
    from .gpu_helpers import device_streams
    y2 = torch.empty_like(x)
    sz.splitzip_decode_devcb(device_streams(ref), n, chunk, cb_dev, y2, fmt,
                             n_escapes=ref["n_escapes"])
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(y2), bits)


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_devcb_invalid_codebook_is_reported(fmt):
    """A device codebook the host cannot check is checked by the encode: a
    repeated entry (or an E5M2 entry above 31) is reported as INVALID_ARG by
    splitzip_encode_status, and the next encode on the same workspace with a
    valid codebook is correct again."""
    ensure_library()
    dt = torch.bfloat16 if fmt == "bf16" else E5
    x = synth.kv_cache(1, 400, seed=2, device=DEV, dtype=dt).reshape(-1)
    n, chunk = x.numel(), 1024
    ws = sz.alloc_workspace(n, DEV)
    st = sz.alloc_streams(n, chunk, fmt, n, DEV)
    good, _ = oracle.calibrate(host_bits(x), fmt)
    bads = [np.concatenate([good[:15], good[:1]])]
    if fmt == "e5m2":
        bads.append(np.concatenate([good[:15], np.array([40], np.uint8)]))
    for bad in bads:
        sz.splitzip_encode_devcb(x, chunk, torch.from_numpy(bad.astype(np.uint8)).to(DEV), st, ws, fmt)
        status, _ = sz.splitzip_encode_status(ws)
        assert status == sz.ERR_INVALID_ARG
    sz.splitzip_encode_devcb(x, chunk, torch.from_numpy(good).to(DEV), st, ws, fmt)
    status, E = sz.splitzip_encode_status(ws)
    assert status == sz.OK
    assert_streams_equal(_device_streams_to_host(st, E), oracle.encode(host_bits(x), chunk, good, fmt))


def _kv(fmt, n, seed):
    dt = torch.bfloat16 if fmt == "bf16" else E5
    layers = max(1, -(-n // (2 * 256 * 1024)))
    return synth.kv_cache(layers, 256, seed=seed, device=DEV, dtype=dt).reshape(-1)[:n].clone()


@pytest.mark.parametrize("where", ["device", "host"])
@pytest.mark.parametrize("fmt,n,chunk,se", [
    ("bf16", 5 * (1 << 19) - 3 * 1024 - 7, 1024, 1 << 19),  # one KV layer per slice, ragged end
    ("bf16", 300_000, 256, 65536),
    ("e5m2", 3 * (1 << 19) + 77, 1024, 1 << 19),
    ("e5m2", 50_000, 64, 4096),
])
def test_per_layer_calibrated_transfer_matches_oracle(fmt, n, chunk, se, where):
    """encode_to_host with no codebooks calibrates each slice on the device:
    the payload equals, byte for byte, the oracle's payload whose slices carry
    the oracle's codebook of that slice (and decodes back bit for bit)."""
    ensure_library()
    # Layers with different scales, so that the slices' codebooks differ.
    parts = [_kv(fmt, min(se, n - s0), seed=11 + i) for i, s0 in enumerate(range(0, n, se))]
    x = torch.cat([(p.float() * 2.0 ** (3 * (i % 4))).to(p.dtype) for i, p in enumerate(parts)])
    bits = host_bits(x)
    scratch = sz.alloc_transfer_scratch(se, chunk, fmt)
    streams = [torch.cuda.Stream() for _ in range(3)]
    src = x if where == "device" else x.cpu().pin_memory()
    payload, nbytes = sz.encode_to_host(src, chunk, None, se, scratch, streams, fmt)
    ref = op.write_calibrated(bits, fmt, chunk, se)
    _, slices = op.read(ref)
    assert len({tuple(s["codebook"]) for s in slices}) > 1
    assert nbytes == len(ref)
    assert payload[:nbytes].numpy().tobytes() == ref
    y = torch.empty_like(x)
    sz.splitzip_decode_from_host(payload, nbytes, y, scratch, streams)
    assert np.array_equal(host_bits(y), bits)
