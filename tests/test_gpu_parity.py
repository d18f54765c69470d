"""GPU parity: the CUDA path, called through the C ABI, against the oracle on
the same seeded inputs.  Integer/byte work, so the bar is exact: every stream
byte-identical, every decode bit-exact, calibration identical."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_kv_gb300 import synth
from tests.gpu_helpers import (check_roundtrip, gpu_calibrate, gpu_encode, host_bits,
                               assert_streams_equal)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _oracle_cb(t: torch.Tensor):
    fmt = "bf16" if t.dtype == torch.bfloat16 else "e5m2"
    cb, cov = oracle.calibrate(host_bits(t), fmt)
    return cb, cov


# ---------------------------------------------------------------- calibrate

@pytest.mark.parametrize("make", [
    lambda: synth.normal_bf16((1024, 4096), seed=1, device=DEV),
    lambda: synth.kv_cache(1, 32768, seed=1, device=DEV),
    lambda: synth.kv_cache(2, 1000, seed=1, device=DEV, dtype=torch.float8_e5m2),
    lambda: synth.all_bf16_patterns().to(DEV),
    lambda: synth.all_e5m2_patterns().to(DEV),
    lambda: synth.normal_bf16((3,), seed=5, device=DEV),
    lambda: synth.student_t_scaled_bf16((100001,), seed=2, device=DEV),
], ids=["n01", "kv_layer", "kv_e5m2", "all_bf16", "all_e5m2", "n3", "t15_odd"])
def test_calibrate_matches_oracle(make):
    x = make()
    cb, cov = gpu_calibrate(x)
    ref_cb, ref_cov = _oracle_cb(x)
    np.testing.assert_array_equal(np.array(cb, np.uint8), ref_cb)
    assert cov == ref_cov


# ------------------------------------------------------------ workloads

@pytest.mark.parametrize("name", ["n01_1024x4096", "kv_layer_32k", "escape_stress_t15",
                                  "escape_stress_t15_u4"])
def test_workload_roundtrip(name):
    w = synth.WORKLOADS[name]
    x = w.make(DEV)
    cb, _ = gpu_calibrate(w.make_calib(DEV))
    ref_cb, _ = _oracle_cb(w.make_calib(DEV))
    np.testing.assert_array_equal(np.array(cb, np.uint8), ref_cb)
    E = check_roundtrip(x, w.chunk, cb, name)
    assert 0 <= E <= x.numel()


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_all_patterns_roundtrip(fmt):
    x = (synth.all_bf16_patterns() if fmt == "bf16" else synth.all_e5m2_patterns()).to(DEV)
    cb, _ = gpu_calibrate(x)
    for chunk in (8, 64, 1024, 65536):
        check_roundtrip(x, chunk, cb, f"{fmt} all patterns chunk {chunk}")
    kv = synth.kv_cache(1, 64, seed=1, device=DEV,
                        dtype=torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2)
    cb2, _ = gpu_calibrate(kv)
    check_roundtrip(x, 1024, cb2, f"{fmt} all patterns, KV codebook")


SMALL_N = [1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 32, 33, 1000, 8191, 8192, 8193, 16383, 16384,
           16385, 100003]
CHUNKS = [8, 24, 1024, 4096, 65528, 65536]


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
@pytest.mark.parametrize("chunk", CHUNKS)
def test_small_shapes(fmt, chunk):
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    for n in SMALL_N:
        # Wide exponent spread so that every size has escapes in several chunks.
        x32 = synth.student_t_scaled_bf16((n,), seed=n, u_lo=-6, u_hi=6, device=DEV).float()
        x = x32.to(dt)
        cal = synth.kv_cache(1, 8, seed=1, device=DEV, dtype=dt)
        cb, _ = gpu_calibrate(cal)
        check_roundtrip(x, chunk, cb, f"{fmt} n={n} chunk={chunk}")


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_multi_tile_ragged(fmt):
    # Several encode/decode tiles plus a ragged tail, chunk sizes that do and
    # do not divide the tile.  256 ... 16384 are multiples of the BF16 encode
    # segment (256 elements), 1024 ... 16384 of the E5M2 one (1024): chunk
    # offsets come from the segment-start path there (by masks and shifts for
    # the ones that divide the 8192-element tile; 12288 and 16384 span tiles)
    # and from the general path otherwise.
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    x = synth.kv_cache(1, 777, seed=3, device=DEV, dtype=dt).reshape(-1)[:1_500_007]
    cb, _ = gpu_calibrate(synth.kv_cache(1, 64, seed=1, device=DEV, dtype=dt))
    for chunk in (8, 40, 256, 512, 1000, 1024, 2048, 3000, 4096, 8192, 12288, 16384, 65536):
        check_roundtrip(x, chunk, cb, f"{fmt} ragged chunk {chunk}")


@pytest.mark.parametrize("fmt,layers,tokens,n", [
    # 4163 full tiles and a ragged one: two superblocks of 4096 tiles, the
    # last block 4 tiles long; placement in one round of tiles per warp.
    ("bf16", 1, 16700, 4163 * 8192 + 777),
    ("e5m2", 1, 16700, 4163 * 8192 + 777),
    # Tens of thousands of tiles ending 38 tiles into a superblock: placement
    # in several rounds of tiles per warp (the grid the 2^31-element encode
    # uses), with a partial last block, superblock and tile.
    ("bf16", 16, 16400, (1 << 29) + 37 * 8192 + 555),
    ("e5m2", 20, 16400, 5 * (1 << 27) + 37 * 8192 + 555),
])
def test_block_and_superblock_boundaries(fmt, layers, tokens, n):
    """Escape offsets come from per-tile, per-block (64 tiles) and
    per-superblock (4096 tiles) counts; sizes that end inside a tile, a block
    and a superblock must still give the oracle's streams."""
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    x = synth.kv_cache(layers, tokens, seed=9, device=DEV, dtype=dt).reshape(-1)[:n].clone()
    cb, _ = gpu_calibrate(synth.kv_cache(1, 64, seed=1, device=DEV, dtype=dt))
    assert check_roundtrip(x, 1024, cb, f"{fmt} n={n}") > 0


def test_zero_and_all_escape_tensors():
    cb = list(range(100, 116))
    zeros = torch.zeros(50000, dtype=torch.bfloat16, device=DEV)  # exponent 0: all escapes
    assert check_roundtrip(zeros, 1024, cb, "all escapes") == 50000
    ones = torch.ones(50000, dtype=torch.bfloat16, device=DEV)    # exponent 127: none
    cb2 = list(range(120, 136))
    assert check_roundtrip(ones, 1024, cb2, "no escapes") == 0


@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_warp_escape_list_boundary(fmt):
    """Encode keeps each warp's first 32 escapes of a tile in one list (BF16:
    its four 256-element segments, at tile offsets 256w + 2048k, in order k;
    E5M2: its 1024 elements) and rebuilds a segment that does not fit from
    the input.  Tile 0 fills warp 0's list exactly, tile 1 overflows it by
    one in its last flagged segment; the streams must still be the oracle's."""
    n = 3 * 8192 + 123
    if fmt == "bf16":
        bits = torch.full((n,), 127 << 7, dtype=torch.int16)   # 1.0: exponent 127, in the codebook
        esc = 27 << 7                                           # exponent 27, not in it
        segs = [(0, 20), (2048, 12), (4096, 0)]                # tile 0: 32 escapes in warp 0
        segs1 = [(0, 20), (2048, 12), (4096, 1)]               # tile 1: 33 (last one overflows)
        cb, dt = list(range(120, 136)), torch.bfloat16
    else:
        bits = torch.full((n,), 15 << 2, dtype=torch.uint8)    # 1.0: exponent 15
        esc = 5 << 2                                            # exponent 5
        segs = [(0, 32)]                                        # warp 0's segment: exactly 32
        segs1 = [(0, 33), (1024, 5)]                            # 33 in warp 0, 5 in warp 1
        cb, dt = list(range(10, 26)), torch.float8_e5m2
    for base, pattern in ((0, segs), (8192, segs1)):
        for off, cnt in pattern:
            bits[torch.arange(cnt) * 7 + base + off] = esc      # spread inside the segment
    x = bits.view(dt).to(DEV)
    for chunk in (1024, 1000, 8):                           # segment-start and general chunk paths
        check_roundtrip(x, chunk, cb, f"{fmt} warp list boundary chunk {chunk}")


def test_deterministic_and_workspace_reuse():
    """Back-to-back encodes on one workspace, with different sizes and
    formats, give identical streams every time."""
    from lossless_bf16_kv_gb300 import splitzip as sz
    ws = sz.alloc_workspace(3_000_000, DEV)
    xs = [synth.kv_cache(1, 1000, seed=s, device=DEV).reshape(-1)[: 1_000_000 + 777 * s]
          for s in range(3)]
    xs.append(synth.kv_cache(1, 1000, seed=9, device=DEV, dtype=torch.float8_e5m2).reshape(-1))
    cbs = [gpu_calibrate(x)[0] for x in xs]
    first = [gpu_encode(x, 1024, cb, ws=ws)[0] for x, cb in zip(xs, cbs)]
    for _ in range(3):
        for x, cb, ref in zip(xs, cbs, first):
            again, status, _, _ = gpu_encode(x, 1024, cb, ws=ws)
            assert status == sz.OK
            assert_streams_equal(again, ref, "repeat")


def test_concurrent_streams():
    """Encodes and decodes of different tensors on different streams, each with
    its own workspace and buffers, overlap on the GPU and still give the
    oracle's streams and bit-exact round trips."""
    from lossless_bf16_kv_gb300 import splitzip as sz
    fmts = ["bf16", "e5m2", "bf16", "e5m2"]
    xs = [synth.kv_cache(2, 2048, seed=10 + i, device=DEV,
                         dtype=torch.bfloat16 if f == "bf16" else torch.float8_e5m2).reshape(-1)
          for i, f in enumerate(fmts)]
    cbs = [gpu_calibrate(x)[0] for x in xs]
    streams = [torch.cuda.Stream() for _ in xs]
    wss = [sz.alloc_workspace(x.numel(), DEV) for x in xs]
    outs = [sz.alloc_streams(x.numel(), 1024, f, x.numel(), DEV) for x, f in zip(xs, fmts)]
    ys = [torch.empty_like(x) for x in xs]
    torch.cuda.synchronize()
    for rep in range(3):
        for x, f, cb, st, ws, o, y in zip(xs, fmts, cbs, streams, wss, outs, ys):
            with torch.cuda.stream(st):
                sz.splitzip_encode(x, 1024, cb, o, ws, f, stream=st)
                sz.splitzip_decode(o, x.numel(), 1024, cb, y, f, stream=st)
        torch.cuda.synchronize()
        for x, f, cb, st, ws, o, y in zip(xs, fmts, cbs, streams, wss, outs, ys):
            status, E = sz.splitzip_encode_status(ws, st)
            assert status == sz.OK
            ref = oracle.encode(host_bits(x), 1024, np.asarray(cb, np.uint8), f)
            assert E == ref["n_escapes"]
            assert np.array_equal(o["codes"].cpu().numpy(), ref["codes"])
            assert np.array_equal(o["esc_pos"][:E].cpu().numpy().view(np.uint16), ref["esc_pos"])
            assert np.array_equal(host_bits(y), host_bits(x))


def test_concurrent_streams_with_a_large_bf16_encode():
    """A BF16 tensor large enough that its dense pass draws tiles from four
    counters (about 2^29 elements), encoded and decoded on one stream while
    small tensors are encoded and decoded on two others (their placements
    launched as dependents of their dense passes): every call's streams are
    the oracle's."""
    from lossless_bf16_kv_gb300 import splitzip as sz
    fmts = ["bf16", "bf16", "e5m2"]
    xs = [synth.kv_cache(16, 16400, seed=21, device=DEV).reshape(-1),
          synth.kv_cache(1, 3000, seed=22, device=DEV).reshape(-1),
          synth.kv_cache(1, 2500, seed=23, device=DEV, dtype=torch.float8_e5m2).reshape(-1)]
    cbs = [gpu_calibrate(x)[0] for x in xs]
    streams = [torch.cuda.Stream() for _ in xs]
    wss = [sz.alloc_workspace(x.numel(), DEV) for x in xs]
    outs = [sz.alloc_streams(x.numel(), 1024, f, x.numel() // 16, DEV) for x, f in zip(xs, fmts)]
    ys = [torch.empty_like(x) for x in xs]
    torch.cuda.synchronize()
    for _ in range(2):
        for x, f, cb, st, ws, o, y in zip(xs, fmts, cbs, streams, wss, outs, ys):
            with torch.cuda.stream(st):
                sz.splitzip_encode(x, 1024, cb, o, ws, f, stream=st)
                sz.splitzip_decode(o, x.numel(), 1024, cb, y, f, stream=st)
        torch.cuda.synchronize()
    for x, f, cb, st, ws, o, y in zip(xs, fmts, cbs, streams, wss, outs, ys):
        status, E = sz.splitzip_encode_status(ws, st)
        assert status == sz.OK
        ref = oracle.encode(host_bits(x), 1024, np.asarray(cb, np.uint8), f)
        got = {"codes": o["codes"].cpu().numpy(), "signman": o["signman"].cpu().numpy(),
               "chunk_off": o["chunk_off"].cpu().numpy().view(np.uint32),
               "esc_pos": o["esc_pos"][:E].cpu().numpy().view(np.uint16),
               "esc_val": o["esc_val"][:E].cpu().numpy(), "n_escapes": E}
        assert_streams_equal(got, ref, f"concurrent {f} n={x.numel()}")
        assert np.array_equal(host_bits(y), host_bits(x))


# ------------------------------------------- the single-launch engine

@pytest.mark.parametrize("fmt", ["bf16", "e5m2"])
def test_pipelined_engine_matches_oracle(fmt):
    """The single-launch pipeline (engine of splitzip_encode_noalloc) gives the
    oracle's streams too, on ragged sizes, small and large chunks, and an
    escape-dense input (tiles beyond its escape slots take the direct path)."""
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    cal = synth.kv_cache(1, 8, seed=1, device=DEV, dtype=dt)
    cb, _ = gpu_calibrate(cal)
    inputs = [synth.kv_cache(1, 777, seed=3, device=DEV, dtype=dt).reshape(-1)[:1_500_007],
              synth.student_t_scaled_bf16((300_001,), seed=7, device=DEV).float().to(dt)]
    for x in inputs:
        xb = host_bits(x)
        for chunk in (8, 24, 1024, 65536):
            ref = oracle.encode(xb, chunk, np.asarray(cb, np.uint8), fmt)
            gpu, status, _, _ = gpu_encode(x, chunk, cb, esc_capacity=ref["n_escapes"] + 16,
                                           engine="pipelined")
            assert status == 0
            assert_streams_equal(gpu, ref, f"pipelined {fmt} n={x.numel()} chunk {chunk}")


# ------------------------------------------------ full-size configurations

@pytest.mark.parametrize("name", ["kv_prefill_64L_16k", "kv_prefill_64L_16k_e5m2"])
def test_full_size_prefill(name):
    """2^31 elements, the launch configuration the benchmark times: every
    stream compared in full with the oracle's."""
    w = synth.WORKLOADS[name]
    cal = w.make_calib(DEV)
    cb, cov = gpu_calibrate(cal)
    ref_cb, ref_cov = _oracle_cb(cal)
    np.testing.assert_array_equal(np.array(cb, np.uint8), ref_cb)
    assert cov == ref_cov
    del cal
    x = w.make(DEV)
    check_roundtrip(x, w.chunk, cb, name)
