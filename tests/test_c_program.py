"""The C ABI used from plain C: tests/c_abi_roundtrip.c (and
tests/c_noalloc_reset.c, run by the no-allocation tests) include only
include/splitzip.h and the CUDA runtime and link libsplitzip.so.  On CPU the
programs must compile and link; on a GPU the round trip's codebook and streams
must be the oracle's, byte for byte, and its decode bit-exact."""
import glob
import os
import subprocess

import numpy as np
import pytest

import oracle
from lossless_bf16_kv_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_roundtrip.c")


def _cuda_dirs():
    root = os.path.dirname(os.path.dirname(os.path.realpath(_build.nvcc())))
    libs = [d for d in [os.path.join(root, "lib64")] + glob.glob(os.path.join(root, "targets", "*", "lib"))
            if os.path.exists(os.path.join(d, "libcudart.so"))]
    return os.path.join(root, "include"), libs[0]


def compile_program(out_dir, src: str = SRC) -> str:
    _build.build_library()
    inc, cudalib = _cuda_dirs()
    exe = os.path.join(str(out_dir), os.path.basename(src)[:-2])
    libdir = os.path.dirname(_build.LIBPATH)
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", f"-I{ROOT}/include", f"-I{inc}",
           src, "-o", exe, f"-L{libdir}", "-lsplitzip", f"-L{cudalib}", "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


@pytest.mark.parametrize("name", ["c_abi_roundtrip.c", "c_noalloc_reset.c"])
def test_c_program_compiles_against_the_header(tmp_path, name):
    exe = compile_program(tmp_path, os.path.join(ROOT, "tests", name))
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
@pytest.mark.parametrize("fmt,chunk", [("bf16", 1024), ("bf16", 1000), ("e5m2", 1024), ("e5m2", 64)])
def test_c_program_round_trip_matches_oracle(tmp_path, fmt, chunk):
    import torch

    from lossless_bf16_kv_gb300 import synth
    dt = torch.bfloat16 if fmt == "bf16" else torch.float8_e5m2
    npdt = np.uint16 if fmt == "bf16" else np.uint8
    x = synth.kv_cache(1, 512, seed=0, device="cpu", dtype=dt).reshape(-1)[:1_000_003]
    cal = synth.kv_cache(1, 128, seed=1, device="cpu", dtype=dt).reshape(-1)
    xb = synth.raw_bits(x).numpy().view(npdt)
    cb_bits = synth.raw_bits(cal).numpy().view(npdt)
    xb.tofile(tmp_path / "x.bin")
    cb_bits.tofile(tmp_path / "cal.bin")
    exe = compile_program(tmp_path)
    prefix = str(tmp_path / "out")
    r = subprocess.run([exe, fmt, str(tmp_path / "x.bin"), str(tmp_path / "cal.bin"), str(chunk), prefix],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    fields = dict(kv.split("=") for kv in r.stdout.split())
    assert fields["exact"] == "1"

    ref_cb, ref_cov = oracle.calibrate(cb_bits, fmt)
    cb = np.fromfile(prefix + ".cb", np.uint8)
    assert list(cb) == list(ref_cb)
    assert float(fields["coverage"]) == ref_cov
    ref = oracle.encode(xb, chunk, ref_cb, fmt)
    E = int(fields["E"])
    assert E == ref["n_escapes"]
    assert int(fields["bytes"]) == oracle.compressed_bytes(xb.size, chunk, E, fmt)
    for name, dtype in (("codes", np.uint8), ("signman", np.uint8), ("esc_pos", np.uint16),
                        ("esc_val", np.uint8), ("chunk_off", np.uint32)):
        got = np.fromfile(f"{prefix}.{name}", dtype)
        assert np.array_equal(got, ref[name]), f"{fmt} chunk {chunk}: {name} differs"
