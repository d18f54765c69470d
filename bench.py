"""SplitZip codec benchmark on GB300.

One step = the whole hot path over one batch: encode of the full tensor
(field split, code lookup, dense streams, escape compaction, chunk offsets)
followed by decode of its streams back to the bitwise-identical tensor.  The
codebook is calibrated once beforehand (offline, as the pages describe it) and
timed separately.

Default workload: 64-layer prefill KV cache, BF16 [64, 2, 16384, 8, 128]
(2^31 elements, 4.29 GB), chunk 1024, codebook from a separate 1024-token
seed-1 sample.  The input is larger than L2 (129 MB), so no L2 flush is
needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

At N=1 the line also carries the other seeded workloads (configs 1, 2, 4
and its 5-20% escape variant, and the FP8 E5M2 prefill KV), each timed the
same way with fewer steps, under "configs".

Prints one JSON line (rank 0).  Multi-GPU runs (torchrun) are independent
replicas: each rank encodes/decodes its own copy, with no collective on the
data path (weak scaling); a barrier brackets the timed region and the time is
the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "encode / decode GB/s (uncompressed bytes) and % of HBM roofline; compression ratio"
DEFAULT_WORKLOAD = "kv_prefill_64L_16k"
FALLBACK_HBM_GBS = 6800.0
# The encode call is three launches (dense pass, escape placement, a one-CTA
# finish; the dense pass takes about 92% of the time), decode one.  The
# roofline is taken per call: algorithmic bytes of the call over its time.
KERNELS = {"encode": ("encode[dense_kernel+place_lists_kernel+finish_kernel]<Bf16Dense>",
                      "encode[dense_kernel+place_kernel+finish_kernel]<E5m2Dense>"),
           "decode": ("decode_kernel<Bf16Seg>", "decode_e5m2_kernel")}


# ------------------------------------------------------------ host helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def aggregate(times_s, units_per_rank: float):
    """Whole-job throughput of weak-scaled replicas: every rank processed
    units_per_rank in its own time; the job took the slowest rank's time."""
    t = max(times_s)
    return units_per_rank * len(times_s) / t, t


def max_over_ranks(seconds: float, device) -> list:
    """The job's time as every rank sees it: one all_reduce(MAX) of each
    rank's own timed region, repeated once per rank (so that aggregate() sees
    world_size entries).  Without an initialised process group it is the
    caller's own time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [seconds]
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [t.item()] * dist.get_world_size()


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Sources of the kernels the bench times (encode passes, decode) and what they
# include; host-only files (the C ABI, transfers) do not change the kernels.
KERNEL_SOURCES = ("encode_multi.cu", "decode.cu", "common.cuh", "fields.cuh", "kernels.h",
                  "lookback.cuh")


def _code_only(src: str) -> str:
    """C++ source without comments and whitespace: what the compiler sees."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return re.sub(r"\s+", "", src)


def kernel_source_sha() -> str:
    """Hash of the timed kernels' sources, comments and whitespace left out; a
    stored ncu traffic figure is used only while it matches (a changed kernel
    makes the figure stale, a changed comment does not)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lossless_bf16_kv_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)
    from profiles/ncu_traffic.txt, scaled to the workload; None if absent or
    taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 5 and not line.startswith("#") and parts[0] == kernel \
                    and parts[1] == workload and parts[4] == sha:
                return float(parts[2]) * float(parts[3])  # bytes/launch x scale
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)  # let the first sample land before the timed region
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i] == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- GPU arm

def algorithmic_bytes(fmt: str, n: int, chunk: int, n_escapes: int) -> int:
    """Bytes one encode (or one decode) must move: the raw tensor on one side,
    the compressed streams (codes, sign+mantissa, 3 bytes per escape, 4 per
    chunk offset) on the other."""
    from lossless_bf16_kv_gb300 import splitzip as sz
    return (2 if fmt == "bf16" else 1) * n + sz.splitzip_compressed_bytes(n, chunk, n_escapes, fmt)


def _fail(msg: str):
    print(json.dumps({"error": msg}), flush=True)
    sys.exit(1)


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from lossless_bf16_kv_gb300 import _build
    from lossless_bf16_kv_gb300 import splitzip as sz
    from lossless_bf16_kv_gb300 import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    _build.build_library()
    w = synth.WORKLOADS[args.workload]
    fmt, chunk = w.fmt, w.chunk
    elem = 2 if fmt == "bf16" else 1

    # Offline calibration on the separate sample (timed on its own).
    cal = w.make_calib(dev).reshape(-1)
    x = w.make(dev).reshape(-1)
    n = x.numel()
    ws = sz.alloc_workspace(n, dev)
    cb, coverage = sz.splitzip_calibrate(cal, ws, fmt)
    cb_dev = torch.empty(16, dtype=torch.uint8, device=dev)
    cov_dev = torch.empty(1, dtype=torch.int64, device=dev)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        sz.splitzip_calibrate_async(cal, cb_dev, cov_dev, ws, fmt)
    c0.record()
    for _ in range(5):
        sz.splitzip_calibrate_async(cal, cb_dev, cov_dev, ws, fmt)
    c1.record()
    torch.cuda.synchronize()
    cal_ms = c0.elapsed_time(c1) / 5
    cal_bytes = cal.numel() * elem
    del cal

    # First encode sizes the escape buffers exactly; then check the round trip.
    streams = sz.alloc_streams(n, chunk, fmt, n // 32 + 1024, dev)
    sz.splitzip_encode(x, chunk, cb, streams, ws, fmt)
    status, E = sz.splitzip_encode_status(ws)
    if status == sz.ERR_ESCAPE_OVERFLOW:
        streams = sz.alloc_streams(n, chunk, fmt, E, dev)
        sz.splitzip_encode(x, chunk, cb, streams, ws, fmt)
        status, E = sz.splitzip_encode_status(ws)
    if status != sz.OK:
        _fail(f"encode status {status}")
    y = torch.empty_like(x)
    sz.splitzip_decode(streams, n, chunk, cb, y, fmt, n_escapes=E)
    if not torch.equal(synth.raw_bits(x), synth.raw_bits(y)):
        _fail("decode is not bit-exact")

    def step():
        sz.splitzip_encode(x, chunk, cb, streams, ws, fmt)
        sz.splitzip_decode(streams, n, chunk, cb, y, fmt, n_escapes=E)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_start.record()
        for i in range(K):
            ev[i][0].record()
            sz.splitzip_encode(x, chunk, cb, streams, ws, fmt)
            ev[i][1].record()
            sz.splitzip_decode(streams, n, chunk, cb, y, fmt, n_escapes=E)
            ev[i][2].record()
        t_end.record()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    status_after, E_after = sz.splitzip_encode_status(ws)
    if status_after != sz.OK or E_after != E:
        _fail(f"timed encodes reported status {status_after}, E {E_after} (expected {E})")
    if not torch.equal(synth.raw_bits(x), synth.raw_bits(y)):
        _fail("timed decode is not bit-exact")

    total_s = t_start.elapsed_time(t_end) / 1e3
    enc_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    times = max_over_ranks(total_s, dev)
    bytes_per_step = n * elem
    value_Bps, max_s = aggregate(times, bytes_per_step * K)
    res = {
        "n": n, "E": E, "fmt": fmt, "chunk": chunk, "codebook": cb, "coverage": coverage,
        "K": K, "total_s": max_s, "value_gbs": value_Bps / 1e9, "enc_ms": enc_ms,
        "dec_ms": dec_ms, "cal_ms": cal_ms, "cal_bytes": cal_bytes,
        "clocks": clocks.summary(), "world": world, "rank": rank,
        "algo_bytes": algorithmic_bytes(fmt, n, chunk, E), "elem": elem,
    }
    if args.e2e:
        del streams, y, ws
        torch.cuda.empty_cache()
        res["e2e"] = run_e2e(x, cb, fmt, chunk, K, dev, world)
        if rank == 0 and world == 1:
            res["transfer"] = run_transfer(x, cb, fmt, chunk, dev)
    if rank == 0 and world == 1 and args.configs:
        del x
        torch.cuda.empty_cache()
        res["configs"] = run_configs(args.workload, max(3, min(K, 50)), dev)
    if world > 1:
        dist.destroy_process_group()
    return res


# The other seeded workloads, each timed like the headline one and reported
# beside it: config 1 (N(0,1)), config 2 (one KV layer), config 4 and its
# 5-20% escape variant, config 5 (FP8 E5M2 prefill KV).
CONFIG_WORKLOADS = ("n01_1024x4096", "kv_layer_32k", "kv_prefill_64L_16k",
                    "escape_stress_t15", "escape_stress_t15_u4", "kv_prefill_64L_16k_e5m2")
L2_BYTES = 129e6


def time_codec(x, cal, w, steps, dev, flush=None):
    """Calibrate on cal, then time `steps` encode + decode pairs of x with CUDA
    events on the launching stream (L2 flushed between steps when the tensor
    would otherwise stay in it).  Checks the round trip and returns the
    per-step times and stream figures."""
    import torch

    from lossless_bf16_kv_gb300 import splitzip as sz
    from lossless_bf16_kv_gb300 import synth

    fmt, chunk = w.fmt, w.chunk
    n = x.numel()
    ws = sz.alloc_workspace(max(n, cal.numel()), dev)
    cb, coverage = sz.splitzip_calibrate(cal, ws, fmt)
    streams = sz.alloc_streams(n, chunk, fmt, n // 32 + 1024, dev)
    sz.splitzip_encode(x, chunk, cb, streams, ws, fmt)
    status, E = sz.splitzip_encode_status(ws)
    if status == sz.ERR_ESCAPE_OVERFLOW:
        streams = sz.alloc_streams(n, chunk, fmt, E, dev)
        sz.splitzip_encode(x, chunk, cb, streams, ws, fmt)
        status, E = sz.splitzip_encode_status(ws)
    if status != sz.OK:
        _fail(f"{w.name}: encode status {status}")
    y = torch.empty_like(x)
    for _ in range(3):
        sz.splitzip_encode(x, chunk, cb, streams, ws, fmt)
        sz.splitzip_decode(streams, n, chunk, cb, y, fmt, n_escapes=E)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        ev[i][0].record()
        sz.splitzip_encode(x, chunk, cb, streams, ws, fmt)
        ev[i][1].record()
        if flush is not None:   # decode would read streams the encode just left in L2
            flush.fill_((i + 1) & 0xFF)
        ev[i][2].record()
        sz.splitzip_decode(streams, n, chunk, cb, y, fmt, n_escapes=E)
        ev[i][3].record()
    torch.cuda.synchronize()
    st_after, E_after = sz.splitzip_encode_status(ws)
    if st_after != sz.OK or E_after != E or not torch.equal(synth.raw_bits(x), synth.raw_bits(y)):
        _fail(f"{w.name}: timed round trip failed (status {st_after}, E {E_after} vs {E})")
    enc = [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)]
    dec = [ev[i][2].elapsed_time(ev[i][3]) for i in range(steps)]
    return enc, dec, E, cb, coverage


def config_figures(w, n, E, enc, dec, peak) -> dict:
    from lossless_bf16_kv_gb300 import splitzip as sz
    elem = 2 if w.fmt == "bf16" else 1
    algo = algorithmic_bytes(w.fmt, n, w.chunk, E)
    e, d = statistics.mean(enc), statistics.mean(dec)
    comp = sz.splitzip_compressed_bytes(n, w.chunk, E, w.fmt)
    return {"workload": w.name, "format": w.fmt, "shape": list(w.shape), "elements": n,
            "steps": len(enc), "encode_ms": round(e, 4), "decode_ms": round(d, 4),
            "encode_ms_median": round(statistics.median(enc), 4),
            "decode_ms_median": round(statistics.median(dec), 4),
            "encode_gbs": round(n * elem / (e / 1e3) / 1e9, 2),
            "decode_gbs": round(n * elem / (d / 1e3) / 1e9, 2),
            "encode_hbm_frac": round(algo / (e / 1e3) / 1e9 / peak, 4),
            "decode_hbm_frac": round(algo / (d / 1e3) / 1e9 / peak, 4),
            "algorithmic_bytes": algo, "n_escapes": E, "escape_rate": round(E / n, 6),
            "compression_ratio": round(n * elem / comp, 5),
            "l2": ("input larger than L2: no flush" if n * elem > L2_BYTES else
                   "L2 flushed (256 MB write) before each encode and each decode; small "
                   "tensors are bound by launch latency, not HBM")}


def run_configs(skip: str, steps: int, dev) -> list:
    """Every other seeded workload, timed and checked like the headline one."""
    import torch

    from lossless_bf16_kv_gb300 import synth
    peak, _ = measured_peak_hbm()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = []
    for name in CONFIG_WORKLOADS:
        if name == skip:
            continue
        w = synth.WORKLOADS[name]
        x = w.make(dev).reshape(-1)
        cal = w.make_calib(dev).reshape(-1)
        n = x.numel()
        big = n * (2 if w.fmt == "bf16" else 1) > L2_BYTES
        enc, dec, E, _, _ = time_codec(x, cal, w, steps, dev, None if big else flush)
        out.append(config_figures(w, n, E, enc, dec, peak))
        del x, cal
        torch.cuda.empty_cache()
    return out


def transfer_slice_elems(n: int, chunk: int) -> int:
    """Slice size of the pipelined transfers: one KV-cache layer (2 x 16384 x
    8 x 128 elements) of the prefill workloads, or the whole tensor rounded up
    to chunk and 16-element multiples when smaller."""
    unit = chunk * 16 // math.gcd(chunk, 16)
    return min(1 << 25, -(-n // unit) * unit)


def run_e2e(x, cb, fmt, chunk, K, dev, world):
    """The step through the public C ABI with host buffers: the tensor in
    pinned host memory is encoded into a host payload (splitzip_encode_to_host:
    slice copies to the device, encode, streams back), and the payload decoded
    into pinned host memory (splitzip_decode_from_host), copies overlapping the
    kernels.  Timed on the host clock around synchronous calls that span three
    streams."""
    import torch
    import torch.distributed as dist

    from lossless_bf16_kv_gb300 import splitzip as sz

    n, eb = x.numel(), x.element_size()
    se = transfer_slice_elems(n, chunk)
    hx = torch.empty(n, dtype=x.dtype).pin_memory()
    hx.copy_(x)
    hy = torch.empty_like(hx).pin_memory()
    scratch = sz.alloc_transfer_scratch(se, chunk, fmt, dev)
    streams = [torch.cuda.Stream(dev) for _ in range(3)]
    payload, nbytes = sz.encode_to_host(hx, chunk, cb, se, scratch, streams, fmt)
    steps = K

    def step():
        st, nb = sz.splitzip_encode_to_host(hx, chunk, cb, se, payload, scratch, streams, fmt)
        assert st == sz.OK and nb == nbytes
        sz.splitzip_decode_from_host(payload, nbytes, hy, scratch, streams)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    secs = time.perf_counter() - t0
    if world > 1:
        tt = torch.tensor([secs], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        secs = tt.item()
    if not torch.equal(hx, hy):
        _fail("end-to-end round trip is not bit-exact")
    raw = n * eb
    return {"value": round(raw * steps * world / secs / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": raw + nbytes, "d2h_bytes_per_step": nbytes + raw,
            "steps": steps, "slice_elems": se, "payload_bytes": nbytes,
            "path": "pinned host tensor -> splitzip_encode_to_host -> host payload -> "
                    "splitzip_decode_from_host -> pinned host tensor (host clock)"}


def run_transfer(x, cb, fmt, chunk, dev):
    """KV transfer over the host link, the codec's use on the pages: a device
    tensor to a host payload and back to the device (splitzip_encode_to_host,
    splitzip_decode_from_host), against moving the raw bytes device -> host ->
    device with one copy each way.  Best of three, host clock."""
    import torch

    from lossless_bf16_kv_gb300 import splitzip as sz

    n, eb = x.numel(), x.element_size()
    se = transfer_slice_elems(n, chunk)
    scratch = sz.alloc_transfer_scratch(se, chunk, fmt, dev)
    streams = [torch.cuda.Stream(dev) for _ in range(3)]
    payload, nbytes = sz.encode_to_host(x, chunk, cb, se, scratch, streams, fmt)
    y = torch.empty_like(x)
    h = torch.empty(n, dtype=x.dtype).pin_memory()

    def best(fn):
        t = []
        for _ in range(3):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            t.append(time.perf_counter() - t0)
        return min(t)

    enc = best(lambda: sz.splitzip_encode_to_host(x, chunk, cb, se, payload, scratch, streams, fmt))
    dec = best(lambda: sz.splitzip_decode_from_host(payload, nbytes, y, scratch, streams))
    if not torch.equal(synth_bits(x), synth_bits(y)):
        _fail("transfer round trip is not bit-exact")
    d2h = best(lambda: h.copy_(x, non_blocking=True))
    h2d = best(lambda: y.copy_(h, non_blocking=True))
    return {"raw_ms": round((d2h + h2d) * 1e3, 3), "splitzip_ms": round((enc + dec) * 1e3, 3),
            "speedup": round((d2h + h2d) / (enc + dec), 4),
            "encode_to_host_ms": round(enc * 1e3, 3), "decode_from_host_ms": round(dec * 1e3, 3),
            "raw_bytes": n * eb, "payload_bytes": nbytes, "slice_elems": se,
            "path": "device tensor -> host payload -> device tensor, vs raw device -> host -> device"}


def synth_bits(t):
    from lossless_bf16_kv_gb300 import synth
    return synth.raw_bits(t)


# ------------------------------------------------------------- CPU oracle

def time_oracle(bits, fmt: str, chunk: int, cb, min_seconds: float = 0.0):
    """Oracle encode + decode of one sample; returns seconds per round trip."""
    import numpy as np

    import oracle
    cbv = np.asarray(cb, np.uint8)
    reps, t = 0, 0.0
    while True:
        t0 = time.perf_counter()
        s = oracle.encode(bits, chunk, cbv, fmt)
        yb = oracle.decode(s, bits.size, chunk, cbv, fmt)
        t += time.perf_counter() - t0
        reps += 1
        if not np.array_equal(yb, bits):
            _fail("oracle round trip is not bit-exact")
        if t >= min_seconds:
            return t / reps


def time_oracle_sharded(bits, fmt: str, chunk: int, cb, threads: int) -> float:
    """The unchanged oracle run concurrently on `threads` chunk-aligned shards
    of bits (contiguous chunk ranges, each an independent encode + decode
    round trip; the C calls release the GIL).  Returns wall seconds."""
    import concurrent.futures

    import numpy as np

    import oracle
    cbv = np.asarray(cb, np.uint8)
    per = -(-bits.size // threads)
    per += (-per) % chunk
    shards = [bits[i:i + per] for i in range(0, bits.size, per)]

    def one(sh):
        st = oracle.encode(sh, chunk, cbv, fmt)
        return np.array_equal(oracle.decode(st, sh.size, chunk, cbv, fmt), sh)

    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(len(shards)) as ex:
        ok = list(ex.map(one, shards))
    sec = time.perf_counter() - t0
    if not all(ok):
        _fail("oracle round trip is not bit-exact")
    return sec


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


# Both CPU measurements -- the GPU line's cpu_baseline and the reference arm --
# time the oracle on one sample: the first CPU_SAMPLE_ELEMS elements of the
# workload, drawn on the host by the workload's own generator (for the prefill
# KV workloads, its first layers), with the codebook the oracle calibrates on
# the workload's calibration recipe drawn the same way.
CPU_SAMPLE_ELEMS = 1 << 28


def cpu_sample(w):
    """(bits, codebook, description) of the oracle's bounded sample of w."""
    import numpy as np
    import torch

    import oracle
    from lossless_bf16_kv_gb300 import synth
    if w.name.startswith("kv_prefill"):
        dt = torch.bfloat16 if w.fmt == "bf16" else torch.float8_e5m2
        layers = max(1, min(w.shape[0], CPU_SAMPLE_ELEMS // math.prod(w.shape[1:])))
        x = synth.kv_cache(layers, w.shape[2], seed=0, device="cpu", dtype=dt)
        cal = synth.kv_cache(w.shape[0], 1024, seed=1, device="cpu", dtype=dt)
        what = f"first {layers} of {w.shape[0]} layers"
    else:
        x, cal = w.make("cpu"), w.make_calib("cpu")
        what = "the whole tensor"
    bits = synth.raw_bits(x).numpy().reshape(-1)[:CPU_SAMPLE_ELEMS]
    cbits = synth.raw_bits(cal).numpy().reshape(-1)
    if w.fmt == "bf16":
        bits, cbits = bits.view(np.uint16), cbits.view(np.uint16)
    cb, _ = oracle.calibrate(cbits, w.fmt)
    desc = (f"{bits.size} elements ({what}) of the workload drawn on the host by the same "
            f"generator; one oracle encode+decode round trip per run")
    return np.ascontiguousarray(bits), cb, desc


def cpu_baseline(w, target_cpu_s: float):
    """The oracle as it stands on the shared sample: on every host core as
    concurrent runs over chunk-aligned shards (the chunk-range sharding of the
    format; the oracle's code is the same), repeated until about target_cpu_s
    of CPU time has been spent, and once on one thread."""
    bits, cb, desc = cpu_sample(w)
    T = host_threads()
    runs, wall = 0, 0.0
    while runs == 0 or wall * T < target_cpu_s:
        wall += time_oracle_sharded(bits, w.fmt, w.chunk, cb, T)
        runs += 1
    sec1 = time_oracle(bits, w.fmt, w.chunk, cb)
    elem = 2 if w.fmt == "bf16" else 1
    return {"value": round(bits.size * elem * runs / wall / 1e9, 4), "unit": "GB/s", "cores": T,
            "kind": "oracle",
            "sample": f"{desc}; {T} concurrent oracle runs over chunk-aligned shards, mean of "
                      f"{runs} runs ({wall:.2f} s wall)",
            "single_thread": {"value": round(bits.size * elem / sec1 / 1e9, 4), "cores": 1,
                              "seconds": round(sec1, 2)}}


# ----------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle (plain C) on the host cores: each step is one encode + decode
    round trip of the shared bounded sample of the workload, as concurrent
    oracle runs over chunk-aligned shards, one per host core."""
    from lossless_bf16_kv_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    bits, cb, desc = cpu_sample(w)
    T = host_threads()
    for _ in range(args.warmup):
        time_oracle_sharded(bits, w.fmt, w.chunk, cb, T)
    secs = 0.0
    for _ in range(args.steps):
        secs += time_oracle_sharded(bits, w.fmt, w.chunk, cb, T)
    elem = 2 if w.fmt == "bf16" else 1
    value = bits.size * elem * args.steps / secs / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.fmt, "data": "synthetic",
        "config": workload_config(w, args.gpus),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": T, "kind": "oracle",
                         "sample": f"{desc}; {T} concurrent oracle runs over chunk-aligned "
                                   f"shards per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def workload_config(w, world: int) -> dict:
    return {"workload": w.name, "shape": list(w.shape), "format": w.fmt, "chunk_size": w.chunk,
            "elements": w.numel, "description": w.description,
            "step": "encode + decode of the whole tensor (codebook calibrated beforehand)",
            "value": "uncompressed bytes per step / step time, summed over replicas",
            "l2": ("no flush: the input is larger than the 129 MB L2" if w.nbytes > 129e6 else
                   "input smaller than L2: numbers are L2-resident, not HBM"),
            "parallelism": f"replicas x{world}"}


# -------------------------------------------------------------------- main

def main():
    from lossless_bf16_kv_gb300 import synth
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["own", "reference"], default="own")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=20.0,
                    help="CPU time (threads x wall) the cpu_baseline spends at least")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip timing the other seeded workloads")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank, world, _ = dist_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    res = run_gpu(args)
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    n, E, elem, K = res["n"], res["E"], res["elem"], res["K"]
    enc = statistics.mean(res["enc_ms"])
    dec = statistics.mean(res["dec_ms"])
    peak, src = measured_peak_hbm()
    algo = res["algo_bytes"]
    dominant = "encode" if enc >= dec else "decode"
    kernel = KERNELS[dominant][0 if res["fmt"] == "bf16" else 1]
    dom_ms = max(enc, dec)
    other_kernel = KERNELS["decode" if dominant == "encode" else "encode"][
        0 if res["fmt"] == "bf16" else 1]
    achieved = algo / (dom_ms / 1e3) / 1e9
    from lossless_bf16_kv_gb300 import splitzip as sz
    comp = sz.splitzip_compressed_bytes(n, res["chunk"], E, res["fmt"])
    line = {
        "metric": METRIC, "value": round(res["value_gbs"], 2), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(res["total_s"] * 1e3 / K, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": res["fmt"], "data": "synthetic",
        "config": workload_config(w, world),
        "encode_gbs": round(n * elem / (enc / 1e3) / 1e9, 2),
        "decode_gbs": round(n * elem / (dec / 1e3) / 1e9, 2),
        "encode_ms": round(enc, 4), "decode_ms": round(dec, 4),
        "encode_ms_median": round(statistics.median(res["enc_ms"]), 4),
        "decode_ms_median": round(statistics.median(res["dec_ms"]), 4),
        "encode_hbm_frac": round(algo / (enc / 1e3) / 1e9 / peak, 4),
        "decode_hbm_frac": round(algo / (dec / 1e3) / 1e9 / peak, 4),
        "compression_ratio": round(n * elem / comp, 5), "compressed_bytes": comp,
        "n_escapes": E, "escape_rate": E / n, "calibration_coverage": res["coverage"],
        "calibrate_gbs": round(res["cal_bytes"] / (res["cal_ms"] / 1e3) / 1e9, 2),
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1),
                     "peak": peak, "peak_source": f"{src} (copy bandwidth, MEASURED_PEAKS hbm_gbs)"
                     if src == "measured" else "fallback", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": stored_traffic(kernel, w.name),
                     "algorithmic_bytes_per_launch": algo},
        "roofline_other": {"op": "decode" if dominant == "encode" else "encode",
                           "achieved": round(algo / (min(enc, dec) / 1e3) / 1e9, 1),
                           "frac": round(algo / (min(enc, dec) / 1e3) / 1e9 / peak, 4),
                           "kernel": other_kernel,
                           "traffic": stored_traffic(other_kernel, w.name)},
        "gpu_launches": 4 * K,  # encode: dense, place, finish; decode: one
        "clocks": res["clocks"],
        "context": {"pages_h200_encode_gbs": 613.3, "pages_h200_decode_gbs": 2181.8,
                    "note": "H200, real Qwen3-32B KV; another machine and data"},
    }
    if "e2e" in res:
        line["e2e"] = res["e2e"]
    if "transfer" in res:
        line["transfer"] = res["transfer"]
    if "configs" in res:
        line["configs"] = res["configs"]
    if world == 1 and args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
