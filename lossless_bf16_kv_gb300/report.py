"""Exponent statistics of KV-cache tensors: entropy, top-k coverage, escapes.

The pages motivate SplitZip with the exponent distribution of real KV caches
(low entropy, a few exponents covering nearly every value) and ship an
analysis script for it on Qwen3 activations ("SplitZip: Ultra-Fast Lossless
KV Compression for Disaggregated LLM Serving", README sections Highlights and
"Reproducing Paper Artifact Scripts").  The real activations are not
available here; this module computes the same kind of statistics for the
seeded synthetic workloads, from exponent histograms taken on the GPU by
``splitzip_histogram``.

    python -m lossless_bf16_kv_gb300.report [--workloads a,b] [--json]

For each workload: Shannon entropy of the exponent (bits), number of distinct
exponents, coverage of the k most frequent exponents (k = 1, 2, 4, 8, 16), the
escape rate of the codebook calibrated (on the GPU) on the workload's
calibration sample,
and the compression ratio the codec reaches with it, next to the ratio an
ideal entropy coder of the exponents would reach (same sign/mantissa bytes).
"""
from __future__ import annotations

import argparse
import json
import math

import numpy as np

TOPK = (1, 2, 4, 8, 16)


def exponent_stats(hist, codebook, fmt: str = "bf16", chunk: int = 1024) -> dict:
    """Statistics of one exponent histogram (256 BF16 / 32 E5M2 bins) under a
    codebook (16 exponents, as splitzip_calibrate returns it).  Sizes come from
    the library's closed forms (pure host functions, no GPU needed)."""
    h = np.asarray(hist, dtype=np.int64)
    n = int(h.sum())
    if n == 0:
        raise ValueError("empty histogram")
    p = h[h > 0] / n
    entropy = float(-(p * np.log2(p)).sum())
    ranked = np.sort(h)[::-1]
    cover = {k: float(ranked[:k].sum() / n) for k in TOPK}
    from . import splitzip as sz
    cb = [int(c) for c in codebook]
    covered = int(h[cb].sum())
    escapes = n - covered
    elem = 2 if fmt == "bf16" else 1
    compressed = sz.splitzip_compressed_bytes(n, chunk, escapes, fmt)
    entropy_bytes = math.ceil(n * entropy / 8) + sz.splitzip_signman_bytes(n, fmt)
    return {"fmt": fmt, "n": n, "entropy_bits": entropy, "distinct_exponents": int((h > 0).sum()),
            "topk_coverage": cover, "codebook": [int(c) for c in cb], "escape_rate": escapes / n,
            "n_escapes": escapes, "compression_ratio": n * elem / compressed,
            "entropy_coded_ratio": n * elem / entropy_bytes}


def gpu_histogram(x, workspace=None):
    """Exponent histogram of a BF16 / E5M2 tensor on the GPU (numpy int64)."""
    import torch

    from . import splitzip as sz
    flat = x.reshape(-1)
    if workspace is None:
        workspace = sz.alloc_workspace(flat.numel(), flat.device)
    out = sz.splitzip_histogram(flat, workspace)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def run(names, device="cuda") -> list:
    import torch

    from . import splitzip as sz
    from . import synth
    rows = []
    for name in names:
        w = synth.WORKLOADS[name]
        cal = w.make_calib(device).reshape(-1)
        ws = sz.alloc_workspace(cal.numel(), cal.device)
        codebook, _ = sz.splitzip_calibrate(cal, ws, w.fmt)
        del cal, ws
        x = w.make(device)
        hist = gpu_histogram(x)
        del x
        torch.cuda.empty_cache()
        r = exponent_stats(hist, codebook, w.fmt, w.chunk)
        r["workload"] = name
        rows.append(r)
    return rows


def markdown(rows) -> str:
    head = ("| workload | format | elements | entropy (bits) | distinct | top-1 | top-4 | top-8 "
            "| top-16 | escape rate | ratio | entropy-coded ratio |\n|" + "---|" * 12)
    lines = [head]
    for r in rows:
        c = r["topk_coverage"]
        lines.append(f"| {r['workload']} | {r['fmt']} | {r['n']} | {r['entropy_bits']:.3f} | "
                     f"{r['distinct_exponents']} | {c[1]:.4f} | {c[4]:.4f} | {c[8]:.4f} | "
                     f"{c[16]:.6f} | {r['escape_rate']:.5f} | {r['compression_ratio']:.4f} | "
                     f"{r['entropy_coded_ratio']:.4f} |")
    return "\n".join(lines)


def main():
    from . import synth
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workloads", default=",".join(sorted(synth.WORKLOADS)))
    ap.add_argument("--json", action="store_true")
    args = ap.parse_args()
    rows = run([w for w in args.workloads.split(",") if w])
    if args.json:
        for r in rows:
            print(json.dumps(r))
    else:
        print(markdown(rows))


if __name__ == "__main__":
    main()
