"""Per-kernel micro-benchmark of the codec on one GPU.

    python -m fp4_communication_compression_gb300.perf [--sizes 16777216 268435456]
        [--kernels compress decompress_bf16_b1 ...] [--iters 30]

Each kernel is timed alone with CUDA events on the launching stream, after an L2 flush
(a write of a buffer larger than L2 followed by a read of another one), and reported as
algorithmic GB/s (the bytes the kernel must move, G = 16; the *_mx kernels use the E8M0
variant, group 32; compress_f32 / roundtrip_f32 take FP32 input; compress_2d reads a strided
[n/4096, 4096] view of an [n/4096, 8192] matrix, one TMA box per tile; the *_2d_blocks
kernels read (and roundtrip writes) [n/1024, 1024] views of [n/1024, 2048] matrices, one
box per block) and as a fraction of the measured
HBM copy bandwidth in MEASURED_PEAKS.json when that file is present. Inputs are N(0,1)
bfloat16 tensors made on the device (timing only; parity is the tests' business).
"""
from __future__ import annotations

import argparse
import json
import os

import numpy as np
import torch

import fp4_communication_compression_gb300 as fq

PAYLOAD = 0.5 + 1 / 16 + 4 / 256          # bytes per element of a G = 16 payload
PAYLOAD_MX = 0.5 + 1 / 32                 # bytes per element of an E8M0 (group 32) payload
ALG_BYTES = {
    "compress": 2 + PAYLOAD,
    "decompress_bf16_b1": PAYLOAD + 4,
    "decompress_bf16_b0": PAYLOAD + 2,
    "decompress_f32_b1": PAYLOAD + 8,
    "roundtrip": 4.0,
    "reduce_r2": 3 * PAYLOAD,
    "reduce_r4": 5 * PAYLOAD,
    "reduce_r8": 9 * PAYLOAD,
    "copy_bf16": 4.0,
    "compress_mx": 2 + PAYLOAD_MX,
    "decompress_mx_bf16_b1": PAYLOAD_MX + 4,
    "roundtrip_mx": 4.0,
    "reduce_mx_r4": 5 * PAYLOAD_MX,
    "compress_f32": 4 + PAYLOAD,
    "roundtrip_f32": 8.0,
    "compress_2d": 2 + PAYLOAD,
    "compress_2d_blocks": 2 + PAYLOAD,
    "roundtrip_2d_blocks": 4.0,
}


# the dual-scale BF16 kernels and a plain copy; the E8M0 (*_mx) and FP32-input kernels on request
DEFAULT_KERNELS = ["compress", "decompress_bf16_b1", "decompress_bf16_b0", "decompress_f32_b1", "roundtrip",
                   "reduce_r2", "reduce_r4", "reduce_r8", "copy_bf16"]


def peak_gbs():
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(path))["hbm_gbs"])
    except (OSError, KeyError, ValueError):
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--sizes", type=int, nargs="+", default=[1 << 24, 1 << 26, 1 << 28])
    ap.add_argument("--kernels", nargs="+", default=DEFAULT_KERNELS)
    ap.add_argument("--iters", type=int, default=30)
    args = ap.parse_args()
    dev = torch.device("cuda:0")
    peak = peak_gbs()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    clean = torch.ones(128 << 20, dtype=torch.float32, device=dev)

    def timed(fn):
        ts = []
        for i in range(args.iters + 3):
            flush.zero_()
            clean.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize(dev)
            if i >= 3:
                ts.append(a.elapsed_time(b) * 1e-3)
        return float(np.mean(ts))

    for n in args.sizes:
        x = torch.randn(n, device=dev).to(torch.bfloat16)
        ps = [fq.compress(x * (r + 1)) for r in range(8)]
        d16 = torch.zeros(n, dtype=torch.bfloat16, device=dev)
        d32 = torch.zeros(n, dtype=torch.float32, device=dev)
        y = torch.empty_like(x)
        out = torch.empty_like(ps[0])
        mx = any("_mx" in k for k in args.kernels)
        f32 = any(k in ("compress_f32", "roundtrip_f32") for k in args.kernels)
        xf = x.float() if f32 else None
        yf = torch.empty_like(xf) if f32 else None
        # rows of 4096 elements every 8192: the left half of a twice wider matrix
        wide = torch.empty(n // 4096, 8192, dtype=torch.bfloat16, device=dev) if "compress_2d" in args.kernels else None
        # rows of 1024 elements every 2048 (4 blocks per row: one TMA box per block)
        blocks = any(k.endswith("_2d_blocks") for k in args.kernels)
        nar = torch.empty(n // 1024, 2048, dtype=torch.bfloat16, device=dev) if blocks else None
        nar_y = torch.empty(n // 1024, 2048, dtype=torch.bfloat16, device=dev) if blocks else None
        if nar is not None:
            nar[:, :1024] = x.view(-1, 1024)
        if wide is not None:
            wide[:, :4096] = x.view(-1, 4096)
        pm = [fq.compress(x * (r + 1), scales="e8m0") for r in range(4)] if mx else None
        outm = torch.empty_like(pm[0]) if mx else None
        fns = {
            "compress": lambda: fq.compress(x, payload=ps[0]),
            "decompress_bf16_b1": lambda: fq.decompress_accumulate(ps[0], n, d16, beta=1),
            "decompress_bf16_b0": lambda: fq.decompress_accumulate(ps[0], n, d16, beta=0),
            "decompress_f32_b1": lambda: fq.decompress_accumulate(ps[0], n, d32, beta=1),
            "roundtrip": lambda: fq.roundtrip(x, y=y),
            "reduce_r2": lambda: fq.reduce_requantize(ps[:2], n, out=out),
            "reduce_r4": lambda: fq.reduce_requantize(ps[:4], n, out=out),
            "reduce_r8": lambda: fq.reduce_requantize(ps[:8], n, out=out),
            "copy_bf16": lambda: y.copy_(x),
            "compress_mx": lambda: fq.compress(x, payload=pm[0], scales="e8m0"),
            "decompress_mx_bf16_b1": lambda: fq.decompress_accumulate(pm[0], n, d16, beta=1, scales="e8m0"),
            "roundtrip_mx": lambda: fq.roundtrip(x, y=y, scales="e8m0"),
            "reduce_mx_r4": lambda: fq.reduce_requantize(pm[:4], n, out=outm, scales="e8m0"),
            "compress_f32": lambda: fq.compress(xf, payload=ps[0]),
            "roundtrip_f32": lambda: fq.roundtrip(xf, y=yf),
            "compress_2d": lambda: fq.compress(wide[:, :4096], payload=ps[0]),
            "compress_2d_blocks": lambda: fq.compress(nar[:, :1024], payload=ps[0]),
            "roundtrip_2d_blocks": lambda: fq.roundtrip(nar[:, :1024], y=nar_y[:, :1024]),
        }
        for k in args.kernels:
            t = timed(fns[k])
            gbs = ALG_BYTES[k] * n / t / 1e9
            print(json.dumps({"n": n, "kernel": k, "us": round(t * 1e6, 2), "alg_gbs": round(gbs, 1),
                              "frac_of_peak": None if not peak else round(gbs / peak, 4)}), flush=True)
        del x, ps, d16, d32, y, out, pm, outm, xf, yf, wide, nar, nar_y


if __name__ == "__main__":
    main()
