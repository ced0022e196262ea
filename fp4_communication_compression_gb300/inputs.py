"""Seeded synthetic inputs for the FP4 codec (no codec arithmetic lives here).

Every tensor is drawn on the host with ``numpy.random.default_rng(seed)`` (PCG64) in
float32, then rounded to bfloat16 (round to nearest even, by torch) so that the CUDA path
and the CPU oracle receive identical bits. Generation order inside one tensor: base
values, then outlier positions (``rng.choice(..., replace=False)``), then outlier signs or
noise.

The five workloads stand in for the tensors a tensor-parallel AllReduce of a 7B-class
model (hidden size 4096) exchanges; the pages on the method name Qwen-7B but publish no
tensors, so all of them are synthetic:

  toy       [8, 512]        N(0,1), 4 entries set to +-40                       seed 0 (and 1)
  tp_act    [4096, 4096]    N(0,1), 4 hidden channels (0.1%) = 20 * Student-t(3)   seed 0
  reduce4   4 x [8192,4096] as toy: N(0,1), 4 entries +-40 per buffer           seeds 1..4
  grad      [16384, 4096]   Laplace(0, 1e-3), 0.01% of entries (6711) x 100      seed 0
  sweep(n)  [n], n = 2^15, 2^17, ..., 2^29   N(0,1), 0.1% of entries x 20        seed 0
"""
from __future__ import annotations

import numpy as np

SWEEP_SIZES = [1 << k for k in range(15, 30, 2)]   # 64 KiB ... 1 GiB of bfloat16


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16) via torch's round-to-nearest-even cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bits_to_torch(h: np.ndarray, device=None):
    """uint16 bfloat16 bit patterns -> torch.bfloat16 tensor (optionally on a device)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(h, np.uint16).view(np.int16)).view(torch.bfloat16)
    return t if device is None else t.to(device)


def torch_to_bits(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _normal(rng, n):
    return rng.standard_normal(n, dtype=np.float32)


def toy(seed: int = 0) -> np.ndarray:
    """[8, 512] N(0,1) with 4 entries set to +-40 (sign drawn from the generator)."""
    rng = np.random.default_rng(seed)
    n = 8 * 512
    x = _normal(rng, n)
    idx = rng.choice(n, 4, replace=False)
    sign = np.where(rng.integers(0, 2, 4) == 0, -1.0, 1.0).astype(np.float32)
    x[idx] = 40.0 * sign
    return to_bf16_bits(x).reshape(8, 512)


def tp_activation(seed: int = 0, tokens: int = 4096, hidden: int = 4096) -> np.ndarray:
    """[tokens, hidden] N(0,1); round(0.001 * hidden) channels replaced by 20 * t(df=3)."""
    rng = np.random.default_rng(seed)
    x = _normal(rng, tokens * hidden).reshape(tokens, hidden)
    k = int(round(0.001 * hidden))
    cols = rng.choice(hidden, k, replace=False)
    x[:, cols] = (20.0 * rng.standard_t(3, size=(tokens, k))).astype(np.float32)
    return to_bf16_bits(x)


def reduce_ranks(R: int = 4, tokens: int = 8192, hidden: int = 4096, first_seed: int = 1):
    """R buffers [tokens, hidden], each N(0,1) with 4 entries +-40, seeds first_seed.."""
    out = []
    for r in range(R):
        rng = np.random.default_rng(first_seed + r)
        n = tokens * hidden
        x = _normal(rng, n)
        idx = rng.choice(n, 4, replace=False)
        sign = np.where(rng.integers(0, 2, 4) == 0, -1.0, 1.0).astype(np.float32)
        x[idx] = 40.0 * sign
        out.append(to_bf16_bits(x).reshape(tokens, hidden))
    return out


def gradient(seed: int = 0, rows: int = 16384, hidden: int = 4096) -> np.ndarray:
    """[rows, hidden] Laplace(0, 1e-3); round(1e-4 * n) entries multiplied by 100."""
    rng = np.random.default_rng(seed)
    n = rows * hidden
    x = rng.laplace(0.0, 1e-3, n).astype(np.float32)
    k = int(round(1e-4 * n))
    idx = rng.choice(n, k, replace=False)
    x[idx] *= 100.0
    return to_bf16_bits(x).reshape(rows, hidden)


def sweep(n: int, seed: int = 0) -> np.ndarray:
    """1-D [n] N(0,1); round(0.001 * n) entries multiplied by 20."""
    rng = np.random.default_rng(seed)
    x = _normal(rng, n)
    k = int(round(0.001 * n))
    idx = rng.choice(n, k, replace=False)
    x[idx] *= 20.0
    return to_bf16_bits(x)


def edge_blocks() -> np.ndarray:
    """Hand-picked 256-element blocks that reach the contract's special cases: all zero,
    all -0, constant, one spike, tiny (subnormal-range) values, values near 2^119, exact
    E4M3/E2M1 ties, alternating signs, spikes at and just below the zero-block limit. Returned as bfloat16 bits, shape [k, 256]."""
    f = np.float32
    blocks = []
    blocks.append(np.zeros(256, f))
    blocks.append(np.full(256, -0.0, f))
    blocks.append(np.full(256, 0.041015625, f))            # 168 * 2^-12: exact round trip
    b = np.zeros(256, f); b[37] = 3.0; blocks.append(b)
    b = np.zeros(256, f); b[0] = 2.0 ** -24; b[1] = -(2.0 ** -24); blocks.append(b)
    blocks.append((np.arange(256, dtype=f) - 128.0) * f(2.0 ** -130))   # subnormal range
    blocks.append(np.full(256, 2.0 ** -90, f) * np.where(np.arange(256) % 2 == 0, 1, -1).astype(f))
    b = np.zeros(256, f); b[5] = 2.0 ** 119; b[6] = -(2.0 ** 118); blocks.append(b)
    blocks.append(np.where(np.arange(256) % 3 == 0, 1.0, -1.0).astype(f) * f(1.5))
    blocks.append(np.linspace(-6.0, 6.0, 256, dtype=f))
    # fwht = 0 ties: group maxima giving r = 136 and 152 (E4M3 ties) and E2M1 midpoints.
    b = np.zeros(256, f)
    b[0:16] = [5.25, -3.5, 2.625, -1.75, 1.3125, 0.875, -0.4375, 0, 0.4375, -0.875, 1.75,
               -2.625, 3.5, -5.25, 0.875, -1.3125]
    b[32:48] = [1.5625, 1.4375, 1.25, 0.625, 0.375, 0.0625, -0.0625, 0.1875, 0.3125, 0.4375,
                0.875, -1.25, -0.625, 0.125, 0.25, 0.5]
    b[48] = 1.59375
    b[64] = 1.78125
    b[80] = 2.0 ** -24; b[81] = -(2.0 ** -24)
    blocks.append(b)
    # the zero-block limit A = 2688 * 2^-100 = 1.3125 * 2^-89 (a bfloat16 value): one spike at
    # the limit and one a bfloat16 ulp below it, without the transform (A = |x|) and with it
    # (a lone spike spreads to |x| / 16 on every element)
    lim, below = 1.3125 * 2.0 ** -89, (1.3125 - 2.0 ** -7) * 2.0 ** -89
    for v, at in ((lim, 9), (-below, 200), (-16 * lim, 77), (16 * below, 140)):
        b = np.zeros(256, f); b[at] = v; blocks.append(b)
    return np.stack([to_bf16_bits(x) for x in blocks])
