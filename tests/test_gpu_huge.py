"""Parity past 32-bit element counts: n = 2^32 + 3 * 256 + 77 elements (8 GiB of bfloat16,
generated on the device). Element offsets pass 2^31 and 2^32 and the payload's code segment
passes 2^31 bytes; the kernels run their dynamic-claim grids, the last tile holds three blocks
and the last block is partial. Sampled blocks, including those on either side of the 2^31-
and 2^32-element boundaries and the tail, are gathered on the device and checked against the
oracle (blocks are independent, so a sample is a payload of its own). About 25 GB of device
memory at most."""
import numpy as np
import pytest
import torch

import oracle
import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import inputs

pytestmark = pytest.mark.gpu
N = (1 << 32) + 3 * 256 + 77
M = (N + 255) // 256 * 256
NB = M // 256
G = 16


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def blocks():
    rng = np.random.default_rng(4242)
    b31, b32 = (1 << 31) // 256, (1 << 32) // 256
    fixed = [0, 1, 7, 8, b31 - 8, b31 - 1, b31, b31 + 1, b31 + 8, b32 - 9, b32 - 8, b32 - 1,
             NB - 5, NB - 4, NB - 3, NB - 2, NB - 1]
    return np.unique(np.concatenate([fixed, rng.choice(NB, 300, replace=False)]))


@pytest.fixture(scope="module")
def x(dev):
    gen = torch.Generator(device=dev).manual_seed(77)
    t = torch.randn(N, generator=gen, device=dev, dtype=torch.bfloat16)
    t[:: (1 << 20) + 7] *= 20.0            # sparse outliers
    return t


def elems(t, blocks, dev):
    """The sampled blocks' elements as bfloat16 bits, zero past N (the payload's padding)."""
    idx = (blocks[:, None] * 256 + np.arange(256)[None, :]).ravel()
    ok = idx < N
    g = t[torch.from_numpy(np.minimum(idx, N - 1)).to(dev)]
    bits = inputs.torch_to_bits(g)
    bits[~ok] = 0
    return bits, ok


def gather(p, blocks, dev):
    """The sampled blocks' segments of payload p as the payload of len(blocks) * 256 elements."""
    b = torch.from_numpy(blocks).to(dev)
    codes = p[:M // 2].view(NB, 128)[b].cpu().numpy().ravel()
    g0 = M // 2
    gsc = p[g0:g0 + M // G].view(NB, 256 // G)[b].cpu().numpy().ravel()
    b0 = oracle.bscale_offset(M, G)
    bsc = p[b0:b0 + 4 * NB].view(NB, 4)[b].cpu().numpy().ravel()
    m = blocks.size * 256
    out = np.zeros(oracle.payload_bytes(m, G), np.uint8)
    out[:m // 2] = codes
    out[m // 2:m // 2 + m // G] = gsc
    ob = oracle.bscale_offset(m, G)
    out[ob:ob + 4 * blocks.size] = bsc
    return out


def test_codec_past_32_bit_counts(dev, x, blocks):
    assert fq.payload_bytes(N) == oracle.payload_bytes(N, G)
    p = fq.compress(x)
    xs, ok = elems(x, blocks, dev)
    want = oracle.compress(xs)
    assert np.array_equal(gather(p, blocks, dev), want)
    m = blocks.size * 256
    for beta in (0, 1):
        d = torch.full_like(x, 0.5)
        fq.decompress_accumulate(p, N, d, beta=beta)
        got, _ = elems(d, blocks, dev)
        ref = oracle.decompress_accumulate(want, m, np.full(m, 0x3F00, np.uint16), beta=beta)
        assert np.array_equal(got[ok], ref[ok])
        del d
    y = fq.roundtrip(x)
    got, _ = elems(y, blocks, dev)
    del y
    assert np.array_equal(got[ok], oracle.roundtrip(xs)[ok])
    assert fq.fault_flags() == 0


def test_two_rank_reduce_past_32_bit_counts(dev, x, blocks):
    p0 = fq.compress(x)
    x1 = x * -0.75
    p1 = fq.compress(x1)
    del x1
    red = fq.reduce_requantize([p0, p1], N)
    want = oracle.reduce_requantize([gather(p0, blocks, dev), gather(p1, blocks, dev)], blocks.size * 256)
    assert np.array_equal(gather(red, blocks, dev), want)
    assert fq.fault_flags() == 0
