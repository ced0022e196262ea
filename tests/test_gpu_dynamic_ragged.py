"""Parity of the dynamic-claim kernels on ragged lengths. n = 2^26 + 3 * 256 + 77 elements is
above the size where compress, roundtrip, decompress-accumulate (BF16, beta = 0 and 1) and the
R <= 2 reduce claim their tiles dynamically; n = 12160 * 2048 + 5 * 256 + 33 is one ragged
tile above the smallest size where compress, roundtrip and decompress-accumulate do (4 tiles
of 2048 elements per warp, 20 (compress) or 16 (decompress) warps per SM, 152 SMs). In both
the last tile is partial and the last block is partial (zero-padded). The oracle checks a
sample of blocks one by one (blocks are independent) that includes the first, the middle, the
last full tile's and the tail blocks."""
import numpy as np
import pytest
import torch

import oracle
import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import inputs

pytestmark = pytest.mark.gpu
SIZES = [(1 << 26) + 3 * 256 + 77, 12160 * 2048 + 5 * 256 + 33]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    return torch.device("cuda:0")


class Case:
    def __init__(self, n):
        self.N = n
        self.M = (n + 255) // 256 * 256      # the payload's (padded) length
        self.NB = self.M // 256


@pytest.fixture(scope="module", params=SIZES, ids=["2p26_ragged", "threshold_ragged"])
def case(request):
    return Case(request.param)


@pytest.fixture(scope="module")
def blocks(case):
    NB = case.NB
    rng = np.random.default_rng(2609)
    fixed = [0, 1, 7, 8, NB // 2, NB - 12, NB - 9, NB - 5, NB - 4, NB - 3, NB - 2, NB - 1]
    return np.unique(np.concatenate([fixed, rng.choice(NB, 400, replace=False)]))


def make_x(case, seed):
    N, NB = case.N, case.NB
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(N, dtype=np.float32)
    v *= np.exp(rng.uniform(-2, 2, NB).astype(np.float32)).repeat(256)[:N]
    return inputs.to_bf16_bits(v)


@pytest.fixture(scope="module")
def xs(dev, case):
    return [make_x(case, s) for s in (261, 262)]


def sample_elems(case, bits, blocks):
    """The sampled blocks' elements, zero-padded past n (the payload's own padding)."""
    out = np.zeros((blocks.size, 256), bits.dtype)
    for i, b in enumerate(blocks):
        seg = bits[b * 256:min((b + 1) * 256, case.N)]
        out[i, :seg.size] = seg
    return out.ravel()


def valid_mask(case, blocks):
    return ((blocks[:, None] * 256 + np.arange(256)[None, :]) < case.N).ravel()


def gather(case, payload, blocks, G=16):
    """The sampled blocks' segments as the payload of len(blocks) * 256 elements."""
    M, NB = case.M, case.NB
    p = payload.cpu().numpy()
    gs = 256 // G
    codes = p[:M // 2].reshape(NB, 128)[blocks].ravel()
    g0 = M // 2
    gsc = p[g0:g0 + M // G].reshape(NB, gs)[blocks].ravel()
    b0 = g0 + (M // G + 15) // 16 * 16
    bsc = p[b0:b0 + 4 * NB].reshape(NB, 4)[blocks].ravel()
    m = blocks.size * 256
    out = np.zeros(oracle.payload_bytes(m, G), np.uint8)
    out[:m // 2] = codes
    out[m // 2:m // 2 + m // G] = gsc
    ob = oracle.bscale_offset(m, G)
    out[ob:ob + 4 * blocks.size] = bsc
    return out


def test_compress_and_decompress_accumulate(dev, case, xs, blocks):
    xb = xs[0]
    p = fq.compress(inputs.bits_to_torch(xb, dev))
    want = oracle.compress(sample_elems(case, xb, blocks))
    assert np.array_equal(gather(case, p, blocks), want)
    # beta = 1 into a BF16 residual
    resid = make_x(case, 263)
    d = inputs.bits_to_torch(resid, dev).clone()
    fq.decompress_accumulate(p, case.N, d, beta=1)
    got = inputs.torch_to_bits(d)
    ref = oracle.decompress_accumulate(want, blocks.size * 256, sample_elems(case, resid, blocks), beta=1)
    keep = valid_mask(case, blocks)
    assert np.array_equal(sample_elems(case, got, blocks)[keep], ref[keep])
    # beta = 0 (the decode alone) into a BF16 buffer
    d0 = torch.full_like(d, 3.0)
    fq.decompress_accumulate(p, case.N, d0, beta=0)
    ref0 = oracle.decompress_accumulate(want, blocks.size * 256, np.zeros(blocks.size * 256, np.uint16), beta=0)
    assert np.array_equal(sample_elems(case, inputs.torch_to_bits(d0), blocks)[keep], ref0[keep])
    assert fq.fault_flags() == 0


def test_roundtrip(dev, case, xs, blocks):
    xb = xs[1]
    y = fq.roundtrip(inputs.bits_to_torch(xb, dev))
    got = sample_elems(case, inputs.torch_to_bits(y), blocks)
    ref = oracle.roundtrip(sample_elems(case, xb, blocks))
    keep = valid_mask(case, blocks)
    assert np.array_equal(got[keep], ref[keep])
    assert fq.fault_flags() == 0


def test_two_rank_reduce(dev, case, xs, blocks):
    pays = [fq.compress(inputs.bits_to_torch(x, dev)) for x in xs]
    red = fq.reduce_requantize(pays, case.N)
    want = oracle.reduce_requantize([gather(case, p, blocks) for p in pays], blocks.size * 256)
    assert np.array_equal(gather(case, red, blocks), want)
    assert fq.fault_flags() == 0
