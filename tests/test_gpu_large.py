"""Parity above the size where the tiled kernels switch to one CTA per SM with dynamic tile
claims (384 tiles of 2048 elements per SM): n = 2^27 elements. The oracle checks a sample
of blocks one by one: blocks are independent, so the sampled blocks' codes and scales are
gathered into a small payload and compared with the oracle run on exactly those blocks."""
import numpy as np
import pytest
import torch

import oracle
import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import inputs

pytestmark = pytest.mark.gpu
N = 1 << 27
NB = N // 256


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def blocks():
    rng = np.random.default_rng(2027)
    return np.unique(np.concatenate([[0, 1, NB // 2, NB - 2, NB - 1], rng.choice(NB, 600, replace=False)]))


@pytest.fixture(scope="module")
def x(dev):
    rng = np.random.default_rng(27)
    xb = inputs.to_bf16_bits((rng.standard_normal(N, dtype=np.float32) *
                              np.exp(rng.uniform(-2, 2, NB).astype(np.float32)).repeat(256)))
    return xb, inputs.bits_to_torch(xb, dev)


def gather(payload, blocks, G, scales):
    """The sampled blocks' segments as the payload of len(blocks) * 256 elements."""
    p = payload if isinstance(payload, np.ndarray) else payload.cpu().numpy()
    gs = 256 // G
    codes = p[:N // 2].reshape(NB, 128)[blocks].ravel()
    g0 = N // 2
    gsc = p[g0:g0 + N // G].reshape(NB, gs)[blocks].ravel()
    m = blocks.size * 256
    out = np.zeros(oracle.payload_bytes(m, G, scales), np.uint8)
    out[:m // 2] = codes
    out[m // 2:m // 2 + m // G] = gsc
    if scales == "dual":
        b0 = g0 + (N // G + 15) // 16 * 16
        bsc = p[b0:b0 + 4 * NB].reshape(NB, 4)[blocks].ravel()
        ob = oracle.bscale_offset(m, G, scales)
        out[ob:ob + 4 * blocks.size] = bsc
    return out


def block_elems(blocks):
    return (blocks[:, None] * 256 + np.arange(256)[None, :]).ravel()


@pytest.mark.parametrize("scales,G,fwht", [("dual", 16, 1), ("dual", 32, 0), ("e8m0", 32, 1)])
def test_large_compress_decompress_roundtrip(dev, x, blocks, scales, G, fwht):
    xb, xt = x
    kw = dict(group=G, fwht=fwht, scales=scales)
    idx = block_elems(blocks)
    p = fq.compress(xt, **kw)
    want = oracle.compress(xb[idx], **kw)
    assert np.array_equal(gather(p, blocks, G, scales), want)
    d = torch.ones(N, dtype=torch.float32, device=dev)
    fq.decompress_accumulate(p, N, d, beta=1, **kw)
    ref = oracle.decompress_accumulate(want, idx.size, np.ones(idx.size, np.float32), beta=1, **kw)
    assert np.array_equal(d[torch.from_numpy(idx).to(dev)].cpu().numpy().view(np.uint32), ref.view(np.uint32))
    del d
    # BF16 destinations (the dynamic-claim decode at this size), beta = 0 and 1 onto 0.5
    for beta in (0, 1):
        d16 = torch.full((N,), 0.5, dtype=torch.bfloat16, device=dev)
        fq.decompress_accumulate(p, N, d16, beta=beta, **kw)
        ref16 = oracle.decompress_accumulate(want, idx.size, np.full(idx.size, 0x3F00, np.uint16), beta=beta, **kw)
        assert np.array_equal(inputs.torch_to_bits(d16[torch.from_numpy(idx).to(dev)]), ref16)
        del d16
    y = fq.roundtrip(xt, **kw)
    assert np.array_equal(inputs.torch_to_bits(y[torch.from_numpy(idx).to(dev)]), oracle.roundtrip(xb[idx], **kw))
    assert fq.fault_flags() == 0


@pytest.mark.parametrize("R", [2, 3, 4, 8])
def test_large_reduce(dev, x, blocks, R):
    """At 2^27 elements R = 2 and R >= 3 run their dynamic-claim CTAs (R = 3, 4 with the
    deferred pipeline start and the prefetched scales, R = 8 without)."""
    xb, xt = x
    idx = block_elems(blocks)
    pays = [fq.compress(xt * (1.0 + 0.25 * r)) for r in range(R)]
    out = fq.reduce_requantize(pays, N)
    want = oracle.reduce_requantize([gather(p, blocks, 16, "dual") for p in pays], idx.size)
    assert np.array_equal(gather(out, blocks, 16, "dual"), want)
    del pays
    assert fq.fault_flags() == 0


def test_large_f32_input_and_strided(dev, x, blocks):
    xb, xt = x
    idx = block_elems(blocks)
    xf = xt.float() * (1.0 + 2.0 ** -10)
    p = fq.compress(xf)
    assert np.array_equal(gather(p, blocks, 16, "dual"),
                          oracle.compress_f32(xf[torch.from_numpy(idx).to(dev)].cpu().numpy()))
    wide = torch.zeros(N // 4096, 4096 + 64, dtype=torch.bfloat16, device=dev)
    wide[:, :4096] = xt.view(-1, 4096)
    p2 = fq.compress(wide[:, :4096])
    assert torch.equal(p2, fq.compress(xt))
    assert fq.fault_flags() == 0
