"""GPU vs oracle parity of the FP32-input entry points (fp4q_compress_f32,
fp4q_roundtrip_f32): payloads and FP32 roundtrips bit-identical to the oracle, for every
scale format, FWHT on and off, whole and partial last blocks."""
import numpy as np
import pytest
import torch

import oracle
import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import inputs

pytestmark = pytest.mark.gpu
FORMATS = [("dual", 16), ("dual", 32), ("e8m0", 32)]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    return torch.device("cuda:0")


def _f32_input(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n) * np.exp(rng.uniform(-4, 4, -(-n // 256)).repeat(256)[:n])
    x[rng.choice(n, max(1, n // 1000), replace=False)] *= 25.0
    return x.astype(np.float32)


@pytest.mark.parametrize("fwht", [1, 0])
@pytest.mark.parametrize("scales,G", FORMATS)
@pytest.mark.parametrize("n", [100, 256, 2048 + 5, 256 * 8 * 9 + 40, 1 << 20, (1 << 22) + 77])
def test_f32_input_parity(dev, n, scales, G, fwht):
    kw = dict(group=G, fwht=fwht, scales=scales)
    x = _f32_input(n, n % 17)
    xt = torch.from_numpy(x).to(dev)
    p = fq.compress(xt, **kw)
    torch.cuda.synchronize()
    assert np.array_equal(p.cpu().numpy(), oracle.compress_f32(x, **kw)), "payload"
    yfull = torch.full((n + 32,), 5.0, dtype=torch.float32, device=dev)
    fq.roundtrip(xt, y=yfull[:n], **kw)
    y = yfull.cpu().numpy()
    assert np.array_equal(y[:n].view(np.uint32), oracle.roundtrip_f32(x, **kw).view(np.uint32)), "roundtrip"
    assert (y[n:] == 5.0).all()
    d = torch.zeros(n, dtype=torch.float32, device=dev)
    fq.decompress_accumulate(p, n, d, beta=0, **kw)
    assert torch.equal(d, yfull[:n])


@pytest.mark.parametrize("scales,G", FORMATS)
def test_bf16_exact_f32_input_gives_the_bf16_payload(dev, scales, G):
    x = inputs.sweep(1 << 21, seed=2).ravel()
    xb = inputs.bits_to_torch(x, dev)
    for fwht in (0, 1):
        assert torch.equal(fq.compress(xb.float(), group=G, fwht=fwht, scales=scales),
                           fq.compress(xb, group=G, fwht=fwht, scales=scales))


def test_f32_gradient_16384x4096(dev):
    x = inputs.bf16_bits_to_f32(inputs.gradient().ravel()).astype(np.float32)
    x = x * np.float32(1.0 + 2.0 ** -12)           # leave the bfloat16 grid
    xt = torch.from_numpy(x).to(dev)
    for fwht in (0, 1):
        p = fq.compress(xt, fwht=fwht)
        y = fq.roundtrip(xt, fwht=fwht)
        torch.cuda.synchronize()
        assert np.array_equal(p.cpu().numpy(), oracle.compress_f32(x, fwht=fwht))
        assert np.array_equal(y.cpu().numpy().view(np.uint32), oracle.roundtrip_f32(x, fwht=fwht).view(np.uint32))
