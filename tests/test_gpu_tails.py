"""GPU vs oracle parity for lengths that are not a multiple of the 256-element block: the
full blocks go through the tiled kernels and the zero-padded last block through the
one-warp tail kernels. Payloads, every decode dtype and beta, roundtrip and reduce must be
bit-identical to the oracle, and nothing past the n-th element of an output may change."""
import numpy as np
import pytest
import torch

import oracle
import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import inputs

pytestmark = pytest.mark.gpu
FORMATS = [("dual", 16), ("dual", 32), ("e8m0", 32)]
GUARD = 64


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("fwht", [1, 0])
@pytest.mark.parametrize("scales,G", FORMATS)
@pytest.mark.parametrize("n", [1, 17, 100, 255, 257, 256 * 3 + 1, 2048 + 5, 256 * 8 * 7 + 131, (1 << 20) + 100,
                               (1 << 24) + 13])
def test_tail_lengths(dev, n, scales, G, fwht):
    kw = dict(group=G, fwht=fwht, scales=scales)
    x = inputs.sweep(-(-n // 4096) * 4096, seed=n % 13).ravel()[:n].copy()
    xt = inputs.bits_to_torch(x, dev)
    p = fq.compress(xt, **kw)
    want = oracle.compress(x, **kw)
    torch.cuda.synchronize()
    assert p.numel() == want.size == fq.payload_bytes(n, G, fwht, scales)
    assert np.array_equal(p.cpu().numpy(), want), "payload"
    rng = np.random.default_rng(n)
    for dt in ("bf16", "f32"):
        for beta in (0, 1):
            base = rng.standard_normal(n + GUARD).astype(np.float32)
            if dt == "bf16":
                d0 = inputs.to_bf16_bits(base)
                full = inputs.bits_to_torch(d0, dev).clone()
            else:
                d0 = base
                full = torch.from_numpy(base).to(dev)
            fq.decompress_accumulate(p, n, full[:n], beta=beta, **kw)
            ref = d0.copy()
            oracle.decompress_accumulate(want, n, ref[:n], beta=beta, **kw)
            got = inputs.torch_to_bits(full) if dt == "bf16" else full.cpu().numpy()
            assert np.array_equal(got.view(np.uint16 if dt == "bf16" else np.uint32),
                                  ref.view(np.uint16 if dt == "bf16" else np.uint32)), (dt, beta)
    yfull = torch.full((n + GUARD,), 7.0, dtype=torch.bfloat16, device=dev)
    fq.roundtrip(xt, y=yfull[:n], **kw)
    y = inputs.torch_to_bits(yfull)
    assert np.array_equal(y[:n], oracle.roundtrip(x, **kw)), "roundtrip"
    assert (inputs.bf16_bits_to_f32(y[n:]) == 7.0).all(), "roundtrip wrote past n"
    x2 = inputs.sweep(-(-n // 4096) * 4096, seed=n % 13 + 1).ravel()[:n].copy()
    p2 = fq.compress(inputs.bits_to_torch(x2, dev), **kw)
    r = fq.reduce_requantize([p, p2], n, **kw)
    rref = oracle.reduce_requantize([want, oracle.compress(x2, **kw)], n, group=G, scales=scales)
    torch.cuda.synchronize()
    assert np.array_equal(r.cpu().numpy(), rref), "reduce"
    assert fq.fault_flags() == 0
