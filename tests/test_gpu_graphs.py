"""The codec's launches inside a captured CUDA graph: a step (compress, a 2-rank reduce,
decompress-accumulate into a BF16 residual) captured once and replayed on new input contents
gives, every replay, the bytes the same calls give eagerly; and the oracle agrees with both.
Sizes cover the fixed grid (2^20 elements) and the dynamic tile claims (2^25). The library
keeps no per-launch host state that a replay could not see: tensor maps are kernel
parameters, tile claims are per-CTA shared-memory counters."""
import numpy as np
import pytest
import torch

import oracle
import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    return torch.device("cuda:0")


def _step(xa, xb, pa, pb, red, dst, n, stream):
    fq.compress(xa, payload=pa, stream=stream)
    fq.compress(xb, payload=pb, stream=stream)
    fq.reduce_requantize([pa, pb], n, out=red, stream=stream)
    fq.decompress_accumulate(red, n, dst, beta=1, stream=stream)


@pytest.mark.parametrize("n", [1 << 20, 1 << 25])
def test_captured_step_replays_like_eager_calls(dev, n):
    pb_bytes = fq.payload_bytes(n)
    xa = torch.empty(n, dtype=torch.bfloat16, device=dev)
    xb = torch.empty_like(xa)
    dst = torch.empty_like(xa)
    pa, pb, red = (torch.empty(pb_bytes, dtype=torch.uint8, device=dev) for _ in range(3))
    s = torch.cuda.Stream(dev)
    # warm the library's per-kernel caches outside the capture, then capture one step
    xa.normal_(); xb.normal_(); dst.zero_()
    with torch.cuda.stream(s):
        _step(xa, xb, pa, pb, red, dst, n, s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _step(xa, xb, pa, pb, red, dst, n, s)
    for seed in (11, 12, 13):
        gen = torch.Generator(device=dev).manual_seed(seed)
        a = torch.randn(n, generator=gen, device=dev).to(torch.bfloat16)
        b = (3.0 * torch.randn(n, generator=gen, device=dev)).to(torch.bfloat16)
        r = torch.randn(n, generator=gen, device=dev).to(torch.bfloat16)
        xa.copy_(a); xb.copy_(b); dst.copy_(r)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        got = (pa.clone(), pb.clone(), red.clone(), dst.clone())
        # the same calls, eagerly, on copies of the same inputs
        ea, eb, ered = (torch.empty_like(pa) for _ in range(3))
        edst = r.clone()
        _step(a, b, ea, eb, ered, edst, n, torch.cuda.current_stream(dev))
        torch.cuda.synchronize()
        assert torch.equal(got[0], ea) and torch.equal(got[1], eb) and torch.equal(got[2], ered)
        assert torch.equal(got[3].view(torch.int16), edst.view(torch.int16))
        assert fq.fault_flags() == 0
    # the oracle on a slice of whole blocks (blocks are independent) of the last replay
    k = 64 * 256
    ab, bb = inputs.torch_to_bits(a[:k]), inputs.torch_to_bits(b[:k])
    pa_o, pb_o = oracle.compress(ab), oracle.compress(bb)
    red_o = oracle.reduce_requantize([pa_o, pb_o], k)
    dst_o = oracle.decompress_accumulate(red_o, k, inputs.torch_to_bits(r[:k]), beta=1)
    assert np.array_equal(inputs.torch_to_bits(got[3][:k]), dst_o)
