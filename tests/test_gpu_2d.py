"""Strided 2-D views on the GPU (fp4q_compress_2d, fp4q_decompress_accumulate_2d,
fp4q_roundtrip_2d): the payload of a [rows, cols] view with row stride ld is the payload of
its dense row-major copy (the oracle is run on that copy), decoded values land in a strided
destination, and the elements between rows are never touched."""
import numpy as np
import pytest
import torch

import oracle
import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import inputs

pytestmark = pytest.mark.gpu
FORMATS = [("dual", 16), ("dual", 32), ("e8m0", 32)]
SHAPES = [(4, 512, 1024), (3, 256, 264), (7, 2048, 2056), (33, 768, 1024), (5, 2304, 2312), (1000, 4096, 8192)]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("fwht", [1, 0])
@pytest.mark.parametrize("scales,G", FORMATS)
@pytest.mark.parametrize("rows,cols,ld", SHAPES)
def test_strided_2d(dev, rows, cols, ld, scales, G, fwht):
    kw = dict(group=G, fwht=fwht, scales=scales)
    full = inputs.sweep(-(-rows * ld // 4096) * 4096, seed=rows + cols).ravel()[:rows * ld].reshape(rows, ld)
    dense = np.ascontiguousarray(full[:, :cols]).ravel()
    xt = inputs.bits_to_torch(full.ravel(), dev).view(rows, ld)
    view = xt[:, :cols]
    assert not view.is_contiguous()
    p = fq.compress(view, **kw)
    want = oracle.compress(dense, **kw)
    torch.cuda.synchronize()
    assert np.array_equal(p.cpu().numpy(), want), "payload"
    assert torch.equal(p, fq.compress(view.contiguous(), **kw))
    n = rows * cols
    rng = np.random.default_rng(rows)
    for dt in ("bf16", "f32"):
        for beta in (0, 1):
            ldd = ld if dt == "bf16" else ld + 4
            base = rng.standard_normal(rows * ldd).astype(np.float32)
            if dt == "bf16":
                b0 = inputs.to_bf16_bits(base)
                dfull = inputs.bits_to_torch(b0, dev).view(rows, ldd)
            else:
                b0 = base
                dfull = torch.from_numpy(base.copy()).to(dev).view(rows, ldd)
            fq.decompress_accumulate(p, n, dfull[:, :cols], beta=beta, **kw)
            ref = b0.copy().reshape(rows, ldd)
            dense_dst = np.ascontiguousarray(ref[:, :cols]).ravel()
            oracle.decompress_accumulate(want, n, dense_dst, beta=beta, **kw)
            ref[:, :cols] = dense_dst.reshape(rows, cols)
            got = (inputs.torch_to_bits(dfull) if dt == "bf16" else dfull.cpu().numpy()).reshape(rows, ldd)
            assert np.array_equal(got.view(np.uint16 if dt == "bf16" else np.uint32),
                                  ref.view(np.uint16 if dt == "bf16" else np.uint32)), (dt, beta)
    yfull = torch.full((rows, ld + 8), 9.0, dtype=torch.bfloat16, device=dev)
    fq.roundtrip(view, y=yfull[:, :cols], **kw)
    y = inputs.torch_to_bits(yfull).reshape(rows, ld + 8)
    assert np.array_equal(np.ascontiguousarray(y[:, :cols]).ravel(), oracle.roundtrip(dense, **kw)), "roundtrip"
    assert (inputs.bf16_bits_to_f32(y[:, cols:]) == 9.0).all(), "roundtrip wrote between rows"
    assert fq.fault_flags() == 0
