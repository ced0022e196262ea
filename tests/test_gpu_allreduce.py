"""The compressed AllReduce on the GPU, and the segment entry points it is built on.

Segment calls must be bit-identical to the contiguous ones. The AllReduce runs as two
processes that share cuda:0 (each its own context and independent kernels; nothing waits on
the other process on the device), exchanging payload slices with gloo through host memory:
every rank's result must equal, bit for bit, the oracle's reduce of both full payloads
followed by its decode."""
import os
import socket

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


def _segs(n, dev, slack=0, **kw):
    return tuple(torch.full((b + slack,), 0x5A, dtype=torch.uint8, device=dev) if b else None
                 for b in fq.segment_bytes(n, **kw))


@pytest.mark.parametrize("kw", [{}, {"group": 32}, {"fwht": 0}, {"scales": "e8m0"}])
@pytest.mark.parametrize("n", [256 * 8, 256 * 37 + 5, 1 << 20])
def test_segments_equal_contiguous_calls(dev, n, kw):
    x = inputs.bits_to_torch(inputs.sweep(n, seed=4), dev)
    p = fq.compress(x, **kw)
    segs = _segs(n, dev, slack=64, **kw)
    fq.compress_segments(x, segs, **kw)
    g0, b0 = fq.gscale_offset(n, **kw), fq.bscale_offset(n, **kw)
    cb, gb, bb = fq.segment_bytes(n, **kw)
    pc = p.cpu().numpy()
    assert np.array_equal(segs[0][:cb].cpu().numpy(), pc[:g0])
    assert np.array_equal(segs[1][:gb].cpu().numpy(), pc[g0:b0])
    if bb:
        assert np.array_equal(segs[2][:bb].cpu().numpy(), pc[b0:])
    for s, b in zip(segs, (cb, gb, bb)):            # nothing written past a segment
        if s is not None:
            assert np.all(s[b:].cpu().numpy() == 0x5A)
    d1 = inputs.bits_to_torch(inputs.sweep(n, seed=5), dev)
    d2 = d1.clone()
    fq.decompress_accumulate(p, n, d1, beta=1, **kw)
    fq.decompress_accumulate_segments(segs, n, d2, beta=1, **kw)
    assert torch.equal(d1.view(torch.int16), d2.view(torch.int16))
    q = fq.compress(inputs.bits_to_torch(inputs.sweep(n, seed=6), dev), **kw)
    qs = _segs(n, dev, **kw)
    fq.compress_segments(inputs.bits_to_torch(inputs.sweep(n, seed=6), dev), qs, **kw)
    r1 = fq.reduce_requantize([p, q], n, **kw)
    r2 = _segs(n, dev, **kw)
    fq.reduce_requantize_segments([segs, qs], n, r2, **kw)
    rc = r1.cpu().numpy()
    assert np.array_equal(r2[0].cpu().numpy(), rc[:g0]) and np.array_equal(r2[1].cpu().numpy(), rc[g0:b0])
    if bb:
        assert np.array_equal(r2[2].cpu().numpy(), rc[b0:])
    assert fq.fault_flags() == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_inputs(n, rank):
    return inputs.sweep(n, seed=200 + rank), inputs.sweep(n, seed=777)


def _worker(rank, world, port, n, kw, q):
    import torch.distributed as dist
    from fp4_communication_compression_gb300.allreduce import CompressedAllReduce
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        x, d0 = _rank_inputs(n, rank)
        ar = CompressedAllReduce(n, dev, staging="host", **kw)
        xt = inputs.bits_to_torch(x, dev)
        for _ in range(2):                       # buffers are reused across calls
            dst = inputs.bits_to_torch(d0, dev).clone()
            ar(xt, dst, beta=1)
        own = fq.compress(xt, **kw)              # this rank's payload, as one contiguous buffer
        torch.cuda.synchronize()
        q.put((rank, inputs.torch_to_bits(dst), fq.fault_flags(), own.cpu().numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("n,kw", [((1 << 20) + 256 * 3 + 77, {}), (256 * 1000, {"group": 32, "fwht": 0}),
                                  ((1 << 20) + 256 * 5, {"fwht": 2})])
def test_two_process_allreduce_matches_oracle(dev, n, kw):
    """Every rank's result equals the oracle's reduce of the two ranks' full payloads followed
    by its decode. With the tensor-core encoder (fwht = 2, relaxed) the reference reduces the
    payloads the ranks' encoder wrote, so that the sharded exchange is still checked bit for
    bit."""
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n, kw, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        r, bits, flags, own = q.get(timeout=600)
        res[r] = (bits, flags, own)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    group, fwht = kw.get("group", 16), kw.get("fwht", 1)
    pays, d0 = [], None
    for r in range(world):
        x, d0 = _rank_inputs(n, r)
        pays.append(res[r][2] if fwht == 2 else oracle.compress(x, group, fwht))
    dec_fwht = min(fwht, 1)
    want = oracle.decompress_accumulate(oracle.reduce_requantize(pays, n, group), n, d0.copy(), 1, group, dec_fwht)
    for r in range(world):
        assert res[r][1] == 0, f"rank {r}: fault word set"
        assert np.array_equal(res[r][0], want), f"rank {r} differs from the oracle's unsharded reduce"


def _nccl_worker(port, n, kw, q):
    import torch.distributed as dist
    from fp4_communication_compression_gb300.allreduce import CompressedAllReduce
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), NCCL_NVLS_ENABLE="0")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=dev)
    try:
        x, d0 = _rank_inputs(n, 0)
        ar = CompressedAllReduce(n, dev, **kw)
        assert ar.staging == "device"
        xt = inputs.bits_to_torch(x, dev)
        for _ in range(2):
            dst = inputs.bits_to_torch(d0, dev).clone()
            ar(xt, dst, beta=1)
        torch.cuda.synchronize()
        q.put((inputs.torch_to_bits(dst), fq.fault_flags()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("n,kw", [((1 << 20) + 256 * 3 + 77, {}), (256 * 1000, {"scales": "e8m0"})])
def test_nccl_single_rank_allreduce_matches_oracle(dev, n, kw):
    """The NCCL path (payload slices staged on the device, NCCL all_to_all / all_gather) with the
    one rank a single GPU allows: the result equals the oracle's reduce of the rank's payload
    followed by its decode."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_nccl_worker, args=(_free_port(), n, kw, q))
    p.start()
    bits, flags = q.get(timeout=600)
    p.join(timeout=120)
    assert p.exitcode == 0
    scales = kw.get("scales", "dual")
    group = 32 if scales == "e8m0" else 16
    x, d0 = _rank_inputs(n, 0)
    pay = oracle.compress(x, group, 1, scales=scales)
    want = oracle.decompress_accumulate(oracle.reduce_requantize([pay], n, group, scales=scales), n, d0.copy(), 1,
                                        group, 1, scales=scales)
    assert flags == 0
    assert np.array_equal(bits, want)
