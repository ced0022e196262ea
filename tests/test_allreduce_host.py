"""The compressed AllReduce's orchestration on CPU: shard plan arithmetic, and W gloo ranks
(127.0.0.1) running the reduce-scatter / fused reduce / all-gather / decode sequence with the
codec steps done by the CPU oracle on host tensors (the CUDA kernels are covered by
test_gpu_allreduce.py). Every rank's result must be bit-identical to the oracle's reduce of
all W full payloads followed by its decode: blocks are independent and the reduce sums in
rank order, so sharding may not change one bit."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from fp4_communication_compression_gb300 import inputs
from fp4_communication_compression_gb300.allreduce import CompressedAllReduce, ShardPlan


@pytest.mark.parametrize("n", [1, 255, 256, 2048, 256 * 37 + 100, 1 << 20, (1 << 20) + 3 * 256])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("group,scales", [(16, "dual"), (32, "dual"), (32, "e8m0")])
def test_shard_plan(n, world, group, scales):
    p = ShardPlan(n, world, group, scales)
    assert p.bps % 8 == 0 and p.bps > 0
    assert world * p.bps >= p.blocks                 # the shards cover the tensor
    assert p.bps - 8 < -(-p.blocks // world)         # and are the smallest whole tiles that do
    assert sum(p.shard_blocks(r) for r in range(world)) == p.blocks
    for b in p.slot_bytes():
        assert b % 16 == 0                      # every shard slice starts 16-byte aligned
    want = (128, 256 // group, 4) if scales == "dual" else (128, 8, 0)
    assert p.per_block == want


class OracleCodec:
    """The segment entry points restated on host tensors with the CPU oracle."""

    @staticmethod
    def _assemble(segs, n, group, scales):
        m = -(-n // 256) * 256
        g = oracle.gscale_offset(n, group, scales=scales)
        b = oracle.bscale_offset(n, group, scales=scales)
        total = oracle.payload_bytes(n, group, scales=scales)
        parts = [segs[0][:m // 2], segs[1][:b - g]] + ([segs[2][:total - b]] if total > b else [])
        return np.concatenate([p.numpy() for p in parts])

    @staticmethod
    def _scatter(p, segs, n, group, scales):
        g = oracle.gscale_offset(n, group, scales=scales)
        b = oracle.bscale_offset(n, group, scales=scales)
        segs[0][:g].copy_(torch.from_numpy(p[:g].copy()))
        segs[1][:b - g].copy_(torch.from_numpy(p[g:b].copy()))
        if p.size > b:
            segs[2][:p.size - b].copy_(torch.from_numpy(p[b:].copy()))

    def compress_segments(self, x, segs, group, fwht, scales):
        p = oracle.compress(inputs.torch_to_bits(x), group, fwht, scales=scales)
        self._scatter(p, segs, x.numel(), group, scales)

    def reduce_requantize_segments(self, ins, n, out, group, fwht, scales):
        ps = [self._assemble(s, n, group, scales) for s in ins]
        self._scatter(oracle.reduce_requantize(ps, n, group, scales=scales), out, n, group, scales)

    def decompress_accumulate_segments(self, segs, n, dst, beta, group, fwht, scales):
        p = self._assemble(segs, n, group, scales)
        d = inputs.torch_to_bits(dst).copy()
        oracle.decompress_accumulate(p, n, d, beta, group, fwht, scales=scales)
        dst.copy_(inputs.bits_to_torch(d))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_inputs(n, world, rank):
    return inputs.sweep(n, seed=100 + rank), inputs.sweep(n, seed=999)


def _worker(rank, world, port, n, kw, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, d0 = _rank_inputs(n, world, rank)
        ar = CompressedAllReduce(n, "cpu", codec=OracleCodec(), **kw)
        dst = inputs.bits_to_torch(d0).clone()
        for _ in range(2):                       # buffers are reused across calls
            dst = inputs.bits_to_torch(d0).clone()
            ar(inputs.bits_to_torch(x), dst, beta=1)
        q.put((rank, inputs.torch_to_bits(dst)))
    finally:
        dist.destroy_process_group()


def _reference(n, world, kw):
    group, fwht, scales = kw.get("group", 16), kw.get("fwht", 1), kw.get("scales", "dual")
    if scales == "e8m0":
        group = 32
    pays, d0 = [], None
    for r in range(world):
        x, d0 = _rank_inputs(n, world, r)
        pays.append(oracle.compress(x, group, fwht, scales=scales))
    red = oracle.reduce_requantize(pays, n, group, scales=scales)
    return oracle.decompress_accumulate(red, n, d0.copy(), 1, group, fwht, scales=scales)


@pytest.mark.parametrize("world,n,kw", [
    (2, 256 * 64, {}),
    (3, 256 * 37 + 100, {}),                     # last shard short, last block partial
    (2, 256 * 21, {"group": 32, "fwht": 0}),
    (4, 256 * 200 + 17, {"scales": "e8m0", "staging": "device"}),
])
def test_gloo_ranks_match_the_unsharded_reduce(world, n, kw):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n, kw, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = _reference(n, world, kw)
    for r in range(world):
        assert np.array_equal(res[r], want), f"rank {r} differs from the unsharded reduce"
