"""Compressed AllReduce across ranks: the tensor-parallel AllReduce of FP4Quant with every
exchanged tensor in the FP4 payload format.

Method: "4-bit compression speeds up LLM training by 56 percent" (zot.news), "Read it as":
the communication being compressed is the AllReduce of tensor parallelism; "FP4Quant"
(shd-paper.top), abstract: the payloads are the micro-grouped dual-scale FP4 format. The
pages do not say how the reduction itself is organised; this module takes the plain
reduce-scatter / all-gather form, in which no rank ever sums uncompressed partials of
another rank:

  1. compress: each rank compresses its partial x_r (n elements) into a payload whose three
     segments (codes, group scales, block scales) are laid out over W shards of `bps` blocks
     each (bps a whole number of 8-block tiles, so every shard boundary is 16-byte aligned
     in every segment; blocks past the tensor's end stay zero);
  2. reduce-scatter of payload slices: all_to_all of each segment, so the owner of shard s
     receives shard s of every rank's payload, in rank order;
  3. the owner runs the fused decompress-sum-requantize (fp4q_reduce_requantize_segments)
     over the W received slices: decode in the transform domain, FP32 sum in rank order,
     requantize;
  4. all-gather of the requantized shards (each segment), which reassembles one payload of
     the whole tensor in the contiguous segment order;
  5. decompress-accumulate of that payload into dst on every rank.

Blocks are independent and the reduce sums in rank order, so the result on every rank is
bit-identical to fp4q_reduce_requantize of the W full payloads followed by
fp4q_decompress_accumulate. The collectives are torch.distributed's (NCCL on GPUs, no
multicast); with a backend that needs host tensors (gloo) the slices are staged through host
memory. Every codec step runs in the CUDA kernels of the library; this module only plans
the shards, owns the buffers and issues the collectives.
"""
from __future__ import annotations

from dataclasses import dataclass

BLOCK = 256
TILE_BLOCKS = 8           # shard boundaries fall on whole 8-block tiles


@dataclass(frozen=True)
class ShardPlan:
    """Block-aligned split of an n-element tensor over `world` ranks."""
    n: int
    world: int
    group: int = 16
    scales: str = "dual"

    @property
    def blocks(self) -> int:
        return -(-self.n // BLOCK)

    @property
    def bps(self) -> int:
        """Blocks per shard: ceil(blocks / world) rounded up to whole 8-block tiles."""
        per = -(-self.blocks // self.world)
        return -(-per // TILE_BLOCKS) * TILE_BLOCKS

    @property
    def per_block(self):
        """Bytes per block of each segment: codes, group scales, block scales."""
        if self.scales == "e8m0":
            return (BLOCK // 2, BLOCK // 32, 0)
        return (BLOCK // 2, BLOCK // self.group, 4)

    def slot_bytes(self):
        """Bytes of one shard in each segment."""
        return tuple(self.bps * b for b in self.per_block)

    def shard_blocks(self, rank: int) -> int:
        """Real (non-padding) blocks of shard `rank`."""
        return max(0, min(self.bps, self.blocks - rank * self.bps))

    @property
    def shard_elems(self) -> int:
        return self.bps * BLOCK


class CudaCodec:
    """The library's segment entry points (the default codec of CompressedAllReduce)."""

    def __init__(self):
        from . import compress_segments, decompress_accumulate_segments, reduce_requantize_segments
        self.compress_segments = compress_segments
        self.decompress_accumulate_segments = decompress_accumulate_segments
        self.reduce_requantize_segments = reduce_requantize_segments


class CompressedAllReduce:
    """dst = beta * dst + decode(AllReduce_FP4(x)) over the ranks of a process group, for
    tensors of n elements (bfloat16 or float32 x; bfloat16 or float32 dst).

    Buffers for one n are allocated once (zeroed) and reused by every call. The host-staged
    mode copies each segment to host memory around the collectives (for gloo)."""

    def __init__(self, n: int, device, process_group=None, group: int = 16, fwht: int = 1,
                 scales: str = "dual", staging: str | None = None, codec=None):
        import torch
        import torch.distributed as dist
        self.dist = dist
        self.pg = process_group
        self.world = dist.get_world_size(process_group)
        self.rank = dist.get_rank(process_group)
        if self.world > 8:
            raise ValueError("the fused reduce takes at most 8 ranks")
        self.kw = dict(group=group if scales != "e8m0" else 32, fwht=fwht, scales=scales)
        self.plan = ShardPlan(int(n), self.world, self.kw["group"], scales)
        if staging is None:
            staging = "device" if dist.get_backend(process_group) == "nccl" else "host"
        if staging not in ("device", "host"):
            raise ValueError("staging must be 'device' or 'host'")
        self.staging = staging
        self.device = torch.device(device)
        self.codec = codec if codec is not None else CudaCodec()
        W = self.world
        slots = self.plan.slot_bytes()

        def bufs(count, where=None):
            return [torch.zeros(count * b, dtype=torch.uint8, device=where or self.device) if b else None
                    for b in slots]
        self.send = bufs(W)              # this rank's payload, W shards per segment
        self.recv = bufs(W)              # shard `rank` of every rank's payload, in rank order
        self.out = bufs(1)               # the requantized shard this rank owns
        self.gath = bufs(W)              # the requantized payload of the whole tensor
        if staging == "host":
            self.h_send, self.h_recv, self.h_out, self.h_gath = (bufs(W, "cpu"), bufs(W, "cpu"), bufs(1, "cpu"),
                                                                 bufs(W, "cpu"))

    # ------------------------------------------------------------------ collectives

    def _exchange(self, src, dst, hsrc, hdst, gather: bool):
        """all_to_all (gather=False) or all_gather_into_tensor (gather=True) of every segment."""
        for i in range(3):
            if src[i] is None:
                continue
            a, b = src[i], dst[i]
            if self.staging == "host":
                hsrc[i].copy_(a)
                a, b = hsrc[i], hdst[i]
            if gather:
                self.dist.all_gather_into_tensor(b, a, group=self.pg)
            else:
                self.dist.all_to_all_single(b, a, group=self.pg)
            if self.staging == "host":
                dst[i].copy_(b)

    def _slot(self, segs, r):
        """Segment slices of shard slot r."""
        return tuple(None if s is None else s[r * b:(r + 1) * b] for s, b in zip(segs, self.plan.slot_bytes()))

    # ------------------------------------------------------------------ the allreduce

    def __call__(self, x, dst, beta: int = 1):
        n, W = self.plan.n, self.world
        if x.numel() != n or dst.numel() != n:
            raise ValueError(f"x and dst must have {n} elements")
        c = self.codec
        # 1. compress into the W-shard segment layout
        c.compress_segments(x, tuple(self.send), **self.kw)
        # 2. reduce-scatter of payload slices
        self._exchange(self.send, self.recv, getattr(self, "h_send", None), getattr(self, "h_recv", None), False)
        # 3. the owner's fused decompress-sum-requantize over the W slices, in rank order
        ins = [self._slot(self.recv, r) for r in range(W)]
        c.reduce_requantize_segments(ins, self.plan.shard_elems, tuple(self.out), **self.kw)
        # 4. all-gather of the requantized shards
        self._exchange(self.out, self.gath, getattr(self, "h_out", None), getattr(self, "h_gath", None), True)
        # 5. decode the whole tensor's payload into dst
        c.decompress_accumulate_segments(tuple(self.gath), n, dst, beta=beta, **self.kw)
        return dst
