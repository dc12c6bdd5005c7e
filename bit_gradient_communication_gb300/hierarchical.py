"""Hierarchical pipeline-A low-bit all-reduce: local reduce -> inter low-bit
all-reduce -> local broadcast (bitscom README, "Implemented Features":
hierarchical pipeline-A; multi-node dual-stream scheduling for pipeline-A,
warmup -> steady -> cooldown; "Hierarchical All-Reduce Options": local_group,
inter_group, chunk_size, local_quantize).

Ranks form local groups (nodes) of L ranks; local rank 0 of every group is its
leader, and the leaders form the inter group (G leaders).  The flat gradient
is processed in pipeline chunks of chunk_size elements.  For chunk k:

  local reduce     the leader gets the sum of its group's chunk, ranks in order:
                   local_quantize=False (the default): the full-precision
                   chunks are gathered and summed in fp32 (bitscom_sum_ranks);
                   local_quantize=True: every local rank encodes its chunk
                   (its own local error buffer) and the leader decodes the L
                   ranks' codes into their rank-ordered sum (the decoder
                   without requantisation);
  inter all-reduce the leaders run the low-bit all-reduce of sharded.py on
                   their local sums, the chunk being one fusion bucket (encoder
                   with the leader's inter error buffer, all-to-all, decode +
                   stage-2 requantisation of its share, all-gather), and decode
                   the gathered codes: out = fl(fl(s*q) * mul);
  local broadcast  the leader sends the chunk to its group: the decoded values
                   (local_quantize=False) or the gathered codes and scales,
                   which every rank decodes itself (local_quantize=True; the
                   same bits).

Pipelining: the local reduce of chunk k+1 is issued before the inter
all-reduce of chunk k, and chunk k's broadcast before chunk k+1's inter
stage (warmup: local reduce of chunk 0; steady state; cooldown: the last inter
stages and broadcasts).  The local and inter groups are separate
communicators, so their transfers overlap; every result depends only on its
chunk, so the schedule cannot change the bits.

Philox indices are global element indices in windows of n per step: the local
stage draws from Philox stream 2 (stage 1 of the inter all-reduce uses 0, its
stage 2 stream 1).
"""
from __future__ import annotations

import dataclasses
import sys
from typing import Optional

from . import QParams
from .sharded import Exchange, LowBitAllReduce, code_bytes, scale_count

LOCAL_PHILOX_STREAM = 2


class PipelineA:
    """One rank's hierarchical low-bit all-reduce of a flat gradient of n elements.

    local: Exchange over this rank's local group (rank 0 = the leader).
    inter: Exchange over the leaders (None on the other ranks).
    p_inter: the leader's stage-1 parameters of the inter all-reduce (its
        seed); p2: stage-2 parameters; p_local: this rank's parameters of the
        quantised local stage (local_quantize=True; its seed).
    codec: the codec steps (default: libbitscom through this package's binding).
    """

    def __init__(self, n: int, dtype, local: Exchange, inter: Optional[Exchange], p_inter: QParams, p2: QParams,
                 chunk_size: int = 1 << 20, local_quantize: bool = False, p_local: Optional[QParams] = None,
                 error_feedback: bool = True, stage2_error_feedback: bool = True, device=None, codec=None):
        import torch
        self.torch = torch
        self.codec = codec if codec is not None else sys.modules[__package__]
        self.local, self.inter = local, inter
        self.L, self.lrank = local.world, local.rank
        self.leader = self.lrank == 0
        if self.leader != (inter is not None):
            raise ValueError("the inter exchange is given on the leaders (local rank 0) only")
        self.n, self.dtype = n, dtype
        self.local_quantize = local_quantize
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.p2 = p2
        if local_quantize and p_local is None:
            raise ValueError("local_quantize needs p_local")
        self.p_local = (dataclasses.replace(p_local, philox_stream=LOCAL_PHILOX_STREAM)
                        if p_local is not None else None)
        U = max(p_inter.block, p2.block, 128, p_local.block if p_local is not None else 0)
        if chunk_size % U:
            raise ValueError(f"chunk_size must be a multiple of {U}")
        self.chunk_size = chunk_size
        self.step = 0
        dev, f32 = self.device, torch.float32
        # the inter all-reduce on the leaders: its fusion buckets are the pipeline chunks
        self.ar = None
        if self.leader:
            self.ar = LowBitAllReduce(n, f32, p_inter, p2, device=dev, error_feedback=error_feedback,
                                      stage2_error_feedback=stage2_error_feedback, bucket_bytes=4 * chunk_size,
                                      codec=self.codec, exchange=inter)
            self.chunks = [(bk.b0, bk.b0 + bk.n) for bk in self.ar.buckets]
        else:
            self.chunks = [(c0, min(c0 + chunk_size, n)) for c0 in range(0, n, chunk_size)]
        cmax = max([c1 - c0 for c0, c1 in self.chunks] or [0])
        self.err_local = torch.zeros(n, dtype=f32, device=dev) if (local_quantize and error_feedback) else None
        # per-chunk buffers (two of each, chunks alternate between them)
        self._r = [torch.empty(cmax, dtype=f32, device=dev) for _ in range(2)]
        if self.leader:
            self._recv = [[torch.empty(cmax, dtype=dtype, device=dev) for _ in range(self.L)] for _ in range(2)]
        if local_quantize:
            pl = self.p_local
            lc, ls = code_bytes(0, cmax, pl.bits, pl.block), scale_count(0, cmax, pl.block)
            self._lc = [torch.empty(lc, dtype=torch.uint8, device=dev) for _ in range(2)]
            self._ls = [torch.empty(ls, dtype=torch.int16, device=dev) for _ in range(2)]
            if self.leader:
                self._glc = [[torch.empty(lc, dtype=torch.uint8, device=dev) for _ in range(self.L)] for _ in range(2)]
                self._gls = [[torch.empty(2 * ls, dtype=torch.uint8, device=dev) for _ in range(self.L)]
                             for _ in range(2)]
            bc2, bs2 = code_bytes(0, cmax, p2.bits, p2.block), scale_count(0, cmax, p2.block)
            self._bcodes = [torch.empty(bc2, dtype=torch.uint8, device=dev) for _ in range(2)]
            self._bscales = [torch.empty(bs2, dtype=torch.int16, device=dev) for _ in range(2)]

    # -- the stages of one chunk -------------------------------------------
    def _local_start(self, k, grad, pl):
        """Issue chunk k's local reduce (gather to the leader)."""
        c0, c1 = self.chunks[k]
        m, j = c1 - c0, k & 1
        if not self.local_quantize:
            outs = [t[:m] for t in self._recv[j]] if self.leader else None
            return self.local.gather(outs, grad[c0:c1].contiguous(), 0)
        p = pl.shifted(c0)
        bits, B = p.bits, p.block
        codes, scales = self._lc[j][:code_bytes(0, m, bits, B)], self._ls[j][:scale_count(0, m, B)]
        self.codec.quantize_pack(grad[c0:c1], p, None if self.err_local is None else self.err_local[c0:c1],
                                 codes, scales)
        oc = [t[:codes.numel()] for t in self._glc[j]] if self.leader else None
        os_ = [t[:2 * scales.numel()] for t in self._gls[j]] if self.leader else None
        return (self.local.gather(oc, codes, 0), self.local.gather(os_, scales.view(self.torch.uint8), 0))

    def _local_finish(self, k, handle):
        """The leader's local sum of chunk k (fp32, in self._r[k & 1])."""
        c0, c1 = self.chunks[k]
        m, j = c1 - c0, k & 1
        r = self._r[j][:m]
        if not self.local_quantize:
            _wait(handle)
            if self.leader:
                self.codec.sum_ranks([t[:m] for t in self._recv[j]], out=r)
            return r
        _wait(handle[0])
        _wait(handle[1])
        if self.leader:
            pl = self.p_local
            nc, ns = code_bytes(0, m, pl.bits, pl.block), scale_count(0, m, pl.block)
            self.codec.unpack_dequant_reduce_requant(
                [t[:nc] for t in self._glc[j]], [t[:2 * ns].view(self.torch.int16) for t in self._gls[j]], m,
                pl, sum_out=r)
        return r

    def _inter_and_broadcast(self, k, r, p1, p2, out, mul):
        """The leaders' low-bit all-reduce of chunk k, then its local broadcast."""
        c0, c1 = self.chunks[k]
        m, j = c1 - c0, k & 1
        if not self.local_quantize:
            if self.leader:
                self.ar.finish_bucket(k, self.ar.reduce_bucket(k, self.ar.send_bucket(k, r, p1), p2), p2,
                                      out[c0:c1], mul)
            return self.local.broadcast(out[c0:c1], 0)
        codes = self._bcodes[j][:code_bytes(0, m, self.p2.bits, self.p2.block)]
        scales = self._bscales[j][:scale_count(0, m, self.p2.block)]
        if self.leader:
            gc, gs = self.ar.gathered(k, self.ar.reduce_bucket(k, self.ar.send_bucket(k, r, p1), p2))
            codes.copy_(gc)
            scales.copy_(gs)
        return (self.local.broadcast(codes, 0), self.local.broadcast(scales.view(self.torch.uint8), 0))

    def _broadcast_finish(self, k, handle, p2, out, mul):
        c0, c1 = self.chunks[k]
        m, j = c1 - c0, k & 1
        if not self.local_quantize:
            _wait(handle)
            return
        _wait(handle[0])
        _wait(handle[1])
        codes = self._bcodes[j][:code_bytes(0, m, self.p2.bits, self.p2.block)]
        scales = self._bscales[j][:scale_count(0, m, self.p2.block)]
        self.codec.unpack_dequant(codes, scales, m, p2, mul, out[c0:c1])

    def __call__(self, grad, out, mul: float = 1.0):
        """All-reduce grad (this rank's n-element gradient) into out (fp32 or
        bf16): out = fl(fl(s*q) * mul) of the requantised SUM over all ranks."""
        if grad.numel() != self.n or grad.dtype != self.dtype or out.numel() != self.n:
            raise ValueError("gradient or output size / dtype differs from the one planned")
        base = self.step * self.n
        self.step += 1
        pl = (dataclasses.replace(self.p_local, index_offset=self.p_local.index_offset + base)
              if self.local_quantize else None)
        p1 = p2 = None
        if self.leader:
            p1, p2 = self.ar.begin_step()
        else:
            p2 = dataclasses.replace(self.p2, index_offset=self.p2.index_offset + base)
        K = len(self.chunks)
        if K == 0:
            return out
        pending_local = self._local_start(0, grad, pl)                        # warmup
        pending_bcast = None
        for k in range(K):                                                     # steady state
            nxt = self._local_start(k + 1, grad, pl) if k + 1 < K else None
            r = self._local_finish(k, pending_local)
            if pending_bcast is not None:
                self._broadcast_finish(k - 1, pending_bcast, p2, out, mul)
            pending_bcast = self._inter_and_broadcast(k, r, p1, p2, out, mul)
            pending_local = nxt
        self._broadcast_finish(K - 1, pending_bcast, p2, out, mul)            # cooldown
        return out


def _wait(handle):
    if handle is not None:
        handle.wait()
