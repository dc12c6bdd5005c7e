"""Low-bit all-reduce across real ranks: one process (and one GPU) per rank.

The method (bitscom README, "Implemented Features": the low-bit all-reduce
pipeline all-to-all -> local reduce -> all-gather; DeAR README, opening
paragraph: an all-reduce is a reduce-scatter followed by an all-gather), per
fusion bucket of the flat gradient:

  1. encoder    every rank quantises and packs its own bucket, with first-stage
                error feedback (bitscom_quantize_pack);
  2. all-to-all rank c receives chunk c of every rank's codes and fp16 scales;
  3. decoder    rank c unpacks, dequantises and sums the W ranks' chunk in rank
                order, adds its shard of the stage-2 error, requantises and
                repacks (bitscom_unpack_dequant_reduce_requant);
  4. all-gather every rank receives every chunk's requantised codes and scales;
  5. decode     every rank turns them into the summed (or averaged) gradient
                (bitscom_unpack_dequant).

Buckets and chunks are those of the single-GPU simulation
(bitscom_sched_allreduce): buckets of bucket_bytes of the input dtype rounded
down to whole units of max(B1, B2, 128) elements, chunk c of a bucket = units
[c*ceil(units/W), (c+1)*ceil(units/W)) with U = max(B1, B2); every Philox
index is the element's global index.  So W processes produce, bit for bit,
the codes, scales and error buffers of the simulated W-rank all-reduce.

Every codec step runs in libbitscom's kernels; this module only plans the
partition, slices buffers and issues torch.distributed collectives on byte
tensors (NCCL on device memory; gloo on host memory, or device memory staged
through the host).  Stage-2 errors are sharded: each rank keeps only the
elements of the chunks it owns.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

from . import QParams, num_blocks


def bucket_elems(bucket_bytes: int, elem_bytes: int, unit: int) -> int:
    """Elements per bucket: bucket_bytes of the input dtype rounded down to a
    whole number of units (at least one unit); 0 = the call is one bucket."""
    if bucket_bytes <= 0:
        return 0
    per = bucket_bytes // elem_bytes // unit * unit
    return per if per >= unit else unit


@dataclasses.dataclass(frozen=True)
class Bucket:
    b0: int                                  # first element of the bucket
    n: int                                   # elements in the bucket
    chunks: Tuple[Tuple[int, int], ...]      # chunk c: global elements [lo, hi) (lo == hi: empty)


def plan(n: int, elem_bytes: int, block1: int, block2: int, W: int, bucket_bytes: int) -> List[Bucket]:
    """Buckets of n elements and, inside each, the W chunks (rank c owns chunk c)."""
    if n < 0 or W < 1:
        raise ValueError("n must be >= 0 and W >= 1")
    U = max(block1, block2)
    per = bucket_elems(bucket_bytes, elem_bytes, max(U, 128))
    out = []
    starts = [0] if per == 0 else list(range(0, n, per))
    for b0 in starts:
        nbk = n if per == 0 else min(per, n - b0)
        units = (nbk + U - 1) // U
        cu = (units + W - 1) // W
        chunks = []
        for c in range(W):
            u0 = c * cu
            if u0 >= units:
                chunks.append((b0 + nbk, b0 + nbk))
            else:
                chunks.append((b0 + u0 * U, b0 + min((u0 + cu) * U, nbk)))
        out.append(Bucket(b0, nbk, tuple(chunks)))
    return out


def code_bytes(lo: int, hi: int, bits: int, block: int) -> int:
    """Bytes of packed codes of elements [lo, hi), lo on a block boundary."""
    if hi <= lo:
        return 0
    return (num_blocks(hi, block) * block - lo) * bits // 8


def scale_count(lo: int, hi: int, block: int) -> int:
    return 0 if hi <= lo else num_blocks(hi, block) - lo // block


class Exchange:
    """The two collectives of the all-reduce on uint8 tensors of one process
    group.  host_staging: the tensors live on a GPU but the group's backend
    works on host memory (gloo): each collective copies its input to the host
    and its output back (synchronously)."""

    def __init__(self, group=None, host_staging: bool = False):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.host_staging = host_staging
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_to_all(self, out, inp, out_splits, in_splits):
        """out = concatenation over ranks w of what rank w sent here."""
        if self.host_staging:
            h_out = out.cpu()
            self.dist.all_to_all_single(h_out, inp.cpu(), list(out_splits), list(in_splits), group=self.group)
            out.copy_(h_out)
            return None
        return self.dist.all_to_all_single(out, inp, list(out_splits), list(in_splits), group=self.group,
                                           async_op=True)

    def all_gather(self, out, inp):
        """out = concatenation over ranks of inp (equal sizes)."""
        if self.host_staging:
            h_out = out.cpu()
            self.dist.all_gather_into_tensor(h_out, inp.cpu(), group=self.group)
            out.copy_(h_out)
            return None
        return self.dist.all_gather_into_tensor(out, inp, group=self.group, async_op=True)

    def _global(self, group_rank: int) -> int:
        return group_rank if self.group is None else self.dist.get_global_rank(self.group, group_rank)

    def gather(self, outs, inp, root: int = 0):
        """The group's root receives every rank's inp into outs[rank] (a list of
        equal-size tensors on the root, None elsewhere)."""
        if self.host_staging:
            h_outs = [o.cpu() for o in outs] if outs is not None else None
            self.dist.gather(inp.cpu(), h_outs, dst=self._global(root), group=self.group)
            if outs is not None:
                for o, h in zip(outs, h_outs):
                    o.copy_(h)
            return None
        return self.dist.gather(inp, outs, dst=self._global(root), group=self.group, async_op=True)

    def broadcast(self, t, root: int = 0):
        """t on every rank becomes the root's t."""
        if self.host_staging:
            h = t.cpu()
            self.dist.broadcast(h, src=self._global(root), group=self.group)
            t.copy_(h)
            return None
        return self.dist.broadcast(t, src=self._global(root), group=self.group, async_op=True)


def _wait(handle):
    if handle is not None:
        handle.wait()


class LowBitAllReduce:
    """One rank's low-bit all-reduce of a flat gradient of n elements.

    p1: this rank's stage-1 parameters (bits, block, rounding, seed; every rank
        must use the same bits and block, seeds differ per rank).
    p2: stage-2 (requantisation) parameters, shared by all ranks.
    error_feedback / stage2_error_feedback: keep the first-stage error buffer
        (n elements) and this rank's shard of the stage-2 error.
    bucket_bytes: fusion-bucket size in bytes of the input dtype (0: one bucket).
    codec: the object whose quantize_pack / unpack_dequant_reduce_requant /
        unpack_dequant run the codec steps; the default is libbitscom through
        this package's binding (device tensors only).
    exchange: an Exchange over the ranks' process group (default: the default
        group, collectives on the tensors' own device).

    Every call advances the Philox window by n elements (index offsets step*n
    on top of p1/p2's), so stochastic rounding draws fresh words each step.
    """

    def __init__(self, n: int, dtype, p1: QParams, p2: QParams, device=None,
                 error_feedback: bool = True, stage2_error_feedback: bool = True,
                 bucket_bytes: int = 25 * 1024 * 1024, codec=None, exchange: Optional[Exchange] = None):
        import sys

        import torch
        if codec is None:
            codec = sys.modules[__package__]      # the libbitscom binding of this package
        self.torch = torch
        self.codec = codec
        self.ex = exchange or Exchange()
        self.W, self.rank = self.ex.world, self.ex.rank
        self.n, self.dtype, self.p1, self.p2 = n, dtype, p1, p2
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        esz = torch.empty(0, dtype=dtype).element_size()
        if esz not in (2, 4):
            raise TypeError("gradients must be float32 or bfloat16")
        if p1.hadamard != p2.hadamard:
            raise ValueError("both stages of one all-reduce use the same Hadamard block (or none)")
        self.buckets = plan(n, esz, p1.block, p2.block, self.W, bucket_bytes)
        self.step = 0
        b1, B1, b2, B2 = p1.bits, p1.block, p2.bits, p2.block
        # this rank's stage-2 error shard: its chunk of every bucket, in bucket order
        self._e2_at = []
        self.shard = 0
        for bk in self.buckets:
            lo, hi = bk.chunks[self.rank]
            self._e2_at.append(self.shard)
            self.shard += hi - lo
        dev, u8 = self.device, torch.uint8
        f32 = torch.float32
        self.err = torch.zeros(n, dtype=f32, device=dev) if error_feedback else None
        self.err2 = torch.zeros(max(self.shard, 1), dtype=f32, device=dev) if stage2_error_feedback else None
        self.codes = torch.empty(code_bytes(0, n, b1, B1), dtype=u8, device=dev)
        self.scales = torch.empty(scale_count(0, n, B1), dtype=torch.int16, device=dev)
        # per bucket: receive buffer of W pieces of this rank's chunk, and the
        # all-gather's send / gather buffers (every piece padded to the largest chunk)
        self._bufs = []
        for bk in self.buckets:
            lo, hi = bk.chunks[self.rank]
            rc, rs = code_bytes(lo, hi, b1, B1), 2 * scale_count(lo, hi, B1)
            gc = max(code_bytes(l, h, b2, B2) for l, h in bk.chunks)
            gs = max(2 * scale_count(l, h, B2) for l, h in bk.chunks)
            self._bufs.append({
                "rc": torch.empty(self.W * rc, dtype=u8, device=dev),
                "rs": torch.empty(self.W * rs, dtype=u8, device=dev),
                "sc": torch.zeros(gc, dtype=u8, device=dev), "ss": torch.zeros(gs, dtype=u8, device=dev),
                "gc": torch.empty(self.W * gc, dtype=u8, device=dev),
                "gs": torch.empty(self.W * gs, dtype=u8, device=dev)})

    # -- the five steps ----------------------------------------------------
    def __call__(self, grad, out=None, mul: float = 1.0, out_codes=None, out_scales=None):
        """All-reduce grad (this rank's n-element gradient).  out: fp32 or bf16
        tensor receiving fl(fl(s*q) * mul) of the requantised SUM (mul = 1/W for
        the mean); None = no decode.  out_codes / out_scales: optional buffers
        (packed_bytes / num_blocks of p2 over n) receiving the gathered
        requantised codes and scales at their global positions.  Returns out.
        The three phases are also callable one by one (send, reduce, finish)."""
        self.finish(self.reduce(self.send(grad)), out, mul, out_codes, out_scales)
        return out

    def send(self, grad):
        """Steps 1 and 2: encode every bucket on the current stream; each
        bucket's all-to-all starts once it is encoded.  Returns the pending state."""
        if grad.numel() != self.n or grad.dtype != self.dtype:
            raise ValueError("gradient size or dtype differs from the one planned")
        p1, p2 = self.begin_step()
        a2a = [self.send_bucket(k, grad[bk.b0:bk.b0 + bk.n], p1) for k, bk in enumerate(self.buckets)]
        return {"p2": p2, "a2a": a2a}

    def reduce(self, state):
        """Steps 3 and 4: decode this rank's chunk of every bucket (rank-ordered
        sum, stage-2 error, requantisation); each chunk's all-gather starts once
        it is requantised."""
        ag = [self.reduce_bucket(k, h, state["p2"]) for k, h in enumerate(state["a2a"])]
        return {"p2": state["p2"], "ag": ag}

    def finish(self, state, out=None, mul: float = 1.0, out_codes=None, out_scales=None):
        """Step 5: every rank decodes the gathered codes of every bucket (and
        copies them to out_codes / out_scales when given)."""
        for k, (bk, h) in enumerate(zip(self.buckets, state["ag"])):
            self.finish_bucket(k, h, state["p2"], None if out is None else out[bk.b0:bk.b0 + bk.n], mul,
                               out_codes, out_scales)
        return out

    # -- one bucket at a time (the pipelined hierarchical all-reduce uses these) --
    def begin_step(self):
        """This step's stage parameters (Philox window step * n); advances the step."""
        base = self.step * self.n
        self.step += 1
        return (dataclasses.replace(self.p1, index_offset=self.p1.index_offset + base),
                dataclasses.replace(self.p2, index_offset=self.p2.index_offset + base))

    def send_bucket(self, k: int, grad_bucket, p1):
        """Encode bucket k (grad_bucket: its elements) and start its all-to-all."""
        torch = self.torch
        bk, buf = self.buckets[k], self._bufs[k]
        b1, B1 = self.p1.bits, self.p1.block
        c0, c1 = bk.b0 * b1 // 8, bk.b0 * b1 // 8 + code_bytes(bk.b0, bk.b0 + bk.n, b1, B1)
        s0, s1 = bk.b0 // B1, bk.b0 // B1 + scale_count(bk.b0, bk.b0 + bk.n, B1)
        self.codec.quantize_pack(grad_bucket, p1.shifted(bk.b0),
                                 None if self.err is None else self.err[bk.b0:bk.b0 + bk.n],
                                 self.codes[c0:c1], self.scales[s0:s1])
        lo, hi = bk.chunks[self.rank]
        in_c = [code_bytes(l, h, b1, B1) for l, h in bk.chunks]
        in_s = [2 * scale_count(l, h, B1) for l, h in bk.chunks]
        rc, rs = code_bytes(lo, hi, b1, B1), 2 * scale_count(lo, hi, B1)
        scales8 = self.scales.view(torch.uint8)
        return (self.ex.all_to_all(buf["rc"], self.codes[c0:c1], [rc] * self.W, in_c),
                self.ex.all_to_all(buf["rs"], scales8[2 * s0:2 * s1], [rs] * self.W, in_s))

    def reduce_bucket(self, k: int, a2a, p2):
        """Decode this rank's chunk of bucket k once its all-to-all is done;
        start the bucket's all-gather."""
        torch = self.torch
        bk, buf = self.buckets[k], self._bufs[k]
        b1, B1, b2, B2 = self.p1.bits, self.p1.block, self.p2.bits, self.p2.block
        _wait(a2a[0])
        _wait(a2a[1])
        lo, hi = bk.chunks[self.rank]
        nc = hi - lo
        if nc > 0:
            rc, rs = code_bytes(lo, hi, b1, B1), 2 * scale_count(lo, hi, B1)
            cin = [buf["rc"][w * rc:(w + 1) * rc] for w in range(self.W)]
            sin = [buf["rs"][w * rs:(w + 1) * rs].view(torch.int16) for w in range(self.W)]
            oc, os_ = code_bytes(lo, hi, b2, B2), scale_count(lo, hi, B2)
            e2_at = self._e2_at[k]
            self.codec.unpack_dequant_reduce_requant(
                cin, sin, nc, self.p1, sum_out=None,
                err2=None if self.err2 is None else self.err2[e2_at:e2_at + nc],
                p_out=p2.shifted(lo), codes_out=buf["sc"][:oc], scales_out=buf["ss"][:2 * os_].view(torch.int16))
        return self.ex.all_gather(buf["gc"], buf["sc"]), self.ex.all_gather(buf["gs"], buf["ss"])

    def gathered(self, k: int, ag):
        """Bucket k's requantised codes and scales once its all-gather is done.
        The gathered pieces are padded to the largest chunk; only the last
        non-empty chunk is shorter, so the bucket's codes are the prefix."""
        torch = self.torch
        bk, buf = self.buckets[k], self._bufs[k]
        b2, B2 = self.p2.bits, self.p2.block
        _wait(ag[0])
        _wait(ag[1])
        nbytes = code_bytes(bk.b0, bk.b0 + bk.n, b2, B2)
        nsc = scale_count(bk.b0, bk.b0 + bk.n, B2)
        return buf["gc"][:nbytes], buf["gs"][:2 * nsc].view(torch.int16)

    def finish_bucket(self, k: int, ag, p2, out_bucket=None, mul: float = 1.0, out_codes=None, out_scales=None):
        """Decode bucket k's gathered codes into out_bucket (its elements)."""
        bk = self.buckets[k]
        b2, B2 = self.p2.bits, self.p2.block
        gcodes, gscales = self.gathered(k, ag)
        if out_codes is not None:
            out_codes[bk.b0 * b2 // 8: bk.b0 * b2 // 8 + gcodes.numel()].copy_(gcodes)
        if out_scales is not None:
            out_scales[bk.b0 // B2: bk.b0 // B2 + gscales.numel()].copy_(gscales)
        if out_bucket is not None:
            self.codec.unpack_dequant(gcodes, gscales, bk.n, p2, mul, out_bucket)
        return out_bucket
