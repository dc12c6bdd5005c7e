"""Single-process simulation of the bucketed W-rank low-bit all-reduce with the
CPU oracle: what W real ranks must produce, bit for bit.

Per step t and bucket k (elements [b0, b0 + nk)), every rank w encodes its
bucket (Philox index offset t*n + b0, its own error buffer); chunk c's owner
decodes the W ranks' chunk c (stage-2 error e2[lo:hi], index offset
t*n + lo) into the requantised codes at the chunk's global position; the
all-gather-side decode multiplies fl(s*q) by mul.  Buckets and chunks come
from the package's host-side planner, whose rule is checked against the C
scheduler in tests/test_sharded_plan.py.
"""
import numpy as np

import oracle as O
from bit_gradient_communication_gb300 import sharded


def simulate(grads, n, bits, block, rounding, seeds, seed2, bucket_bytes, elem_bytes=4, mul=1.0, out_dtype=O.F32,
             bits2=None, block2=None, hadamard=0):
    """grads[t][w]: rank w's gradient of step t (fp32 array, or uint16 bf16 bits).
    Stage 1 codes bits/block, stage 2 bits2/block2 (default: the same), both
    rotated by the Walsh-Hadamard transform of `hadamard` elements when set.
    Returns per step (codes, scales, out) of stage 2 and the final (errs, e2)."""
    W = len(seeds)
    bits2 = bits if bits2 is None else bits2
    block2 = block if block2 is None else block2
    buckets = sharded.plan(n, elem_bytes, block, block2, W, bucket_bytes)
    errs = [np.zeros(n, np.float32) for _ in range(W)]
    e2 = np.zeros(n, np.float32)
    results = []
    for t, gw in enumerate(grads):
        codes = np.zeros(O.packed_bytes(n, bits2, block2), np.uint8)
        scales = np.zeros(O.num_blocks(n, block2), np.uint16)
        for bk in buckets:
            b0, nk = bk.b0, bk.n
            enc = []
            for w in range(W):
                p1 = O.params(bits, block, rounding, seed=seeds[w], index_offset=t * n + b0, hadamard=hadamard)
                enc.append(O.quantize_pack(np.ascontiguousarray(gw[w][b0:b0 + nk]), p1, errs[w][b0:b0 + nk]))
            for lo, hi in bk.chunks:
                if hi <= lo:
                    continue
                c0 = (lo - b0) * bits // 8
                c1 = sharded.code_bytes(lo - b0, hi - b0, bits, block) + c0
                s0 = (lo - b0) // block
                s1 = s0 + sharded.scale_count(lo - b0, hi - b0, block)
                p2 = O.params(bits2, block2, rounding, seed=seed2, index_offset=t * n + lo, philox_stream=1,
                              hadamard=hadamard)
                _, co, so = O.unpack_dequant_reduce_requant([c[c0:c1] for c, _ in enc], [s[s0:s1] for _, s in enc],
                                                            hi - lo, O.params(bits, block, hadamard=hadamard), False,
                                                            e2[lo:hi], p2)
                codes[lo * bits2 // 8: lo * bits2 // 8 + co.size] = co
                scales[lo // block2: lo // block2 + so.size] = so
        out = O.unpack_dequant(codes, scales, n, O.params(bits2, block2, rounding, seed=seed2, philox_stream=1,
                                                          hadamard=hadamard), mul, out_dtype)
        results.append((codes, scales, out))
    return results, errs, e2


def shard_of(e2, n, W, rank, block, bucket_bytes, elem_bytes=4, block2=None):
    """Rank `rank`'s stage-2 error shard: its chunks of every bucket, in order."""
    block2 = block if block2 is None else block2
    parts = [e2[bk.chunks[rank][0]:bk.chunks[rank][1]]
             for bk in sharded.plan(n, elem_bytes, block, block2, W, bucket_bytes)]
    return np.concatenate(parts) if parts else np.zeros(0, np.float32)
