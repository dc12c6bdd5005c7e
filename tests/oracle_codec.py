"""The codec interface of the binding (quantize_pack, unpack_dequant_reduce_requant,
unpack_dequant) on host torch tensors, computed by the CPU oracle.

Test infrastructure: it lets the multi-rank orchestration code run on gloo
ranks without a GPU.  The library itself never uses it (its default codec is
libbitscom, which rejects host tensors).
"""
import numpy as np
import torch

import oracle as O


def params(p):
    """oracle parameters of a binding QParams."""
    return O.params(p.bits, p.block, p.rounding, seed=p.seed, index_offset=p.index_offset,
                    philox_stream=p.philox_stream, hadamard=p.hadamard)


def _np(x):
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    if x.dtype == torch.int16:
        return x.numpy().view(np.uint16)
    return x.numpy()


class OracleCodec:
    def quantize_pack(self, x, p, err=None, codes=None, scales=None, stream=None):
        c, s = O.quantize_pack(np.ascontiguousarray(_np(x)), params(p), None if err is None else err.numpy())
        codes.numpy()[:] = c
        _np(scales)[:] = s
        return codes, scales

    def unpack_dequant_reduce_requant(self, codes_in, scales_in, n, p_in, sum_out=None, err2=None, p_out=None,
                                      codes_out=None, scales_out=None, stream=None):
        sm, co, so = O.unpack_dequant_reduce_requant(
            [c.numpy() for c in codes_in], [_np(s) for s in scales_in], n, params(p_in), sum_out is not None,
            None if err2 is None else err2.numpy(), None if p_out is None else params(p_out))
        if sum_out is not None:
            sum_out.numpy()[:] = sm
        if p_out is not None:
            codes_out.numpy()[:] = co
            _np(scales_out)[:] = so
        return sum_out, codes_out, scales_out

    def unpack_dequant(self, codes, scales, n, p, mul=1.0, out=None, out_dtype=None, stream=None):
        dt = O.F32 if out.dtype == torch.float32 else O.BF16
        _np(out)[:] = O.unpack_dequant(codes.numpy(), _np(scales), n, params(p), mul, dt)
        return out

    def sum_ranks(self, xs, out=None, stream=None):
        out.numpy()[:] = O.sum_ranks([np.ascontiguousarray(_np(x)) for x in xs])
        return out
