"""GB300-native low-bit gradient codec: Python binding of libbitscom.so.

Argument marshalling only -- every step of the path runs in the CUDA kernels
behind the C ABI of ``include/bitscom.h``; PyTorch supplies device memory and
streams.  There is no CPU fallback: if the compiled library is missing or a
tensor is not on a CUDA device, the call raises.

The names follow the C ABI:
  quantize_pack                  encoder (absmax/mean + fp16 scale + quantise +
                                 pack + first-stage error feedback)
  unpack_dequant_reduce_requant  decoder of one chunk between the all-to-all
                                 and the all-gather (rank-ordered fp32 sum,
                                 stage-2 error feedback, requantise + repack)
  unpack_dequant                 all-gather-side decode into fp32 / bf16
  qwd_encode, qwd_apply          weight-difference quantisation (sharded
                                 weight all-gather)
  roundtrip                      quantise then dequantise
  sum_ranks                      rank-ordered fp32 sum (full-precision local reduce)
  Scheduler                      fusion buckets on CUDA streams
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libbitscom.so")

F32, BF16 = 0, 1
RTN, SR = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "pointer not aligned", 3: "unsupported combination",
          4: "CUDA error", 5: "timed out"}


class BitscomError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        msg = f"{what}: {STATUS.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class _QParams(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("block", ctypes.c_int32),
                ("rounding", ctypes.c_int32), ("philox_stream", ctypes.c_uint32),
                ("seed", ctypes.c_uint64), ("index_offset", ctypes.c_uint64),
                ("hadamard", ctypes.c_int32), ("reserved", ctypes.c_int32)]


@dataclass
class QParams:
    """One quantisation stage: bits in {1,2,4,8,12,16}, block a power of two in
    [8, 4096], rounding RTN or SR, Philox seed / stream word, the global
    element index of the call's first element, and the Walsh-Hadamard
    transform block (0 = none)."""
    bits: int
    block: int
    rounding: int = RTN
    seed: int = 0
    index_offset: int = 0
    philox_stream: int = 0
    hadamard: int = 0

    def c(self) -> _QParams:
        return _QParams(self.bits, self.block, self.rounding, self.philox_stream,
                        self.seed, self.index_offset, self.hadamard, 0)

    def shifted(self, offset: int) -> "QParams":
        return QParams(self.bits, self.block, self.rounding, self.seed,
                       self.index_offset + offset, self.philox_stream, self.hadamard)


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded libbitscom.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with "
                                  "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            P = ctypes.POINTER(_QParams)
            st = ctypes.c_int
            L.bitscom_num_blocks.restype = i64
            L.bitscom_num_blocks.argtypes = [i64, i32]
            L.bitscom_packed_bytes.restype = i64
            L.bitscom_packed_bytes.argtypes = [i64, i32, i32]
            L.bitscom_status_string.restype = ctypes.c_char_p
            L.bitscom_status_string.argtypes = [st]
            L.bitscom_last_cuda_error.restype = ctypes.c_char_p
            L.bitscom_last_cuda_error.argtypes = []
            L.bitscom_quantize_pack.restype = st
            L.bitscom_quantize_pack.argtypes = [vp, st, i64, vp, P, vp, vp, vp]
            L.bitscom_unpack_dequant_reduce_requant.restype = st
            L.bitscom_unpack_dequant_reduce_requant.argtypes = [vp, vp, i32, i64, P, vp, vp, P, vp, vp, vp]
            L.bitscom_roundtrip.restype = st
            L.bitscom_roundtrip.argtypes = [vp, st, i64, vp, P, vp, vp, vp, vp]
            L.bitscom_unpack_dequant.restype = st
            L.bitscom_unpack_dequant.argtypes = [vp, vp, i64, P, ctypes.c_float, st, vp, vp]
            L.bitscom_sum_ranks.restype = st
            L.bitscom_sum_ranks.argtypes = [vp, st, i32, i64, vp, vp]
            L.bitscom_qwd_encode.restype = st
            L.bitscom_qwd_encode.argtypes = [vp, st, i64, vp, P, vp, vp, vp]
            L.bitscom_qwd_apply.restype = st
            L.bitscom_qwd_apply.argtypes = [vp, vp, i64, P, vp, vp, st, vp]
            L.bitscom_roundtrip_noalloc.restype = st
            L.bitscom_roundtrip_noalloc.argtypes = [vp, st, i64, vp, P, vp, vp]
            L.bitscom_roundtrip_noalloc_max_elements.restype = i64
            L.bitscom_roundtrip_noalloc_max_elements.argtypes = [i32, i32]
            L.bitscom_sched_create.restype = st
            L.bitscom_sched_create.argtypes = [i32, i64, ctypes.POINTER(vp)]
            L.bitscom_sched_destroy.restype = st
            L.bitscom_sched_destroy.argtypes = [vp]
            L.bitscom_sched_plan.restype = i64
            L.bitscom_sched_plan.argtypes = [i64, i32, i32, i64, vp, i64]
            L.bitscom_sched_quantize_pack.restype = st
            L.bitscom_sched_quantize_pack.argtypes = [vp, vp, st, i64, vp, P, vp, vp, vp]
            L.bitscom_sched_allreduce.restype = st
            L.bitscom_sched_allreduce.argtypes = [vp, i32, vp, st, i64, vp, P, vp, vp, P, vp, vp, vp, vp, vp]
            L.bitscom_sched_wait.restype = st
            L.bitscom_sched_wait.argtypes = [vp, vp, dbl]
            _lib = L
    return _lib


def _check(status: int, what: str):
    if status != 0:
        detail = lib().bitscom_last_cuda_error().decode() if status == 4 else ""
        raise BitscomError(status, what, detail)


def num_blocks(n: int, block: int) -> int:
    return (n + block - 1) // block


def packed_bytes(n: int, bits: int, block: int) -> int:
    return num_blocks(n, block) * block * bits // 8


def plan_buckets(n: int, elem_bytes: int, block: int, bucket_bytes: int):
    """Bucket boundaries [starts[k], starts[k+1]) of the scheduler (host only)."""
    L = lib()
    count = L.bitscom_sched_plan(n, elem_bytes, block, bucket_bytes, None, 0)
    if count < 0:
        raise ValueError("bad bucket plan arguments")
    starts = (ctypes.c_int64 * (count + 1))()
    L.bitscom_sched_plan(n, elem_bytes, block, bucket_bytes, starts, count)
    return list(starts)


# ---- tensor helpers (torch is imported lazily: plumbing only) -------------

def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dev_ptr(t, name: str) -> int:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(x) -> int:
    torch = _torch()
    if x.dtype == torch.float32:
        return F32
    if x.dtype == torch.bfloat16:
        return BF16
    raise TypeError("gradients must be float32 or bfloat16")


def alloc_codes(n: int, p: QParams, device="cuda"):
    """(codes uint8[packed_bytes], scales int16[num_blocks]) device buffers."""
    torch = _torch()
    return (torch.empty(packed_bytes(n, p.bits, p.block), dtype=torch.uint8, device=device),
            torch.empty(num_blocks(n, p.block), dtype=torch.int16, device=device))


def quantize_pack(x, p: QParams, err=None, codes=None, scales=None, stream=None):
    """Encoder.  x: fp32/bf16 CUDA tensor; err: fp32 error buffer updated in
    place (None = no error feedback).  Returns (codes, scales)."""
    n = x.numel()
    if codes is None or scales is None:
        codes, scales = alloc_codes(n, p, x.device)
    _check(lib().bitscom_quantize_pack(_dev_ptr(x, "x"), _dtype_code(x), n, _dev_ptr(err, "err"),
                                       ctypes.byref(p.c()), _dev_ptr(codes, "codes"),
                                       _dev_ptr(scales, "scales"), _stream(stream)),
           "bitscom_quantize_pack")
    return codes, scales


def unpack_dequant_reduce_requant(codes_in: Sequence, scales_in: Sequence, n: int, p_in: QParams,
                                  sum_out=None, err2=None, p_out: Optional[QParams] = None,
                                  codes_out=None, scales_out=None, stream=None):
    """Decoder over W = len(codes_in) ranks' codes of one chunk of n elements.
    sum_out: fp32 tensor, or True to allocate one, or None.  With p_out the
    rank sum (+ err2) is requantised into (codes_out, scales_out), allocated
    when None.  Returns (sum_out, codes_out, scales_out)."""
    torch = _torch()
    W = len(codes_in)
    dev = codes_in[0].device
    if sum_out is True:
        sum_out = torch.empty(n, dtype=torch.float32, device=dev)
    if p_out is not None and (codes_out is None or scales_out is None):
        codes_out, scales_out = alloc_codes(n, p_out, dev)
    cp = (ctypes.c_void_p * W)(*[_dev_ptr(c, "codes_in") for c in codes_in])
    sp = (ctypes.c_void_p * W)(*[_dev_ptr(s, "scales_in") for s in scales_in])
    _check(lib().bitscom_unpack_dequant_reduce_requant(
        ctypes.cast(cp, ctypes.c_void_p), ctypes.cast(sp, ctypes.c_void_p), W, n,
        ctypes.byref(p_in.c()), _dev_ptr(sum_out, "sum_out"), _dev_ptr(err2, "err2"),
        ctypes.byref(p_out.c()) if p_out is not None else None,
        _dev_ptr(codes_out, "codes_out") if p_out is not None else None,
        _dev_ptr(scales_out, "scales_out") if p_out is not None else None, _stream(stream)),
        "bitscom_unpack_dequant_reduce_requant")
    return sum_out, codes_out, scales_out


def unpack_dequant(codes, scales, n: int, p: QParams, mul: float = 1.0, out=None, out_dtype=None,
                   stream=None):
    """All-gather-side decode: out = fl(fl(s*q) * mul) as fp32 or bf16 (out's
    dtype, or out_dtype when out is None; fp32 by default)."""
    torch = _torch()
    if out is None:
        out = torch.empty(n, dtype=out_dtype or torch.float32, device=codes.device)
    _check(lib().bitscom_unpack_dequant(_dev_ptr(codes, "codes"), _dev_ptr(scales, "scales"), n,
                                        ctypes.byref(p.c()), ctypes.c_float(mul), _dtype_code(out),
                                        _dev_ptr(out, "out"), _stream(stream)), "bitscom_unpack_dequant")
    return out


def sum_ranks(xs: Sequence, out=None, stream=None):
    """Rank-ordered fp32 sum of W = len(xs) fp32 or bf16 tensors of one size:
    out = fl(...fl(x_0 + x_1)... + x_{W-1}).  Returns out (allocated when None)."""
    torch = _torch()
    W = len(xs)
    n = xs[0].numel()
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=xs[0].device)
    if any(x.numel() != n or x.dtype != xs[0].dtype for x in xs) or out.numel() != n:
        raise ValueError("sum_ranks: every input and the output need the same size, inputs one dtype")
    xp = (ctypes.c_void_p * W)(*[_dev_ptr(x, "x") for x in xs])
    _check(lib().bitscom_sum_ranks(ctypes.cast(xp, ctypes.c_void_p), _dtype_code(xs[0]), W, n,
                                   _dev_ptr(out, "out"), _stream(stream)), "bitscom_sum_ranks")
    return out


def qwd_encode(w, ref, p: QParams, codes=None, scales=None, stream=None):
    """Weight-difference encoder: codes of w - ref; ref (fp32) advances in place."""
    n = w.numel()
    if codes is None or scales is None:
        codes, scales = alloc_codes(n, p, w.device)
    _check(lib().bitscom_qwd_encode(_dev_ptr(w, "w"), _dtype_code(w), n, _dev_ptr(ref, "ref"),
                                    ctypes.byref(p.c()), _dev_ptr(codes, "codes"), _dev_ptr(scales, "scales"),
                                    _stream(stream)), "bitscom_qwd_encode")
    return codes, scales


def qwd_apply(codes, scales, n: int, p: QParams, ref, w_out=None, stream=None):
    """Receiver update ref += s*q in place; w_out (fp32 or bf16) gets the weights."""
    _check(lib().bitscom_qwd_apply(_dev_ptr(codes, "codes"), _dev_ptr(scales, "scales"), n,
                                   ctypes.byref(p.c()), _dev_ptr(ref, "ref"), _dev_ptr(w_out, "w_out"),
                                   _dtype_code(w_out) if w_out is not None else F32, _stream(stream)),
           "bitscom_qwd_apply")
    return w_out


def roundtrip(x, p: QParams, err=None, codes_tmp=None, scales_tmp=None, deq_out=None, stream=None):
    """Quantise then dequantise x (fp32 result).  Returns deq_out."""
    torch = _torch()
    n = x.numel()
    if codes_tmp is None or scales_tmp is None:
        codes_tmp, scales_tmp = alloc_codes(n, p, x.device)
    if deq_out is None:
        deq_out = torch.empty(n, dtype=torch.float32, device=x.device)
    _check(lib().bitscom_roundtrip(_dev_ptr(x, "x"), _dtype_code(x), n, _dev_ptr(err, "err"),
                                   ctypes.byref(p.c()), _dev_ptr(codes_tmp, "codes_tmp"),
                                   _dev_ptr(scales_tmp, "scales_tmp"), _dev_ptr(deq_out, "deq_out"),
                                   _stream(stream)), "bitscom_roundtrip")
    return deq_out


def roundtrip_noalloc_max_elements(bits: int, block: int) -> int:
    return lib().bitscom_roundtrip_noalloc_max_elements(bits, block)


def roundtrip_noalloc(x, p: QParams, err=None, deq_out=None, stream=None):
    """roundtrip() for callers that cannot allocate device memory: the codes and
    scales go to the library's fixed device scratch (see include/bitscom.h for
    its capacity and sharing rules).  deq_out must be given by such callers;
    when it is None this wrapper allocates it for convenience."""
    torch = _torch()
    n = x.numel()
    cap = roundtrip_noalloc_max_elements(p.bits, p.block)
    if n > cap:
        raise ValueError(f"n = {n} exceeds the static scratch capacity ({cap} elements for "
                         f"{p.bits}-bit, block {p.block})")
    if deq_out is None:
        deq_out = torch.empty(n, dtype=torch.float32, device=x.device)
    _check(lib().bitscom_roundtrip_noalloc(_dev_ptr(x, "x"), _dtype_code(x), n, _dev_ptr(err, "err"),
                                           ctypes.byref(p.c()), _dev_ptr(deq_out, "deq_out"),
                                           _stream(stream)), "bitscom_roundtrip_noalloc")
    return deq_out


class Scheduler:
    """Fusion-bucket scheduler on its own CUDA streams (see bitscom_sched_*)."""

    def __init__(self, n_streams: int = 2, bucket_bytes: int = 25 * 1024 * 1024):
        h = ctypes.c_void_p()
        _check(lib().bitscom_sched_create(n_streams, bucket_bytes, ctypes.byref(h)), "bitscom_sched_create")
        self._h = h
        self.n_streams = n_streams
        self.bucket_bytes = bucket_bytes

    def close(self):
        if self._h:
            lib().bitscom_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def quantize_pack(self, x, p: QParams, err=None, codes=None, scales=None, stream=None):
        n = x.numel()
        if codes is None or scales is None:
            codes, scales = alloc_codes(n, p, x.device)
        _check(lib().bitscom_sched_quantize_pack(self._h, _dev_ptr(x, "x"), _dtype_code(x), n,
                                                 _dev_ptr(err, "err"), ctypes.byref(p.c()),
                                                 _dev_ptr(codes, "codes"), _dev_ptr(scales, "scales"),
                                                 _stream(stream)), "bitscom_sched_quantize_pack")
        return codes, scales

    def allreduce(self, xs: Sequence, p1: Sequence[QParams], codes: Sequence, scales: Sequence,
                  errs: Optional[Sequence] = None, p2: Optional[QParams] = None, err2=None,
                  codes_out=None, scales_out=None, sum_out=None, stream=None):
        """Simulated W-rank low-bit all-reduce (W = len(xs)) on one GPU."""
        W = len(xs)
        n = xs[0].numel()
        dt = _dtype_code(xs[0])
        xp = (ctypes.c_void_p * W)(*[_dev_ptr(x, "x") for x in xs])
        ep = None
        if errs is not None:
            ep = ctypes.cast((ctypes.c_void_p * W)(*[_dev_ptr(e, "err") for e in errs]), ctypes.c_void_p)
        qp = (_QParams * W)(*[q.c() for q in p1])
        cp = (ctypes.c_void_p * W)(*[_dev_ptr(c, "codes") for c in codes])
        sp = (ctypes.c_void_p * W)(*[_dev_ptr(s, "scales") for s in scales])
        _check(lib().bitscom_sched_allreduce(
            self._h, W, ctypes.cast(xp, ctypes.c_void_p), dt, n, ep,
            ctypes.cast(qp, ctypes.POINTER(_QParams)), ctypes.cast(cp, ctypes.c_void_p),
            ctypes.cast(sp, ctypes.c_void_p), ctypes.byref(p2.c()) if p2 is not None else None,
            _dev_ptr(err2, "err2"), _dev_ptr(codes_out, "codes_out"), _dev_ptr(scales_out, "scales_out"),
            _dev_ptr(sum_out, "sum_out"), _stream(stream)), "bitscom_sched_allreduce")

    def wait(self, stream=None, timeout_s: float = 60.0):
        _check(lib().bitscom_sched_wait(self._h, _stream(stream), timeout_s), "bitscom_sched_wait")
