"""CPU oracle of the low-bit gradient codec -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library's product path never does,
and it shares no code with the CUDA path: the oracle is plain single-threaded
C++ (``bitscom_oracle.cpp``) loaded through ctypes, working on numpy arrays.

Parity status of each function (details in the tests):
  f32_to_f16, f16_to_f32, bf16_to_f32   pinned (exhaustive vs numpy casts)
  philox4x32_10, random_word(s)          pinned (cuRAND host generator)
  quantize_pack                          pinned (hand-worked blocks, bounds,
                                         unbiasedness, numpy packbits)
  unpack_dequant_reduce_requant          pinned (W=1 == dequant, hand sums,
                                         telescoping error-feedback bound)
  unpack_dequant, f32_to_bf16            pinned (W=1 decoder sums, torch bf16 cast)
  fwht (Hadamard smoothing)              pinned (scipy Sylvester matrix, involution)
  sum_ranks (full-precision local reduce) pinned (hand-worked order and -0 cases,
                                         exact sums of small integers)
  qwd_encode, qwd_apply                  pinned (hand block, bound, telescoping)
  tail blocks (n mod B != 0), 1-bit SR   pinned to their readings (hand-worked
                                         tails, tail == zero-padded block,
                                         1-bit SR == RTN); the readings
                                         themselves have no page support
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bitscom_oracle.cpp")
_HDR = os.path.join(_HERE, "bitscom_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_FLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
          "-fexcess-precision=standard", "-fPIC", "-shared", "-Wall"]

_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
RTN, SR = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (IEEE-exact flags); returns the .so path.

    BITSCOM_ORACLE_LIB names a prebuilt library to load instead (the tests use
    it to check that deliberately broken copies of the oracle fail the pins)."""
    override = os.environ.get("BITSCOM_ORACLE_LIB")
    if override:
        return override
    stale = (not os.path.exists(_LIB) or
             os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["g++", *_FLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class Params(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("block", ctypes.c_int32),
                ("rounding", ctypes.c_int32), ("philox_stream", ctypes.c_uint32),
                ("seed", ctypes.c_uint64), ("index_offset", ctypes.c_uint64),
                ("hadamard", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def params(bits, block, rounding=RTN, seed=0, index_offset=0, philox_stream=0, hadamard=0) -> Params:
    return Params(bits, block, rounding, philox_stream, seed, index_offset, hadamard, 0)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i64, i32, u32, u64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_uint32, ctypes.c_uint64)
            P = ctypes.POINTER(Params)
            L.orc_f32_to_f16.restype = ctypes.c_uint16
            L.orc_f32_to_f16.argtypes = [ctypes.c_float]
            L.orc_f16_to_f32.restype = ctypes.c_float
            L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_f32.restype = ctypes.c_float
            L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f32_to_f16_many.argtypes = [vp, vp, i64]
            L.orc_philox4x32_10.argtypes = [vp, vp, vp]
            L.orc_random_word.restype = u32
            L.orc_random_word.argtypes = [u64, u32, u64]
            L.orc_random_words.restype = None
            L.orc_random_words.argtypes = [u64, u32, u64, ctypes.c_int64, ctypes.c_void_p]
            L.orc_quantize_pack.restype = ctypes.c_int
            L.orc_quantize_pack.argtypes = [vp, i32, i64, vp, P, vp, vp]
            L.orc_unpack_dequant_reduce_requant.restype = ctypes.c_int
            L.orc_unpack_dequant_reduce_requant.argtypes = [vp, vp, i32, i64, P, vp, vp, P, vp, vp]
            L.orc_roundtrip.restype = ctypes.c_int
            L.orc_roundtrip.argtypes = [vp, i32, i64, vp, P, vp, vp, vp]
            L.orc_unpack_dequant.restype = ctypes.c_int
            L.orc_unpack_dequant.argtypes = [vp, vp, i64, P, ctypes.c_float, i32, vp]
            L.orc_f32_to_bf16.restype = ctypes.c_uint16
            L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
            L.orc_qwd_encode.restype = ctypes.c_int
            L.orc_qwd_encode.argtypes = [vp, i32, i64, vp, P, vp, vp]
            L.orc_qwd_apply.restype = ctypes.c_int
            L.orc_qwd_apply.argtypes = [vp, vp, i64, P, vp, vp, i32]
            L.orc_sum_ranks.restype = ctypes.c_int
            L.orc_sum_ranks.argtypes = [vp, i32, i32, i64, vp]
            L.orc_fwht.restype = ctypes.c_int
            L.orc_fwht.argtypes = [vp, i64, i32]
            L.orc_num_blocks.restype = i64
            L.orc_num_blocks.argtypes = [i64, i32]
            L.orc_packed_bytes.restype = i64
            L.orc_packed_bytes.argtypes = [i64, i32, i32]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_blocks(n, block):
    return (n + block - 1) // block


def packed_bytes(n, bits, block):
    return num_blocks(n, block) * block * bits // 8


# ---- scalar helpers -------------------------------------------------------

def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_f16_many(_ptr(x), _ptr(out), x.size)
    return out


def f16_to_f32(h: int) -> float:
    return lib().orc_f16_to_f32(int(h))


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def random_word(seed, stream, i):
    return lib().orc_random_word(seed, stream, i)


def random_words(seed, stream, i0, n):
    out = np.zeros(n, dtype=np.uint32)
    lib().orc_random_words(seed, stream, i0, n, _ptr(out))
    return out


# ---- codec ----------------------------------------------------------------

def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.uint16:   # bf16 bit patterns
        return BF16
    raise TypeError("x must be float32 or uint16 (bf16 bits)")


def quantize_pack(x: np.ndarray, p: Params, err: np.ndarray | None = None):
    """Encoder.  Returns (codes uint8[packed_bytes], scales uint16[nb]);
    ``err`` (float32) is updated in place when given."""
    x = np.ascontiguousarray(x)
    n = x.size
    codes = np.zeros(packed_bytes(n, p.bits, p.block), dtype=np.uint8)
    scales = np.zeros(num_blocks(n, p.block), dtype=np.uint16)
    if err is not None:
        assert err.dtype == np.float32 and err.flags.c_contiguous and err.size == n
    rc = lib().orc_quantize_pack(_ptr(x), _dtype_code(x), n, _ptr(err), ctypes.byref(p),
                                 _ptr(codes), _ptr(scales))
    if rc:
        raise ValueError("oracle rejected the arguments")
    return codes, scales


def unpack_dequant_reduce_requant(codes_in, scales_in, n: int, p_in: Params,
                                  want_sum: bool = True, err2: np.ndarray | None = None,
                                  p_out: Params | None = None):
    """Decoder over W = len(codes_in) ranks.  Returns (sum or None, codes_out or
    None, scales_out or None); ``err2`` is updated in place when given."""
    W = len(codes_in)
    codes_in = [np.ascontiguousarray(c, dtype=np.uint8) for c in codes_in]
    scales_in = [np.ascontiguousarray(s, dtype=np.uint16) for s in scales_in]
    cp = (ctypes.c_void_p * W)(*[c.ctypes.data for c in codes_in])
    sp = (ctypes.c_void_p * W)(*[s.ctypes.data for s in scales_in])
    sum_out = np.zeros(n, dtype=np.float32) if want_sum else None
    codes_out = scales_out = None
    if p_out is not None:
        codes_out = np.zeros(packed_bytes(n, p_out.bits, p_out.block), dtype=np.uint8)
        scales_out = np.zeros(num_blocks(n, p_out.block), dtype=np.uint16)
    if err2 is not None:
        assert err2.dtype == np.float32 and err2.flags.c_contiguous and err2.size == n
    rc = lib().orc_unpack_dequant_reduce_requant(
        ctypes.cast(cp, ctypes.c_void_p), ctypes.cast(sp, ctypes.c_void_p), W, n,
        ctypes.byref(p_in), _ptr(sum_out), _ptr(err2),
        ctypes.byref(p_out) if p_out is not None else None, _ptr(codes_out), _ptr(scales_out))
    if rc:
        raise ValueError("oracle rejected the arguments")
    return sum_out, codes_out, scales_out


def unpack_dequant(codes, scales, n: int, p: Params, mul: float = 1.0, out_dtype: int = F32):
    """All-gather-side decode: fl(fl(s*q) * mul) as fp32, or bf16 bit patterns."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    out = np.zeros(n, dtype=np.float32 if out_dtype == F32 else np.uint16)
    rc = lib().orc_unpack_dequant(_ptr(codes), _ptr(scales), n, ctypes.byref(p), ctypes.c_float(mul),
                                  out_dtype, _ptr(out))
    if rc:
        raise ValueError("oracle rejected the arguments")
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    L = lib()
    return np.array([L.orc_f32_to_bf16(float(v)) for v in x], dtype=np.uint16)


def qwd_encode(w: np.ndarray, ref: np.ndarray, p: Params):
    """Weight-difference encoder: codes of w - ref; ref advances in place."""
    w = np.ascontiguousarray(w)
    n = w.size
    assert ref.dtype == np.float32 and ref.flags.c_contiguous and ref.size == n
    codes = np.zeros(packed_bytes(n, p.bits, p.block), dtype=np.uint8)
    scales = np.zeros(num_blocks(n, p.block), dtype=np.uint16)
    if lib().orc_qwd_encode(_ptr(w), _dtype_code(w), n, _ptr(ref), ctypes.byref(p), _ptr(codes), _ptr(scales)):
        raise ValueError("oracle rejected the arguments")
    return codes, scales


def qwd_apply(codes, scales, n: int, p: Params, ref: np.ndarray, w_dtype=None):
    """Receiver update ref += s*q in place; returns the weights (fp32 or bf16 bits) or None."""
    out = None
    if w_dtype is not None:
        out = np.zeros(n, dtype=np.float32 if w_dtype == F32 else np.uint16)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    if lib().orc_qwd_apply(_ptr(codes), _ptr(scales), n, ctypes.byref(p), _ptr(ref), _ptr(out),
                           0 if w_dtype in (None, F32) else 1):
        raise ValueError("oracle rejected the arguments")
    return out


def sum_ranks(xs) -> np.ndarray:
    """Rank-ordered fp32 sum of W arrays (float32, or uint16 bf16 bits)."""
    xs = [np.ascontiguousarray(x) for x in xs]
    n, W = xs[0].size, len(xs)
    ptrs = (ctypes.c_void_p * W)(*[x.ctypes.data for x in xs])
    out = np.zeros(n, dtype=np.float32)
    if lib().orc_sum_ranks(ctypes.cast(ptrs, ctypes.c_void_p), _dtype_code(xs[0]), W, n, _ptr(out)):
        raise ValueError("oracle rejected the arguments")
    return out


def fwht(x: np.ndarray, H: int) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform of every H-block (a copy)."""
    y = np.ascontiguousarray(x, dtype=np.float32).copy()
    if lib().orc_fwht(_ptr(y), y.size, H):
        raise ValueError("bad transform arguments")
    return y


def roundtrip(x: np.ndarray, p: Params, err: np.ndarray | None = None):
    codes, scales = quantize_pack(x, p, err)
    deq = unpack_dequant(codes, scales, x.size, p)
    return codes, scales, deq
