"""Test helpers that read the codec's wire format with numpy alone.

They re-derive nothing from the oracle or from the CUDA path: unpacking uses
``numpy.unpackbits(bitorder="little")`` on the LSB-first bit stream, and scales
are read with numpy's own binary16 type.
"""
import numpy as np


def unpack_codes(codes: np.ndarray, bits: int, n: int) -> np.ndarray:
    """Unsigned codes u[0:n) from an LSB-first packed byte stream."""
    raw = np.frombuffer(np.ascontiguousarray(codes).view(np.uint8).tobytes(), dtype=np.uint8)
    stream = np.unpackbits(raw, bitorder="little")[: n * bits].reshape(n, bits).astype(np.uint64)
    return (stream << np.arange(bits, dtype=np.uint64)).sum(axis=1).astype(np.int64)


def pack_codes(u: np.ndarray, bits: int) -> np.ndarray:
    """Inverse of unpack_codes (numpy packbits, LSB-first)."""
    u = np.asarray(u, dtype=np.uint64)
    bitmat = ((u[:, None] >> np.arange(bits, dtype=np.uint64)) & 1).astype(np.uint8)
    return np.packbits(bitmat.reshape(-1), bitorder="little")


def codes_to_q(u: np.ndarray, bits: int) -> np.ndarray:
    """Offset-binary code -> signed integer level."""
    if bits == 1:
        return 2 * u - 1
    return u - (1 << (bits - 1))


def scales_f64(scales_bits: np.ndarray) -> np.ndarray:
    return np.asarray(scales_bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def qmax(bits: int) -> int:
    return (1 << (bits - 1)) - 1
