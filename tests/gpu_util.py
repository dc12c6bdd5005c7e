"""Helpers for the GPU parity tests: guarded device buffers and host copies."""
import numpy as np
import pytest

GUARD = 4096          # bytes of sentinel before and after every output buffer
SENTINEL = 0xA5


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_gradient_communication_gb300 as bc
    from bit_gradient_communication_gb300 import _build
    _build.build()
    bc.lib()
    return torch, bc


class Guarded:
    """A device byte buffer with sentinel bands; .view(dtype) is the payload."""

    def __init__(self, torch, nbytes, fill=None, device="cuda"):
        self.torch = torch
        self.nbytes = nbytes
        self.raw = torch.full((nbytes + 2 * GUARD,), SENTINEL, dtype=torch.uint8, device=device)
        if fill is not None:
            src = torch.as_tensor(np.frombuffer(np.ascontiguousarray(fill).tobytes(), dtype=np.uint8).copy())
            self.raw[GUARD:GUARD + nbytes].copy_(src.to(device))

    def view(self, dtype):
        return self.raw[GUARD:GUARD + self.nbytes].view(dtype)

    def host(self, np_dtype):
        return self.raw[GUARD:GUARD + self.nbytes].cpu().numpy().view(np_dtype).copy()

    def guards_intact(self):
        g = self.raw.cpu().numpy()
        return bool((g[:GUARD] == SENTINEL).all() and (g[GUARD + self.nbytes:] == SENTINEL).all())


def bf16_bits_of(torch, x_f32_np):
    """bf16 bit patterns (uint16) of an fp32 array, rounded by torch's cast."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32_np)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()
