"""bitscom_roundtrip_noalloc: the allocation-free roundtrip for callers that
cannot allocate device memory where they quantise (for example a gradient
hook that only holds the gradient buffer and must not call the CUDA
allocator).  Its codes and scales live in the library's fixed device array,
so its results must equal bitscom_roundtrip's with caller scratch -- checked
through the C ABI on two calls in a row (the second reuses the array the
first one left behind), at 0 ulp like every other parity test here.  This
file is collected last so that a run stopping at its first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu


def _abi_roundtrip(torch, bc, x, p, err, noalloc):
    L = bc.lib()
    n = x.numel()
    deq = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    dt = bc.F32 if x.dtype == torch.float32 else bc.BF16
    stream = torch.cuda.current_stream().cuda_stream
    errp = err.data_ptr() if err is not None else None
    if noalloc:
        st = L.bitscom_roundtrip_noalloc(x.data_ptr(), dt, n, errp, ctypes.byref(p.c()),
                                         deq.data_ptr(), stream)
    else:
        codes, scales = bc.alloc_codes(n, p)
        st = L.bitscom_roundtrip(x.data_ptr(), dt, n, errp, ctypes.byref(p.c()), codes.data_ptr(),
                                 scales.data_ptr(), deq.data_ptr(), stream)
    assert st == 0, bc.STATUS.get(st, st)
    torch.cuda.synchronize()
    return deq


@pytest.mark.parametrize("dtype,bits,block,rounding,ef,hadamard", [
    ("f32", 4, 128, 0, False, 0), ("bf16", 4, 128, 0, True, 0), ("f32", 2, 64, 1, True, 0),
    ("f32", 1, 256, 0, True, 0), ("bf16", 16, 8, 1, False, 0), ("f32", 12, 4096, 0, True, 0),
    ("f32", 4, 128, 0, True, 128)])
def test_noalloc_matches_roundtrip_twice(dtype, bits, block, rounding, ef, hadamard):
    # hadamard: the rotated codec takes the two-kernel path (encoder, then the
    # single-rank decoder) through the shared array
    torch, bc = need_gpu()
    p = bc.QParams(bits, block, rounding, seed=17, hadamard=hadamard)
    sizes = [3 * 4096, 5 * 4096] if hadamard else [3 * 4096 + 11, 5 * 4096]
    for call, n in enumerate(sizes):
        g = torch.Generator(device="cuda").manual_seed(100 + call)
        x = torch.randn(n, generator=g, device="cuda") * 1e-3
        if dtype == "bf16":
            x = x.to(torch.bfloat16)
        e0 = torch.randn(n, generator=g, device="cuda") * 1e-4
        e_ref = e0.clone() if ef else None
        e_new = e0.clone() if ef else None
        ref = _abi_roundtrip(torch, bc, x, p, e_ref, noalloc=False)
        got = _abi_roundtrip(torch, bc, x, p, e_new, noalloc=True)
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), f"call {call}"
        if ef:
            assert torch.equal(e_new.view(torch.int32), e_ref.view(torch.int32)), f"call {call}"


def test_noalloc_rejects_sizes_beyond_its_capacity():
    torch, bc = need_gpu()
    L = bc.lib()
    p = bc.QParams(16, 8)
    cap = L.bitscom_roundtrip_noalloc_max_elements(16, 8)
    assert cap == 4_194_304
    x = torch.zeros(cap + 8, device="cuda")
    deq = torch.empty(cap + 8, device="cuda")
    st = L.bitscom_roundtrip_noalloc(x.data_ptr(), bc.F32, cap + 8, None, ctypes.byref(p.c()),
                                     deq.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 1
    with pytest.raises(ValueError, match="capacity"):
        bc.roundtrip_noalloc(x, p, deq_out=deq)
    # the largest accepted size still works and matches
    xs = torch.randn(cap, device="cuda")
    ref = bc.roundtrip(xs, p)
    got = bc.roundtrip_noalloc(xs, p, deq_out=torch.empty(cap, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
    assert np.isfinite(got.cpu().numpy()).all()


def test_noalloc_call_allocates_nothing():
    # The point of the entry point: once the array is in place (a first call at
    # set-up) and the caller's own buffers exist, a call allocates no device
    # memory -- neither through torch's caching allocator nor outside it
    # (cudaMemGetInfo's free bytes are the same before and after, at points
    # where the device is idle).
    torch, bc = need_gpu()
    L = bc.lib()
    n = 5 * 4096 + 3
    p = bc.QParams(4, 128, bc.SR, seed=3)
    x = torch.randn(n, device="cuda")
    err = torch.zeros(n, device="cuda")
    deq = torch.empty(n, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        st = L.bitscom_roundtrip_noalloc(x.data_ptr(), bc.F32, n, err.data_ptr(), ctypes.byref(p.c()),
                                         deq.data_ptr(), stream)
        assert st == 0, bc.STATUS.get(st, st)

    call()                                   # set-up: the array's address, the kernels' modules
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), torch.cuda.mem_get_info()[0])
    call()
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(), torch.cuda.mem_get_info()[0])
    assert after == before
