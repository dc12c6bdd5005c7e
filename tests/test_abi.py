"""The C ABI without a GPU: the library builds and loads, exports every symbol
include/bitscom.h declares, and rejects bad arguments on the host before any
CUDA call (so these run on a CPU-only machine).  The bucket planner is host
code and is checked here too."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bitscom.h")


@pytest.fixture(scope="module")
def bc():
    from bit_gradient_communication_gb300 import _build
    _build.build()
    import bit_gradient_communication_gb300 as bc
    bc.lib()
    return bc


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bitscom_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("bitscom_quantize_pack", "bitscom_unpack_dequant_reduce_requant",
                     "bitscom_roundtrip", "bitscom_sched_allreduce"):
        assert required in names


def test_library_exports_every_declared_symbol(bc):
    out = subprocess.run(["nm", "-D", "--defined-only", bc.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(bitscom_\w+)", out))
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, missing
    L = bc.lib()
    for f in declared_functions():
        assert hasattr(L, f)


def test_library_is_built_for_sm_103a(bc):
    r = subprocess.run(["cuobjdump", "--list-elf", bc.LIB_PATH], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in r.stdout


def _p(bc, bits=4, block=128, rounding=0):
    return ctypes.byref(bc.QParams(bits, block, rounding).c())


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_sizes(bc):
    L = bc.lib()
    assert L.bitscom_num_blocks(1000, 128) == 8
    assert L.bitscom_packed_bytes(1000, 4, 128) == 8 * 128 * 4 // 8
    assert L.bitscom_packed_bytes(1000, 12, 128) == 8 * 128 * 12 // 8
    assert L.bitscom_packed_bytes(8, 1, 8) == 1
    assert L.bitscom_packed_bytes(-1, 4, 128) == -1
    assert L.bitscom_packed_bytes(10, 3, 128) == -1
    assert L.bitscom_status_string(2) == b"pointer not aligned"


@pytest.mark.parametrize("bits,block,rounding", [(3, 128, 0), (4, 100, 0), (4, 4, 0), (4, 8192, 0),
                                                 (4, 128, 2), (0, 128, 0)])
def test_encoder_rejects_bad_params(bc, bits, block, rounding):
    L = bc.lib()
    st = L.bitscom_quantize_pack(_fake(0x10000), 0, 1024, None, _p(bc, bits, block, rounding),
                                 _fake(0x20000), _fake(0x30000), None)
    assert st == 1


def test_encoder_argument_checks(bc):
    L = bc.lib()
    good = dict(x=0x10000, err=0x40000, codes=0x20000, scales=0x30000)

    def call(n=1024, dt=0, **kw):
        a = {**good, **kw}
        return L.bitscom_quantize_pack(_fake(a["x"]) if a["x"] else None, dt, n,
                                       _fake(a["err"]) if a["err"] else None, _p(bc),
                                       _fake(a["codes"]) if a["codes"] else None,
                                       _fake(a["scales"]) if a["scales"] else None, None)
    assert call(n=-1) == 1
    assert call(n=0, x=0, codes=0, scales=0) == 0        # nothing to do, nothing enqueued
    assert call(x=0) == 1
    assert call(codes=0) == 1
    assert call(x=0x10010) == 2                           # fp32 x needs 32 bytes
    assert call(dt=1, x=0x10008) == 2                     # bf16 x needs 16 bytes
    assert call(dt=1, x=0x10010, err=0x40010) == 2        # ... and error feedback 32 whatever x's type
    assert call(err=0x40004) == 2
    assert call(codes=0x20002) == 2                       # 4-bit codes need 4 bytes
    assert call(scales=0x30001) == 2
    assert call(dt=7) == 1
    assert L.bitscom_quantize_pack(_fake(0x10000), 0, 10, None, None, _fake(0x20000),
                                   _fake(0x30000), None) == 1


def test_decoder_argument_checks(bc):
    L = bc.lib()
    W = 3
    codes = (ctypes.c_void_p * W)(0x10000, 0x20000, 0x30000)
    scales = (ctypes.c_void_p * W)(0x40000, 0x50000, 0x60000)
    c = ctypes.cast(codes, ctypes.c_void_p)
    s = ctypes.cast(scales, ctypes.c_void_p)

    def call(W=3, n=1000, sum_out=0x70000, err2=None, p_out=None, co=None, so=None, c=c, s=s):
        return L.bitscom_unpack_dequant_reduce_requant(
            c, s, W, n, _p(bc), _fake(sum_out) if sum_out else None, _fake(err2) if err2 else None,
            p_out, _fake(co) if co else None, _fake(so) if so else None, None)
    assert call(W=0) == 1
    assert call(W=65) == 1
    assert call(sum_out=None) == 1                     # nothing to compute
    assert call(err2=0x80000) == 1                     # stage-2 error without requantisation
    assert call(p_out=_p(bc), co=None, so=0x90000) == 1
    assert call(sum_out=0x70010) == 2
    bad = (ctypes.c_void_p * W)(0x10000, 0x20002, 0x30000)
    assert call(c=ctypes.cast(bad, ctypes.c_void_p)) == 2
    nul = (ctypes.c_void_p * W)(0x10000, None, 0x30000)
    assert call(c=ctypes.cast(nul, ctypes.c_void_p)) == 1
    assert call(n=0) == 0


def test_roundtrip_argument_checks(bc):
    L = bc.lib()
    assert L.bitscom_roundtrip(_fake(0x10000), 0, 100, None, _p(bc), _fake(0x20000), _fake(0x30000),
                               None, None) == 1
    assert L.bitscom_roundtrip(_fake(0x10000), 0, 100, None, _p(bc), _fake(0x20000), _fake(0x30000),
                               _fake(0x40008), None) == 2


def test_scheduler_argument_checks(bc):
    L = bc.lib()
    h = ctypes.c_void_p()
    assert L.bitscom_sched_create(0, 0, ctypes.byref(h)) == 1
    assert L.bitscom_sched_create(9, 0, ctypes.byref(h)) == 1
    assert L.bitscom_sched_create(2, 0, None) == 1
    assert L.bitscom_sched_destroy(None) == 1
    assert L.bitscom_sched_wait(None, None, 1.0) == 1


def test_bucket_plan(bc):
    # 25 MiB of fp32 = 6,553,600 elements: one bucket (the single fusion bucket)
    assert bc.plan_buckets(6_553_600, 4, 256, 25 * 2 ** 20) == [0, 6_553_600]
    # 6.7e9 bf16 in 25 MiB buckets: 13,107,200 elements each, 512 buckets, last 2,220,800
    starts = bc.plan_buckets(6_700_000_000, 2, 64, 25 * 2 ** 20)
    assert len(starts) == 513
    assert starts[1] == 13_107_200
    assert starts[-1] - starts[-2] == 2_220_800
    # buckets are multiples of max(block, 128) elements
    s = bc.plan_buckets(10_000, 4, 512, 3000)
    assert all((b - a) % 512 == 0 for a, b in zip(s[:-2], s[1:-1]))
    assert s[0] == 0 and s[-1] == 10_000
    assert bc.plan_buckets(1000, 4, 128, 0) == [0, 1000]     # no bucketing
    assert bc.plan_buckets(0, 4, 128, 100) == [0]
    L = bc.lib()
    assert L.bitscom_sched_plan(10, 3, 128, 100, None, 0) == -1
    assert L.bitscom_sched_plan(10, 4, 100, 100, None, 0) == -1


def test_binding_refuses_cpu_tensors(bc):
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError, match="CUDA"):
        bc.quantize_pack(torch.zeros(16), bc.QParams(4, 8))


def test_hadamard_argument_checks(bc):
    L = bc.lib()
    def call(bits=4, block=128, H=128, n=1024, reserved=0):
        q = bc.QParams(bits, block, hadamard=H).c()
        q.reserved = reserved
        return L.bitscom_quantize_pack(_fake(0x10000), 0, n, None, ctypes.byref(q), _fake(0x20000),
                                       _fake(0x30000), None)
    assert call(H=4) == 1            # below 8
    assert call(H=96) == 1           # not a power of two
    assert call(H=512, block=512) == 1   # above 256
    assert call(H=128, block=64) == 1    # does not divide the block
    assert call(n=1000) == 1         # n not a multiple of H
    assert call(reserved=1) == 1
    assert call(bits=12) == 3        # no rotated kernel for 12-bit codes
    # decoder: both stages must share the rotation
    codes = (ctypes.c_void_p * 1)(0x10000)
    scales = (ctypes.c_void_p * 1)(0x40000)
    st = L.bitscom_unpack_dequant_reduce_requant(
        ctypes.cast(codes, ctypes.c_void_p), ctypes.cast(scales, ctypes.c_void_p), 1, 1024,
        ctypes.byref(bc.QParams(4, 128, hadamard=128).c()), None, None,
        ctypes.byref(bc.QParams(4, 128).c()), _fake(0x20000), _fake(0x30000), None)
    assert st == 1


def test_qwd_argument_checks(bc):
    L = bc.lib()
    q = bc.QParams(4, 2048).c()
    assert L.bitscom_qwd_encode(_fake(0x10000), 0, 4096, None, ctypes.byref(q), _fake(0x20000),
                                _fake(0x30000), None) == 1          # reference required
    qh = bc.QParams(4, 128, hadamard=128).c()
    assert L.bitscom_qwd_encode(_fake(0x10000), 0, 4096, _fake(0x40000), ctypes.byref(qh), _fake(0x20000),
                                _fake(0x30000), None) == 1          # no rotation for weights
    q12 = bc.QParams(12, 2048).c()
    assert L.bitscom_qwd_encode(_fake(0x10000), 0, 4096, _fake(0x40000), ctypes.byref(q12),
                                _fake(0x20000), _fake(0x30000), None) == 3
    assert L.bitscom_qwd_apply(_fake(0x20000), _fake(0x30000), 4096, ctypes.byref(q), _fake(0x40004),
                               None, 0, None) == 2                  # reference alignment
    assert L.bitscom_qwd_apply(_fake(0x20000), _fake(0x30000), 0, ctypes.byref(q), None, None, 0, None) == 0


def test_sum_ranks_argument_checks(bc):
    L = bc.lib()
    xs = (ctypes.c_void_p * 3)(0x10000, 0x20000, 0x30000)
    call = lambda W=3, n=1024, dt=0, out=0x40000, x=xs: L.bitscom_sum_ranks(
        ctypes.cast(x, ctypes.c_void_p) if x is not None else None, dt, W, n, _fake(out) if out else None, None)
    assert call(n=0) == 0                                   # nothing enqueued
    assert call(W=0) == 1 and call(W=65) == 1 and call(n=-1) == 1 and call(dt=2) == 1
    assert call(out=0) == 1 and call(x=None) == 1
    assert call(x=(ctypes.c_void_p * 3)(0x10000, 0, 0x30000)) == 1
    assert call(x=(ctypes.c_void_p * 3)(0x10000, 0x20010, 0x30000)) == 2    # fp32 inputs need 32 bytes
    assert call(dt=1, x=(ctypes.c_void_p * 3)(0x10000, 0x20008, 0x30000)) == 2  # bf16 inputs need 16
    assert call(out=0x40010) == 2
