"""The codec's divisions, checked on the GPU against CUDA's correctly rounded
operations: the quotient v / s (reciprocal of the fp16 scale + one residual
correction) against __fdiv_rn for every positive finite fp16 scale with
65,536 values each, concentrated where rounding decisions are made; the
reciprocal itself against __frcp_rn for every fp16 scale; and the block scale
fp16(absmax / Qmax) for every fp32 absmax in [2^-100, 2^100) and every Qmax."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "bit_gradient_communication_gb300", "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    need_gpu()
    so = tmp_path_factory.mktemp("probe") / "division_probe.so"
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                           "-fmad=false", "-Xcompiler", "-fPIC", "-shared", "-I", CSRC, "-I", INCLUDE,
                           os.path.join(HERE, "gpu_probes", "division_probe.cu"), "-o", str(so)])
    return ctypes.CDLL(str(so))


def test_reciprocal_of_every_fp16_scale(probe):
    # the reciprocal behind the quotient: hardware approximation + one Newton
    # step equals __frcp_rn for all 31,743 positive finite fp16 values
    bad = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 48)()
    assert probe.run_scale_probe(0, ctypes.byref(bad), first) == 0
    cases = np.array(first[:], dtype=np.uint32).reshape(16, 3)[: min(16, bad.value)]
    assert bad.value == 0, [(hex(h), hex(g), hex(r)) for h, g, r in cases]


def test_block_scale_exhaustive(probe):
    # the fp16 scale from every fp32 absmax in [2^-100, 2^100) for every Qmax
    # equals fp16(min(absmax / Qmax, 65504)) with CUDA's IEEE division
    bad = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 48)()
    assert probe.run_scale_probe(1, ctypes.byref(bad), first) == 0
    cases = np.array(first[:], dtype=np.uint32).reshape(16, 3)[: min(16, bad.value)]
    assert bad.value == 0, [(hex(u), int(b), hex(g)) for u, b, g in cases]


def test_quotient_matches_fdiv_rn(probe):
    lib = probe
    bad = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 48)()
    rc = lib.run_division_probe(ctypes.c_uint32(65536), ctypes.byref(bad), first)
    assert rc == 0
    cases = np.array(first[:], dtype=np.uint32).reshape(16, 3)[: min(16, bad.value)]
    assert bad.value == 0, [(hex(v), hex(h), hex(g)) for v, h, g in cases]
