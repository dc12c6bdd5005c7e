"""The codec's fp32 quotient v / s (reciprocal of the fp16 scale + two
residual corrections) equals CUDA's correctly rounded __fdiv_rn: checked on
the GPU for every positive finite fp16 scale with 65,536 values each,
concentrated where rounding decisions are made (quotients within a few ulps
of integers and half-integers up to 32768)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "bit_gradient_communication_gb300", "csrc")


def test_quotient_matches_fdiv_rn(tmp_path):
    need_gpu()
    so = tmp_path / "division_probe.so"
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                           "-fmad=false", "-Xcompiler", "-fPIC", "-shared", "-I", CSRC,
                           os.path.join(HERE, "gpu_probes", "division_probe.cu"), "-o", str(so)])
    lib = ctypes.CDLL(str(so))
    bad = ctypes.c_ulonglong(0)
    first = (ctypes.c_uint32 * 48)()
    rc = lib.run_division_probe(ctypes.c_uint32(65536), ctypes.byref(bad), first)
    assert rc == 0
    cases = np.array(first[:], dtype=np.uint32).reshape(16, 3)[: min(16, bad.value)]
    assert bad.value == 0, [(hex(v), hex(h), hex(g)) for v, h, g in cases]
