"""Regression vectors written by tests/golden/make_golden.py (oracle only):
the oracle must still reproduce them, and so must the CUDA path."""
import json
import os

import numpy as np
import pytest

import oracle as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "oracle_vectors.json")))


def _arr(h, dt):
    return np.frombuffer(bytes.fromhex(h), dtype=dt).copy()


def _case_inputs(c):
    x = _arr(c["x"], np.float32 if c["dtype"] == "f32" else np.uint16)
    e = _arr(c["err_in"], np.float32)
    return x, e


@pytest.mark.parametrize("k", range(len(GOLD["encoder"])))
def test_oracle_reproduces_golden_encoder(orc, k):
    c = GOLD["encoder"][k]
    x, e = _case_inputs(c)
    p = orc.params(c["bits"], c["block"], c["rounding"], seed=c["seed"], index_offset=c["index_offset"],
                   hadamard=c["hadamard"])
    e_out = e.copy() if c["ef"] else None
    codes, scales = orc.quantize_pack(x, p, e_out)
    assert codes.tobytes().hex() == c["codes"] and scales.tobytes().hex() == c["scales"]
    if c["ef"]:
        assert e_out.tobytes().hex() == c["err_out"]
    assert orc.unpack_dequant(codes, scales, c["n"], p, 0.5, orc.BF16).tobytes().hex() == c["mean_bf16"]


def test_golden_exact_fraction_case_hits_the_tie():
    # the stochastic-rounding case built at the exact fraction: the stored codes
    # give the q the construction fixes (q = 0 where 1 + t rounded to fp32
    # would have given -1)
    from codec_util import codes_to_q, unpack_codes
    cases = [c for c in GOLD["encoder"] if c.get("expect_q")]
    assert len(cases) == 1
    c = cases[0]
    q = codes_to_q(unpack_codes(_arr(c["codes"], np.uint8), c["bits"], c["n"]), c["bits"])
    assert len(c["expect_q"]) == 9
    for pos, q_expected in c["expect_q"]:
        assert q[pos] == q_expected, pos


def test_oracle_reproduces_golden_decoder(orc):
    d = GOLD["decoder"]
    e2 = _arr(d["err2_in"], np.float32)
    s, co, so = orc.unpack_dequant_reduce_requant(
        [_arr(h, np.uint8) for h in d["codes_in"]], [_arr(h, np.uint16) for h in d["scales_in"]], d["n"],
        orc.params(4, 128), True, e2, orc.params(4, 128, 1, seed=5, philox_stream=1))
    assert s.tobytes().hex() == d["sum"] and co.tobytes().hex() == d["codes_out"]
    assert so.tobytes().hex() == d["scales_out"] and e2.tobytes().hex() == d["err2_out"]


@pytest.mark.gpu
@pytest.mark.parametrize("k", range(len(GOLD["encoder"])))
def test_cuda_reproduces_golden_encoder(k):
    from gpu_util import need_gpu
    torch, bc = need_gpu()
    c = GOLD["encoder"][k]
    x, e = _case_inputs(c)
    xg = torch.from_numpy(x if c["dtype"] == "f32" else x.view(np.int16)).cuda()
    if c["dtype"] == "bf16":
        xg = xg.view(torch.bfloat16)
    p = bc.QParams(c["bits"], c["block"], c["rounding"], seed=c["seed"], index_offset=c["index_offset"],
                   hadamard=c["hadamard"])
    eg = torch.from_numpy(e.copy()).cuda() if c["ef"] else None
    codes, scales = bc.quantize_pack(xg, p, eg)
    mean = bc.unpack_dequant(codes, scales, c["n"], p, 0.5, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert codes.cpu().numpy().tobytes().hex() == c["codes"]
    assert scales.cpu().numpy().tobytes().hex() == c["scales"]
    if c["ef"]:
        assert eg.cpu().numpy().tobytes().hex() == c["err_out"]
    assert mean.view(torch.int16).cpu().numpy().tobytes().hex() == c["mean_bf16"]
