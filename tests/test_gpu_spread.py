"""Launches large enough for the encoders' spread grids (short-lived CTAs of a
few rows each, taken once a launch spans at least twelve waves of resident
CTAs): the 16-element encoder with error feedback and round to nearest
(every bf16 width, fp32), a launch just below its threshold (the 8-element
kernel's persistent grid), the 8-element kernel with stochastic rounding and
with the Walsh-Hadamard rotation, the 16-element encoder without error
feedback, the one-pass roundtrip, the weight-difference sender and the
rank-ordered sum of the full-precision local reduce.  The sizes
leave a margin of 1.4x or more on either side of the thresholds for a
152-SM GB300; every code, scale, error and output element is compared with
the CPU oracle, and guard bands around every output must survive."""
import numpy as np
import pytest

import oracle as O
from gpu_util import Guarded, bf16_bits_of, need_gpu

pytestmark = pytest.mark.gpu

N16 = 64 * 2 ** 20 + 77         # 16-element error-feedback encoder: 8,193 CTAs of 2 rows
N16_BELOW = 32 * 2 ** 20 + 5    # 4,097 two-row CTAs: below twelve waves, persistent 8-element kernel
N8 = 160 * 2 ** 20 + 77         # 8-element kernel: 5,121 CTAs of 8 rows
N8_HAD = 160 * 2 ** 20          # a multiple of the rotation block
N16_NOEF = 256 * 2 ** 20 + 77   # 16-element kernel without error feedback: 8,193 CTAs of 8 rows


def _x_and_err(n, dt, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(n, dtype=np.float32) * np.float32(1e-3))
    x[rng.integers(0, n, 64)] = 0.0
    x[rng.integers(0, n, 16)] *= 1000.0
    e = rng.standard_normal(n, dtype=np.float32) * np.float32(1e-6)
    return x, e


def _encode(torch, bc, x_host, dt, n, p, err_host, deq=False):
    xg = torch.from_numpy(x_host).cuda() if dt == "f32" else \
        torch.from_numpy(x_host.view(np.int16)).cuda().view(torch.bfloat16)
    codes = Guarded(torch, bc.packed_bytes(n, p.bits, p.block))
    scales = Guarded(torch, 2 * bc.num_blocks(n, p.block))
    err = Guarded(torch, 4 * n, fill=err_host) if err_host is not None else None
    out = Guarded(torch, 4 * n) if deq else None
    if deq:
        bc.roundtrip(xg, p, None, codes.view(torch.uint8), scales.view(torch.int16), out.view(torch.float32))
    else:
        bc.quantize_pack(xg, p, err.view(torch.float32) if err else None, codes.view(torch.uint8),
                         scales.view(torch.int16))
    torch.cuda.synchronize()
    del xg
    for g in (codes, scales, err, out):
        assert g is None or g.guards_intact()
    return (codes.host(np.uint8), scales.host(np.uint16), err.host(np.uint32) if err else None,
            out.host(np.uint32) if out else None)


def _check_encoder(torch, bc, dt, bits, block, n, rounding, hadamard=0, ef=True, seed=0):
    x, e = _x_and_err(n, dt, seed)
    xh = x if dt == "f32" else bf16_bits_of(torch, x)
    del x
    p = bc.QParams(bits, block, rounding, seed=123, index_offset=4 * 1000, hadamard=hadamard)
    po = O.params(bits, block, rounding, seed=123, index_offset=4 * 1000, hadamard=hadamard)
    codes, scales, err, _ = _encode(torch, bc, xh, dt, n, p, e if ef else None)
    e_ref = e if ef else None
    c_ref, s_ref = O.quantize_pack(xh, po, e_ref)
    assert codes.tobytes() == c_ref.tobytes(), "codes"
    assert np.array_equal(scales, s_ref), "scales"
    if ef:
        assert np.array_equal(err, e_ref.view(np.uint32)), "error feedback"


@pytest.mark.parametrize("dt,bits,block", [("bf16", b, 128) for b in (1, 2, 4, 8, 16)] +
                         [("f32", 4, 128), ("f32", 8, 4096), ("bf16", 4, 16)])
def test_ef_rtn_encoder_spread(dt, bits, block):
    torch, bc = need_gpu()
    _check_encoder(torch, bc, dt, bits, block, N16, bc.RTN, seed=bits * 7 + block)


def test_ef_rtn_encoder_below_spread_threshold():
    torch, bc = need_gpu()
    _check_encoder(torch, bc, "bf16", 4, 128, N16_BELOW, bc.RTN, seed=3)


@pytest.mark.parametrize("dt,bits,block", [("bf16", 2, 64), ("f32", 4, 128)])
def test_ef_sr_encoder_spread(dt, bits, block):
    torch, bc = need_gpu()
    _check_encoder(torch, bc, dt, bits, block, N8, bc.SR, seed=bits + block)


def test_hadamard_ef_encoder_spread():
    torch, bc = need_gpu()
    _check_encoder(torch, bc, "bf16", 8, 512, N8_HAD, bc.RTN, hadamard=128, seed=11)


@pytest.mark.parametrize("dt,bits", [("f32", 4), ("bf16", 2)])
def test_rtn_encoder_without_ef_spread(dt, bits):
    torch, bc = need_gpu()
    _check_encoder(torch, bc, dt, bits, 128, N16_NOEF, bc.RTN, ef=False, seed=bits)


def test_one_pass_roundtrip_spread():
    torch, bc = need_gpu()
    x, _ = _x_and_err(N16_NOEF, "f32", 21)
    p = bc.QParams(4, 128)
    codes, scales, _, deq = _encode(torch, bc, x, "f32", N16_NOEF, p, None, deq=True)
    c_ref, s_ref, d_ref = O.roundtrip(x, O.params(4, 128))
    assert codes.tobytes() == c_ref.tobytes()
    assert np.array_equal(scales, s_ref)
    assert np.array_equal(deq, d_ref.view(np.uint32))


def test_qwd_sender_spread():
    torch, bc = need_gpu()
    rng = np.random.default_rng(17)
    n = N8
    w = rng.standard_normal(n, dtype=np.float32) * np.float32(2e-2)
    ref = w - np.float32(1e-3) * rng.standard_normal(n, dtype=np.float32)
    wh = bf16_bits_of(torch, w)
    del w
    p = bc.QParams(4, 2048)
    wg = torch.from_numpy(wh.view(np.int16)).cuda().view(torch.bfloat16)
    rg = Guarded(torch, 4 * n, fill=ref)
    codes, scales = bc.qwd_encode(wg, rg.view(torch.float32), p)
    torch.cuda.synchronize()
    assert rg.guards_intact()
    h_ref = ref.copy()
    c_ref, s_ref = O.qwd_encode(wh, h_ref, O.params(4, 2048))
    assert codes.cpu().numpy().tobytes() == c_ref.tobytes()
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), s_ref)
    assert np.array_equal(rg.host(np.uint32), h_ref.view(np.uint32))


@pytest.mark.parametrize("dt,W", [("bf16", 4), ("f32", 2)])
def test_sum_ranks_spread(dt, W):
    # 4.2e7 elements: 20,508 stretches of 2,048 (one per CTA; twelve waves of
    # at most eight 256-thread CTAs on each of 152 SMs are 14,592), a ragged
    # last piece
    torch, bc = need_gpu()
    n = 42_000_003
    rng = np.random.default_rng(40 + W)
    xs = []
    for w in range(W):
        x = rng.standard_normal(n, dtype=np.float32) * np.float32(10.0 ** (w - 2))
        x[rng.integers(0, n, 64)] = -0.0
        xs.append(x if dt == "f32" else bf16_bits_of(torch, x))
    ref = O.sum_ranks(xs)
    dev = [torch.from_numpy(x if dt == "f32" else x.view(np.int16)).cuda() for x in xs]
    if dt == "bf16":
        dev = [d.view(torch.bfloat16) for d in dev]
    out = Guarded(torch, 4 * n)
    bc.sum_ranks(dev, out=out.view(torch.float32))
    torch.cuda.synchronize()
    assert out.guards_intact()
    assert np.array_equal(out.host(np.uint32), ref.view(np.uint32))
