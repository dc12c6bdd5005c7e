"""Launches large enough for the encoders' spread grids (short-lived CTAs of a
few rows each, taken once a launch spans at least twelve waves of resident
CTAs): the 16-element encoder with error feedback and round to nearest
(every bf16 width, fp32), a launch just below its threshold (the 8-element
kernel's persistent grid), the 8-element kernel with stochastic rounding and
with the Walsh-Hadamard rotation, the 16-element encoder without error
feedback, the one-pass roundtrip, the weight-difference sender, the
rank-ordered sum of the full-precision local reduce, and the decoders whose
grids spread (eight ranks 8 -> 4 bits, and the eight-rank sum alone).  The
sizes
leave a margin of 1.4x or more on either side of the thresholds for a
152-SM GB300; every code, scale, error and output element is compared with
the CPU oracle (the decoders on block-aligned windows: every output block
depends only on the same block of every rank and on its own stage-2 error,
so a window is a complete oracle problem), and guard bands around every
output must survive."""
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


def _random_ranks(torch, n, bits, block, seed, W=8):
    """W ranks of random codes and fp16 scales (with some zero scales) on the
    device, from a seeded device generator."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    nbytes = (n + block - 1) // block * block * bits // 8
    nb = (n + block - 1) // block
    codes, scales = [], []
    for _ in range(W):
        codes.append(torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g))
        s = (torch.randn(nb, device="cuda", generator=g).abs() * 1e-3).half()
        s[torch.randint(0, nb, (max(1, nb // 50),), device="cuda", generator=g)] = 0.0
        scales.append(s.view(torch.int16))
    return codes, scales


def _windows(n, unit, count, seed):
    """Block-aligned windows [lo, hi) of 16 units: the first, the last (ragged
    when n is) and `count` others."""
    nu = (n + unit - 1) // unit
    rng = np.random.default_rng(seed)
    starts = {0, max(0, nu - 16)} | set(int(v) for v in rng.integers(0, max(1, nu - 16), count))
    return [(b * unit, min((b + 16) * unit, n)) for b in sorted(starts)]


def _host(t, lo, hi):
    return t[lo:hi].cpu().numpy()


def test_decoder_8_to_4_spread():
    # 1.6e8 + 1,613 outputs of eight ranks' 8-bit codes in blocks of 512,
    # requantised to 4 bits in blocks of 128 with stage-2 error: 40,961 rows,
    # 5,121 CTAs of eight rows (twelve waves of 304 resident are 3,648)
    torch, bc = need_gpu()
    n = 160 * 2 ** 20 + 1613
    p_in, p_out = bc.QParams(8, 512), bc.QParams(4, 128)
    codes, scales = _random_ranks(torch, n, 8, 512, 7)
    e2_0 = torch.randn(n, device="cuda") * 1e-6
    e2 = Guarded(torch, 4 * n)
    e2.view(torch.float32).copy_(e2_0)
    co = Guarded(torch, bc.packed_bytes(n, 4, 128))
    so = Guarded(torch, 2 * bc.num_blocks(n, 128))
    bc.unpack_dequant_reduce_requant(codes, scales, n, p_in, err2=e2.view(torch.float32), p_out=p_out,
                                     codes_out=co.view(torch.uint8), scales_out=so.view(torch.int16))
    torch.cuda.synchronize()
    assert e2.guards_intact() and co.guards_intact() and so.guards_intact()
    e2_out, co_out, so_out = e2.view(torch.float32), co.view(torch.uint8), so.view(torch.int16)
    for lo, hi in _windows(n, 512, 12, 3):
        m = hi - lo
        cw = [_host(c, lo, lo + (m + 511) // 512 * 512) for c in codes]
        sw = [_host(sc, lo // 512, lo // 512 + (m + 511) // 512).view(np.uint16) for sc in scales]
        ew = _host(e2_0, lo, hi).copy()
        _, c_ref, s_ref = O.unpack_dequant_reduce_requant(cw, sw, m, O.params(8, 512), False, ew, O.params(4, 128))
        assert _host(co_out, lo // 2, lo // 2 + c_ref.size).tobytes() == c_ref.tobytes(), f"codes at {lo}"
        assert np.array_equal(_host(so_out, lo // 128, lo // 128 + s_ref.size).view(np.uint16), s_ref), f"scales at {lo}"
        assert np.array_equal(_host(e2_out, lo, hi).view(np.uint32), ew.view(np.uint32)), f"e2 at {lo}"


def test_sum_only_decoder_spread():
    # 5.2e8 + 77 outputs, the sum of eight ranks' 4-bit codes in blocks of
    # 128 (the 16-element kernel without requantisation): 126,954 rows, 7,935
    # CTAs of sixteen rows (twelve waves of 456 resident are 5,472)
    torch, bc = need_gpu()
    n = 520_000_077
    p = bc.QParams(4, 128)
    codes, scales = _random_ranks(torch, n, 4, 128, 8)
    out = Guarded(torch, 4 * n)
    bc.unpack_dequant_reduce_requant(codes, scales, n, p, sum_out=out.view(torch.float32))
    torch.cuda.synchronize()
    assert out.guards_intact()
    sums = out.view(torch.float32)
    for lo, hi in _windows(n, 128, 16, 4):
        m = hi - lo
        cw = [_host(c, lo // 2, (lo + (m + 127) // 128 * 128) // 2) for c in codes]
        sw = [_host(sc, lo // 128, lo // 128 + (m + 127) // 128).view(np.uint16) for sc in scales]
        ref, _, _ = O.unpack_dequant_reduce_requant(cw, sw, m, O.params(4, 128), True)
        assert np.array_equal(_host(sums, lo, hi).view(np.uint32), ref.view(np.uint32)), f"sum at {lo}"


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_rotated_decode_spread(out):
    # The all-gather-side decode with the inverse Walsh-Hadamard rotation
    # (H = 128, 4-bit blocks of 128) over 4e7 elements: 4,883 rows of 8192,
    # four rows per CTA, the fp32 output staged through shared memory; every
    # transform block depends only on its own codes and scale, so block-aligned
    # windows are complete oracle problems
    torch, bc = need_gpu()
    n = 40_000_000
    p = bc.QParams(4, 128, hadamard=128)
    po = O.params(4, 128, hadamard=128)
    codes, scales = _random_ranks(torch, n, 4, 128, 21, W=1)
    esz = 4 if out == "f32" else 2
    g = Guarded(torch, esz * n)
    mul = float(np.float32(1 / 8))
    bc.unpack_dequant(codes[0], scales[0], n, p, mul, out=g.view(torch.float32 if out == "f32" else torch.bfloat16))
    torch.cuda.synchronize()
    assert g.guards_intact()
    res = g.view(torch.int32 if out == "f32" else torch.int16)
    for lo, hi in _windows(n, 128, 16, 5):
        m = hi - lo
        cw = _host(codes[0], lo // 2, hi // 2)
        sw = _host(scales[0], lo // 128, hi // 128).view(np.uint16)
        ref = O.unpack_dequant(cw, sw, m, po, mul, O.F32 if out == "f32" else O.BF16)
        got = _host(res, lo, hi).view(np.uint32 if out == "f32" else np.uint16)
        assert np.array_equal(got, ref.view(np.uint32 if out == "f32" else np.uint16)), f"window at {lo}"
