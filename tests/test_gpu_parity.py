"""CUDA path vs the CPU oracle, bit for bit, through the C ABI.

Codes, packed bytes, fp16 scales, error-feedback buffers, rank sums and
dequantised values must be identical (0 ulp): every fp32 step of the method
is a fixed sequence of correctly rounded operations.  Sizes span several
4096-element rows with ragged tails; every output buffer sits between
sentinel bands that must survive the call.
"""
import numpy as np
import pytest

import oracle as O
from codec_util import codes_to_q, unpack_codes
from gpu_util import Guarded, bf16_bits_of, need_gpu

pytestmark = pytest.mark.gpu

BITS = [1, 2, 4, 8, 12, 16]
SIZES = [1, 13, 4096, 3 * 4096 + 40, 5 * 4096 + 1]


def _inputs(n, dtype, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-4, 1)).astype(np.float32)
    # a few exact zeros, negative zeros and outliers
    if n > 16:
        x[rng.integers(0, n, 3)] = 0.0
        x[rng.integers(0, n, 2)] = -0.0
        x[rng.integers(0, n, 2)] *= 1000.0
    e = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    return x, e


def _run_encode(torch, bc, x_host, dt, n, p, err_host):
    """GPU encoder on guarded buffers; returns codes, scales, err (host)."""
    if dt == "f32":
        xg = torch.from_numpy(x_host).cuda()
    else:
        xg = torch.from_numpy(x_host.view(np.int16)).cuda().view(torch.bfloat16)
    codes = Guarded(torch, bc.packed_bytes(n, p.bits, p.block))
    scales = Guarded(torch, 2 * bc.num_blocks(n, p.block))
    err = Guarded(torch, 4 * n, fill=err_host) if err_host is not None else None
    bc.quantize_pack(xg, p, err.view(torch.float32) if err else None,
                     codes.view(torch.uint8), scales.view(torch.int16))
    torch.cuda.synchronize()
    assert codes.guards_intact() and scales.guards_intact() and (err is None or err.guards_intact())
    return codes.host(np.uint8), scales.host(np.uint16), (err.host(np.float32) if err else None)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("block", [8, 16, 32, 128, 512, 4096])
@pytest.mark.parametrize("mode", ["rtn", "rtn_ef", "sr", "sr_ef"])
def test_encoder_matches_oracle(dt, bits, block, mode):
    # (block 16: the 16-element encoders' stochastic path, which blocks of 32
    # and more leave to the 32-element one)
    torch, bc = need_gpu()
    sr = mode.startswith("sr")
    ef = mode.endswith("ef")
    for k, n in enumerate(SIZES):
        x, e = _inputs(n, dt, seed=bits * 1000 + block + k)
        xh = x if dt == "f32" else bf16_bits_of(torch, x)
        offset = [0, 3, 2 ** 33 + 5, 6, 2 ** 38 + 1][k]     # the last: counter word 1 non-zero
        p = bc.QParams(bits, block, bc.SR if sr else bc.RTN, seed=0x1234_5678_9ABC + k,
                       index_offset=offset, philox_stream=k & 1)
        po = O.params(bits, block, O.SR if sr else O.RTN, seed=p.seed, index_offset=offset,
                      philox_stream=p.philox_stream)
        codes, scales, err = _run_encode(torch, bc, xh, dt, n, p, e.copy() if ef else None)
        e_ref = e.copy() if ef else None
        c_ref, s_ref = O.quantize_pack(xh, po, e_ref)
        assert codes.tobytes() == c_ref.tobytes(), f"codes differ at n={n}"
        assert np.array_equal(scales, s_ref), f"scales differ at n={n}"
        if ef:
            assert np.array_equal(err.view(np.uint32), e_ref.view(np.uint32)), f"e' differs at n={n}"


def test_encoder_is_deterministic():
    torch, bc = need_gpu()
    n = 7 * 4096 + 3
    x, e = _inputs(n, "f32", 5)
    p = bc.QParams(4, 128, bc.SR, seed=7)
    a = _run_encode(torch, bc, x, "f32", n, p, e.copy())
    b = _run_encode(torch, bc, x, "f32", n, p, e.copy())
    assert a[0].tobytes() == b[0].tobytes() and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_encoder_sr_alignment_paths(bits, dt):
    # Stochastic rounding without error feedback takes a 16-elements-per-thread
    # encoder when the code pointer is aligned to 2b bytes and the general one
    # when it is aligned to b bytes only; both must give the oracle's bits.
    torch, bc = need_gpu()
    n = 3 * 4096 + 77
    x, _ = _inputs(n, dt, 123 + bits)
    xh = x if dt == "f32" else bf16_bits_of(torch, x)
    xg = torch.from_numpy(xh).cuda() if dt == "f32" else torch.from_numpy(xh.view(np.int16)).cuda().view(torch.bfloat16)
    p = bc.QParams(bits, 128, bc.SR, seed=17, index_offset=6)
    c_ref, s_ref = O.quantize_pack(xh, O.params(bits, 128, O.SR, seed=17, index_offset=6))
    nb = bc.packed_bytes(n, bits, 128)
    for offset in (0, bits):
        buf = torch.zeros(nb + 32, dtype=torch.uint8, device="cuda")
        codes = buf[offset:offset + nb]
        scales = torch.zeros(bc.num_blocks(n, 128), dtype=torch.int16, device="cuda")
        bc.quantize_pack(xg, p, None, codes, scales)
        torch.cuda.synchronize()
        assert codes.cpu().numpy().tobytes() == c_ref.tobytes(), f"offset {offset}"
        assert np.array_equal(scales.cpu().numpy().view(np.uint16), s_ref), f"offset {offset}"


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits", [2, 4, 8, 12, 16])
@pytest.mark.parametrize("block", [32, 64, 128, 256, 512, 1024, 2048, 4096])
def test_sr_encoder_32_per_thread_paths(dt, bits, block):
    # Stochastic rounding without error feedback of 2- to 16-bit codes in
    # blocks of 32 .. 4096 takes an encoder with 32 elements per thread
    # (8192-element rows; blocks of 2048 and 4096 reduce across warps).  Its
    # straight-line form covers index offsets that are multiples of 4 and
    # elements of magnitude 2^-96 or more, with a one- or two-sided clamp
    # chosen per warp from the scales; a thread's row with anything else is
    # redone on the general path.  Rows on both paths, full rows and a ragged
    # last one, subnormal and saturated scales, offsets on both sides of a
    # Philox counter carry, and code pointers aligned for it and only for the
    # older encoders (shifted by 2b bytes) must all give the oracle's bits.
    torch, bc = need_gpu()
    rng = np.random.default_rng(bits * 100 + block)
    R = 8192
    n = 5 * R + 3 * 1024 + 40
    x = rng.laplace(0.0, 1e-3, n).astype(np.float32)
    x[R + 5] = 1e-35                                  # 0 < |v| < 2^-96
    x[R + 6] = 0.0                                    # a zero in the same thread's 32 elements
    x[2 * R + 64] = 0.0                               # zeros alone keep the straight-line form
    x[3 * R + 7 * 32 + 1] = -0.0
    x[2 * R + 1024:3 * R][rng.random(R - 1024) < 0.05] = 0.0
    b0 = (4 * R) // block                             # a subnormal (or zero) scale, then a saturated one
    x[b0 * block:(b0 + 1) * block] *= np.float32(1e-3)
    x[(b0 + 1) * block:(b0 + 2) * block] *= np.float32(1e11)
    xh = x if dt == "f32" else bf16_bits_of(torch, x)
    xg = torch.from_numpy(xh).cuda() if dt == "f32" else torch.from_numpy(xh.view(np.int16)).cuda().view(torch.bfloat16)
    nb = bc.packed_bytes(n, bits, block)
    for off in (0, 4 * 12345, (1 << 34) - R - 64, 2):
        p = bc.QParams(bits, block, bc.SR, seed=0xC0FFEE + off, index_offset=off)
        c_ref, s_ref = O.quantize_pack(xh, O.params(bits, block, O.SR, seed=p.seed, index_offset=off))
        for shift in (0, 2 * bits):
            buf = torch.zeros(nb + 64, dtype=torch.uint8, device="cuda")
            codes = buf[shift:shift + nb]
            scales = torch.zeros(bc.num_blocks(n, block), dtype=torch.int16, device="cuda")
            bc.quantize_pack(xg, p, None, codes, scales)
            torch.cuda.synchronize()
            tag = f"offset {off} code shift {shift}"
            assert codes.cpu().numpy().tobytes() == c_ref.tobytes(), tag
            assert np.array_equal(scales.cpu().numpy().view(np.uint16), s_ref), tag
            assert not buf[:shift].any() and not buf[shift + nb:].any(), tag


def test_encoder_special_blocks():
    # zero blocks, underflowing and subnormal scales, saturation, negative zero
    torch, bc = need_gpu()
    n = 4096
    x = np.zeros(n, np.float32)
    x[128:256] = 2.0 ** -26          # absmax/7 underflows fp16 -> s = 0
    x[256:384] = 3 * 2.0 ** -24 * 7  # subnormal scale
    x[384:512] = 1e6                 # saturated scale
    x[512] = -0.0
    x[640:768] = np.linspace(-3, 3, 128)
    for bits in BITS:
        for rounding in (bc.RTN, bc.SR):
            for ef in (False, True):
                e = np.zeros(n, np.float32)
                p = bc.QParams(bits, 128, rounding, seed=3)
                codes, scales, err = _run_encode(torch, bc, x, "f32", n, p, e.copy() if ef else None)
                e_ref = e.copy() if ef else None
                c_ref, s_ref = O.quantize_pack(x, O.params(bits, 128, rounding, seed=3), e_ref)
                tag = f"bits={bits} rounding={rounding} ef={ef}"
                assert codes.tobytes() == c_ref.tobytes() and np.array_equal(scales, s_ref), tag
                if ef:
                    assert np.array_equal(err.view(np.uint32), e_ref.view(np.uint32)), tag


@pytest.mark.parametrize("bits", [2, 4, 8, 12, 16])
@pytest.mark.parametrize("block", [32, 128, 4096])
def test_sr_codes_past_the_range_are_clamped(bits, block):
    # Blocks whose scale rounds down by half an fp16 ulp (absmax / Qmax = 1 +
    # 2^-11, a tie that goes to 1.0) give t = +-Qmax (1 + 2^-11) at the block
    # maximum.  Placed where the element's u = (r mod 2^23) 2^-23 is within
    # Qmax 2^-11 of 1 (for -absmax) or of 0 (for +absmax), stochastic rounding
    # lands on -Qmax - 1 or Qmax + 1 before the clamp; the codes must be the
    # oracle's (the clamped ones) with and without error feedback.
    torch, bc = need_gpu()
    Q = (1 << (bits - 1)) - 1
    A = np.float32(Q * (1 + 2.0 ** -11))
    assert np.float32(A / np.float32(Q)).astype(np.float16) == np.float16(1.0)
    n, seed, off = 1 << 18, 21, 1 << 20
    u = (O.random_words(seed, 0, off, n) & 0x7FFFFF).astype(np.float64) * 2.0 ** -23
    rng = np.random.default_rng(bits + block)
    x = rng.uniform(-A / 2, A / 2, n).astype(np.float32)
    idx = np.arange(n)
    low = np.nonzero((u >= 1 - Q * 2.0 ** -11) & (idx % 2 == 0))[0]      # disjoint sets (at 12 and 16
    high = np.nonzero((u < Q * 2.0 ** -11) & (idx % 2 == 1))[0]           # bits every u qualifies)
    x[low], x[high] = -A, A
    # the unclamped stochastic rounding of the planted elements leaves the range
    t = np.float64(np.float32(A)) / 1.0
    assert (np.floor(-t) + (u[low] < -t - np.floor(-t)) < -Q).any()
    assert (np.floor(t) + (u[high] < t - np.floor(t)) > Q).any()
    p = bc.QParams(bits, block, bc.SR, seed=seed, index_offset=off)
    for ef in (False, True):
        e = np.zeros(n, np.float32)
        codes, scales, err = _run_encode(torch, bc, x, "f32", n, p, e.copy() if ef else None)
        e_ref = e.copy() if ef else None
        c_ref, s_ref = O.quantize_pack(x, O.params(bits, block, O.SR, seed=seed, index_offset=off), e_ref)
        assert np.array_equal(scales, s_ref)
        assert codes.tobytes() == c_ref.tobytes(), f"ef={ef}"
        if ef:
            assert np.array_equal(err.view(np.uint32), e_ref.view(np.uint32))
        q = codes_to_q(unpack_codes(codes, bits, n), bits)
        assert q.min() == -Q and q.max() == Q


def _zero_fraction_indices(seed, count=3):
    """Global indices whose Philox word has zero low 23 bits (u = 0), found
    with the oracle's generator: there a positive t however small rounds up."""
    words = O.random_words(seed, 0, 0, 1 << 24)
    hits = np.nonzero((words & 0x7FFFFF) == 0)[0]
    assert hits.size >= count
    return [int(h) for h in hits[:count]]


@pytest.mark.parametrize("bits", [2, 4, 8, 12, 16])
@pytest.mark.parametrize("absmax", [10.5, 14.0, 21.0])
def test_encoder_sr_tiny_elements(bits, absmax):
    # Stochastic rounding of elements whose quotient t = v/s is tiny or
    # subnormal, placed where u = 0 so that only t > 0 decides q = 1; v/s near
    # the bottom of the subnormal range (2^-149 / s for s around 1.5 .. 3)
    # rounds to 0 or to 2^-149 by IEEE division.  Also -0, +0, the 2^-96
    # boundary and a block whose scale underflows.
    torch, bc = need_gpu()
    seed = 11
    n = 4096
    rng = np.random.default_rng(bits * 13 + int(absmax))
    specials = [2.0 ** -149, -2.0 ** -149, 3 * 2.0 ** -149, 2.0 ** -100, -2.0 ** -97, 2.0 ** -96,
                -2.0 ** -96, 0.0, -0.0, 1.5 * 2.0 ** -126, 2.0 ** -130]
    for h in _zero_fraction_indices(seed):
        for pos in (200, 203):                       # 203: index offset not a multiple of 4
            for tiny in specials[:4]:
                x = (rng.standard_normal(n) * absmax / 8).astype(np.float32)
                x[128:256] = np.clip(x[128:256], -absmax / 2, absmax / 2)
                x[130] = absmax
                x[pos] = tiny
                x[pos + 1:pos + 1 + len(specials)] = specials
                x[1024:1152] = 2.0 ** -140           # scale underflows to 0
                x[1030] = 2.0 ** -149
                p = bc.QParams(bits, 128, bc.SR, seed=seed, index_offset=h - pos)
                for ef in (False, True):
                    e = np.zeros(n, np.float32)
                    codes, scales, err = _run_encode(torch, bc, x, "f32", n, p, e.copy() if ef else None)
                    e_ref = e.copy() if ef else None
                    c_ref, s_ref = O.quantize_pack(x, O.params(bits, 128, O.SR, seed=seed, index_offset=h - pos),
                                                   e_ref)
                    tag = f"h={h} pos={pos} tiny={tiny} ef={ef}"
                    assert codes.tobytes() == c_ref.tobytes(), tag
                    assert np.array_equal(scales, s_ref), tag
                    if ef:
                        assert np.array_equal(err.view(np.uint32), e_ref.view(np.uint32)), tag


def _fraction_ties(bits, n, block, seed, stream, index_offset):
    """Values whose stochastic rounding needs the exact fraction t - floor(t):
    every block has scale 1 (its first element is Qmax, the rest lie inside
    +-Qmax), and wherever the element's u = (r mod 2^23) 2^-23 lies in
    (1/2, 3/4) its t is u + d - 1 for d = 2^-25, 0, -2^-25 in turn.  Those
    round to q = 0, -1, -1: for d = 2^-25, 1 + t rounded to fp32 would be a
    tie that goes to u itself (words from the oracle's Philox)."""
    Q = (1 << (bits - 1)) - 1
    rng = np.random.default_rng(bits * 7 + block)
    x = rng.uniform(-Q, Q, n).astype(np.float32)
    x[::block] = Q
    m = O.random_words(seed, stream, index_offset, n) & 0x7FFFFF
    sel = np.nonzero((m > 1 << 22) & (m < 3 << 21))[0]
    sel = sel[sel % block != 0]
    d = np.array([2.0 ** -25, 0.0, -2.0 ** -25])[np.arange(sel.size) % 3]
    t = m[sel].astype(np.float64) * 2.0 ** -23 + d - 1.0
    assert (t.astype(np.float32).astype(np.float64) == t).all()
    x[sel] = t.astype(np.float32)
    return x, sel, np.where(d > 0, 0, -1)


@pytest.mark.parametrize("bits", [2, 4, 8, 12, 16])
def test_sr_takes_the_exact_fraction(bits):
    # Both encoder layouts (8 elements per thread with error feedback, 16
    # without) and the stage-2 requantisation of the decoders (one rank and
    # the eight-rank 4-bit decoder, whose summed zeros plus e2 give exactly
    # these values) against the oracle and against the expected levels.
    torch, bc = need_gpu()
    n, B = 4096 * 3 + 64, 128
    x, sel, q_exp = _fraction_ties(bits, n, B, 5, 0, 0)
    p = bc.QParams(bits, B, bc.SR, seed=5)
    for ef in (False, True):
        e = np.zeros(n, np.float32)
        codes, scales, err = _run_encode(torch, bc, x, "f32", n, p, e.copy() if ef else None)
        e_ref = e.copy() if ef else None
        c_ref, s_ref = O.quantize_pack(x, O.params(bits, B, O.SR, seed=5), e_ref)
        assert codes.tobytes() == c_ref.tobytes() and np.array_equal(scales, s_ref), f"ef={ef}"
        if ef:
            assert np.array_equal(err.view(np.uint32), e_ref.view(np.uint32))
        q = codes_to_q(unpack_codes(codes, bits, n), bits)
        assert (q[sel] == q_exp).all()
    # decoders: zero codes (scale 0) from W ranks, stage-2 error = x
    for W, bin_ in ((1, bits), (8, 4)):
        if W == 8 and bits != 4:
            continue
        x2, sel2, q2_exp = _fraction_ties(bits, n, B, 9, 1, 12)
        zc, zs = O.quantize_pack(np.zeros(n, np.float32), O.params(bin_, B))
        cin = [torch.from_numpy(zc).cuda() for _ in range(W)]
        sin = [torch.from_numpy(zs.view(np.int16)).cuda() for _ in range(W)]
        e2_g = torch.from_numpy(x2.copy()).cuda()
        co, so = bc.alloc_codes(n, bc.QParams(bits, B))
        pout = bc.QParams(bits, B, bc.SR, seed=9, index_offset=12, philox_stream=1)
        bc.unpack_dequant_reduce_requant(cin, sin, n, bc.QParams(bin_, B), err2=e2_g, p_out=pout,
                                         codes_out=co, scales_out=so)
        torch.cuda.synchronize()
        e2_ref = x2.copy()
        _, c_ref, sc_ref = O.unpack_dequant_reduce_requant(
            [zc] * W, [zs] * W, n, O.params(bin_, B), True, e2_ref,
            O.params(bits, B, O.SR, seed=9, index_offset=12, philox_stream=1))
        got = co.cpu().numpy()
        assert got.tobytes() == c_ref.tobytes() and np.array_equal(so.cpu().numpy().view(np.uint16), sc_ref)
        assert np.array_equal(e2_g.cpu().numpy().view(np.uint32), e2_ref.view(np.uint32))
        q = codes_to_q(unpack_codes(got, bits, n), bits)
        assert (q[sel2] == q2_exp).all(), f"W={W}"


@pytest.mark.parametrize("bits", [2, 4, 8, 16])
def test_sr_philox_counter_carry(bits):
    # Element indices around 2^34, where the Philox counter i/4 carries into its
    # high word: the kernels share Philox products between consecutive counters
    # only while the high word stays the same, and fall back at the carry.  The
    # encoders (16 elements per thread without error feedback, 8 with it) and
    # the stochastic requantisation of the decoders (W = 3 general, W = 8
    # 4-bit 16-element layout) must give the oracle's bits on both sides.
    torch, bc = need_gpu()
    n, off = 8192, (1 << 34) - 4096 - 24
    x, e = _inputs(n, "f32", 77 + bits)
    for ef in (False, True):
        p = bc.QParams(bits, 128, bc.SR, seed=99, index_offset=off)
        codes, scales, err = _run_encode(torch, bc, x, "f32", n, p, e.copy() if ef else None)
        e_ref = e.copy() if ef else None
        c_ref, s_ref = O.quantize_pack(x, O.params(bits, 128, O.SR, seed=99, index_offset=off), e_ref)
        assert codes.tobytes() == c_ref.tobytes() and np.array_equal(scales, s_ref), f"ef={ef}"
        if ef:
            assert np.array_equal(err.view(np.uint32), e_ref.view(np.uint32))
    rng = np.random.default_rng(bits)
    for W in (3, 8):
        ins = [_random_codes(rng, n, bits, 128) for _ in range(W)]
        e2 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        e2_g = torch.from_numpy(e2.copy()).cuda()
        pout = bc.QParams(bits, 128, bc.SR, seed=5, index_offset=off, philox_stream=1)
        co, so = bc.alloc_codes(n, pout)
        bc.unpack_dequant_reduce_requant([torch.from_numpy(c).cuda() for c, _ in ins],
                                         [torch.from_numpy(s.view(np.int16)).cuda() for _, s in ins], n,
                                         bc.QParams(bits, 128), err2=e2_g, p_out=pout, codes_out=co, scales_out=so)
        torch.cuda.synchronize()
        _, c_ref, s_ref = O.unpack_dequant_reduce_requant(
            [c for c, _ in ins], [s for _, s in ins], n, O.params(bits, 128), False, e2,
            O.params(bits, 128, O.SR, seed=5, index_offset=off, philox_stream=1))
        assert co.cpu().numpy().tobytes() == c_ref.tobytes(), f"W={W}"
        assert np.array_equal(so.cpu().numpy().view(np.uint16), s_ref), f"W={W}"
        assert np.array_equal(e2_g.cpu().numpy().view(np.uint32), e2.view(np.uint32)), f"W={W}"


def _random_codes(rng, n, bits, block, scale_sigma=1e-3):
    nbytes = O.packed_bytes(n, bits, block)
    codes = rng.integers(0, 256, nbytes, dtype=np.uint8)
    s = np.abs(rng.standard_normal(O.num_blocks(n, block)) * scale_sigma).astype(np.float16)
    s[rng.integers(0, s.size, max(1, s.size // 50))] = 0.0
    return codes, s.view(np.uint16)


DEC_CASES = [(b, 0, 128, 128) for b in BITS] + [(b, b, 128, 128) for b in BITS] + \
            [(b, b, B, B) for b in (1, 4, 16) for B in (8, 32, 512, 4096)] + \
            [(8, 4, 512, 128), (8, 4, 128, 512), (8, 4, 32, 4096)]


@pytest.mark.parametrize("bin_,bout,Bin,Bout", DEC_CASES)
@pytest.mark.parametrize("W", [1, 3, 8, 9])
@pytest.mark.parametrize("mode", ["plain", "ef2", "sr_ef2"])
def test_decoder_matches_oracle(bin_, bout, Bin, Bout, W, mode):
    torch, bc = need_gpu()
    if bout == 0 and mode != "plain":
        pytest.skip("stage-2 options need requantisation")
    rng = np.random.default_rng(bin_ * 7919 + bout * 31 + W + Bin + Bout)
    for n in (5, 4096 + 8, 3 * 4096 + 77):
        ins = [_random_codes(rng, n, bin_, Bin) for _ in range(W)]
        pin = bc.QParams(bin_, Bin)
        sr = mode == "sr_ef2"
        pout = bc.QParams(bout, Bout, bc.SR if sr else bc.RTN, seed=99, index_offset=2 ** 32 + 1,
                          philox_stream=1) if bout else None
        e2 = (rng.standard_normal(n) * 1e-3).astype(np.float32) if mode != "plain" else None

        cin = [Guarded(torch, c.size, fill=c) for c, _ in ins]
        sin = [Guarded(torch, 2 * s.size, fill=s) for _, s in ins]
        sum_g = Guarded(torch, 4 * n)
        e2_g = Guarded(torch, 4 * n, fill=e2) if e2 is not None else None
        co = Guarded(torch, bc.packed_bytes(n, bout, Bout)) if bout else None
        so = Guarded(torch, 2 * bc.num_blocks(n, Bout)) if bout else None
        bc.unpack_dequant_reduce_requant(
            [c.view(torch.uint8) for c in cin], [s.view(torch.int16) for s in sin], n, pin,
            sum_out=sum_g.view(torch.float32), err2=e2_g.view(torch.float32) if e2_g else None,
            p_out=pout, codes_out=co.view(torch.uint8) if co else None,
            scales_out=so.view(torch.int16) if so else None)
        torch.cuda.synchronize()
        for g in [sum_g, e2_g, co, so] + cin + sin:
            assert g is None or g.guards_intact()

        po = O.params(bout, Bout, O.SR if sr else O.RTN, seed=99, index_offset=2 ** 32 + 1,
                      philox_stream=1) if bout else None
        e2_ref = e2.copy() if e2 is not None else None
        s_ref, c_ref, sc_ref = O.unpack_dequant_reduce_requant(
            [c for c, _ in ins], [s for _, s in ins], n, O.params(bin_, Bin), True, e2_ref, po)
        assert np.array_equal(sum_g.host(np.uint32), s_ref.view(np.uint32)), f"sum differs n={n}"
        if bout:
            assert co.host(np.uint8).tobytes() == c_ref.tobytes(), f"codes differ n={n}"
            assert np.array_equal(so.host(np.uint16), sc_ref), f"scales differ n={n}"
        if e2 is not None:
            assert np.array_equal(e2_g.host(np.uint32), e2_ref.view(np.uint32)), f"e2' differs n={n}"


@pytest.mark.parametrize("offset", [0, 4])
@pytest.mark.parametrize("sr", [False, True])
def test_decoder_w8_alignment_paths(offset, sr):
    # Eight ranks of 4-bit codes take a 16-elements-per-thread decoder when the
    # code pointers are 8-byte aligned (offset 0) and the general one when they
    # are only 4-byte aligned (offset 4); both must give the oracle's bits, with
    # and without the fp32 sum output.
    torch, bc = need_gpu()
    rng = np.random.default_rng(31 + offset + sr)
    W, B = 8, 128
    for n in (4096 * 3 + 77, 16 * 40):
        for with_sum in (False, True):
            ins = [_random_codes(rng, n, 4, B) for _ in range(W)]
            nb = bc.packed_bytes(n, 4, B)
            cin = []
            for c, _ in ins:
                buf = torch.zeros(nb + 16, dtype=torch.uint8, device="cuda")
                buf[offset:offset + nb].copy_(torch.from_numpy(c).cuda())
                cin.append(buf[offset:offset + nb])
            sin = [torch.from_numpy(sc.view(np.int16)).cuda() for _, sc in ins]
            e2 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
            e2_g = torch.from_numpy(e2.copy()).cuda()
            cob = torch.zeros(nb + 16, dtype=torch.uint8, device="cuda")
            co = cob[offset:offset + nb]
            so = torch.zeros(bc.num_blocks(n, B), dtype=torch.int16, device="cuda")
            pout = bc.QParams(4, B, bc.SR if sr else bc.RTN, seed=5, index_offset=12, philox_stream=1)
            sm, _, _ = bc.unpack_dequant_reduce_requant(cin, sin, n, bc.QParams(4, B),
                                                        sum_out=True if with_sum else None, err2=e2_g,
                                                        p_out=pout, codes_out=co, scales_out=so)
            torch.cuda.synchronize()
            e2_ref = e2.copy()
            s_ref, c_ref, sc_ref = O.unpack_dequant_reduce_requant(
                [c for c, _ in ins], [sc for _, sc in ins], n, O.params(4, B), True, e2_ref,
                O.params(4, B, O.SR if sr else O.RTN, seed=5, index_offset=12, philox_stream=1))
            tag = f"n={n} sum={with_sum}"
            assert co.cpu().numpy().tobytes() == c_ref.tobytes(), tag
            assert np.array_equal(so.cpu().numpy().view(np.uint16), sc_ref), tag
            assert np.array_equal(e2_g.cpu().numpy().view(np.uint32), e2_ref.view(np.uint32)), tag
            if with_sum:
                assert np.array_equal(sm.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), tag
            # the sum alone (no requantisation): the 16-element kernel without
            # its requantisation, or the general decoder
            sm2, _, _ = bc.unpack_dequant_reduce_requant(cin, sin, n, bc.QParams(4, B), sum_out=True)
            torch.cuda.synchronize()
            assert np.array_equal(sm2.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), tag + " sum only"


@pytest.mark.parametrize("bin_blk,bout_blk", [(32, 512), (512, 32), (16, 4096), (4096, 16)])
def test_decoder_w8_mixed_blocks(bin_blk, bout_blk):
    # Eight ranks of 4-bit codes requantised to 4 bits with a different block
    # size on each side (the 16-elements-per-thread decoder handles both).
    torch, bc = need_gpu()
    rng = np.random.default_rng(bin_blk * 3 + bout_blk)
    W = 8
    for n in (4 * 4096 + 48, 4096):
        ins = [_random_codes(rng, n, 4, bin_blk) for _ in range(W)]
        cin = [torch.from_numpy(c).cuda() for c, _ in ins]
        sin = [torch.from_numpy(sc.view(np.int16)).cuda() for _, sc in ins]
        e2 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        e2_g = torch.from_numpy(e2.copy()).cuda()
        pout = bc.QParams(4, bout_blk, bc.RTN, philox_stream=1)
        sm, co, so = bc.unpack_dequant_reduce_requant(cin, sin, n, bc.QParams(4, bin_blk), sum_out=True,
                                                      err2=e2_g, p_out=pout)
        torch.cuda.synchronize()
        e2_ref = e2.copy()
        s_ref, c_ref, sc_ref = O.unpack_dequant_reduce_requant(
            [c for c, _ in ins], [sc for _, sc in ins], n, O.params(4, bin_blk), True, e2_ref,
            O.params(4, bout_blk, philox_stream=1))
        assert np.array_equal(sm.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), f"n={n}"
        assert co.cpu().numpy().tobytes() == c_ref.tobytes(), f"n={n}"
        assert np.array_equal(so.cpu().numpy().view(np.uint16), sc_ref), f"n={n}"
        assert np.array_equal(e2_g.cpu().numpy().view(np.uint32), e2_ref.view(np.uint32)), f"n={n}"


def test_decoder_requant_without_sum_output():
    torch, bc = need_gpu()
    rng = np.random.default_rng(11)
    n, W = 2 * 4096 + 9, 4
    ins = [_random_codes(rng, n, 4, 128) for _ in range(W)]
    cin = [torch.from_numpy(c).cuda() for c, _ in ins]
    sin = [torch.from_numpy(s.view(np.int16)).cuda() for _, s in ins]
    p = bc.QParams(4, 128)
    _, co, so = bc.unpack_dequant_reduce_requant(cin, sin, n, p, sum_out=None, p_out=p)
    _, c_ref, s_ref = O.unpack_dequant_reduce_requant([c for c, _ in ins], [s for _, s in ins], n,
                                                      O.params(4, 128), False, None, O.params(4, 128))
    assert co.cpu().numpy().tobytes() == c_ref.tobytes()
    assert np.array_equal(so.cpu().numpy().view(np.uint16), s_ref)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits", BITS)
def test_roundtrip_matches_oracle(dt, bits):
    torch, bc = need_gpu()
    n = 3 * 4096 + 5
    x, e = _inputs(n, dt, bits)
    xh = x if dt == "f32" else bf16_bits_of(torch, x)
    xg = torch.from_numpy(xh if dt == "f32" else xh.view(np.int16)).cuda()
    if dt == "bf16":
        xg = xg.view(torch.bfloat16)
    eg = torch.from_numpy(e.copy()).cuda()
    p = bc.QParams(bits, 128)
    deq = bc.roundtrip(xg, p, err=eg)
    e_ref = e.copy()
    _, _, d_ref = O.roundtrip(xh, O.params(bits, 128), e_ref)
    torch.cuda.synchronize()
    assert np.array_equal(deq.cpu().numpy().view(np.uint32), d_ref.view(np.uint32))
    assert np.array_equal(eg.cpu().numpy().view(np.uint32), e_ref.view(np.uint32))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("rounding", ["rtn", "sr"])
@pytest.mark.parametrize("block", [8, 32, 128, 4096])
def test_roundtrip_without_feedback_matches_oracle(dt, bits, rounding, block):
    # Without error feedback the roundtrip runs in one pass (codes, scales and
    # fl(s*q) from the same registers) where the layout allows it (B >= 16,
    # b != 12); the result, the codes and the scales must be the oracle's.
    torch, bc = need_gpu()
    sr = rounding == "sr"
    for k, n in enumerate((3 * 4096 + 5, 16, 4096 + 40)):
        x, _ = _inputs(n, dt, bits * 17 + block + k)
        xh = x if dt == "f32" else bf16_bits_of(torch, x)
        xg = torch.from_numpy(xh if dt == "f32" else xh.view(np.int16)).cuda()
        if dt == "bf16":
            xg = xg.view(torch.bfloat16)
        p = bc.QParams(bits, block, bc.SR if sr else bc.RTN, seed=21, index_offset=8 * k + 2)
        codes, scales = bc.alloc_codes(n, p)
        deq = bc.roundtrip(xg, p, codes_tmp=codes, scales_tmp=scales)
        c_ref, s_ref, d_ref = O.roundtrip(xh, O.params(bits, block, O.SR if sr else O.RTN, seed=21,
                                                       index_offset=8 * k + 2))
        torch.cuda.synchronize()
        assert codes.cpu().numpy().tobytes() == c_ref.tobytes(), f"n={n}"
        assert np.array_equal(scales.cpu().numpy().view(np.uint16), s_ref), f"n={n}"
        assert np.array_equal(deq.cpu().numpy().view(np.uint32), d_ref.view(np.uint32)), f"n={n}"


@pytest.mark.parametrize("bits", [1, 2, 8, 16])
def test_roundtrip_in_place_all_widths(bits):
    torch, bc = need_gpu()
    n = 4096 * 2 + 19
    x, _ = _inputs(n, "f32", 91 + bits)
    xg = torch.from_numpy(x.copy()).cuda()
    p = bc.QParams(bits, 64, bc.SR, seed=4)
    bc.roundtrip(xg, p, deq_out=xg)
    _, _, d_ref = O.roundtrip(x, O.params(bits, 64, O.SR, seed=4))
    assert np.array_equal(xg.cpu().numpy().view(np.uint32), d_ref.view(np.uint32))


def test_roundtrip_in_place():
    # deq_out may alias x for fp32 (the simulate-quantization mode)
    torch, bc = need_gpu()
    n = 4096 * 2 + 3
    x, _ = _inputs(n, "f32", 77)
    xg = torch.from_numpy(x.copy()).cuda()
    p = bc.QParams(4, 128)
    bc.roundtrip(xg, p, deq_out=xg)
    _, _, d_ref = O.roundtrip(x, O.params(4, 128))
    assert np.array_equal(xg.cpu().numpy().view(np.uint32), d_ref.view(np.uint32))


def test_empty_input_is_a_no_op():
    torch, bc = need_gpu()
    x = torch.empty(0, device="cuda")
    codes, scales = bc.quantize_pack(x, bc.QParams(4, 128))
    assert codes.numel() == 0 and scales.numel() == 0


@pytest.mark.parametrize("bits", BITS)
def test_decoder_extreme_scales(bits):
    # fp16 scales 0, 2^-24 (smallest subnormal), largest subnormal, 2^-14,
    # 1.0 and 65504 with random codes: the dequantise-accumulate must stay
    # bit-exact at both ends of the fp16 range.
    torch, bc = need_gpu()
    rng = np.random.default_rng(bits)
    n, W, B = 4 * 4096 + 24, 8, 32
    special = np.array([0x0000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF], dtype=np.uint16)
    ins = []
    for _ in range(W):
        codes = rng.integers(0, 256, O.packed_bytes(n, bits, B), dtype=np.uint8)
        scales = special[rng.integers(0, special.size, O.num_blocks(n, B))]
        ins.append((codes, scales))
    cin = [torch.from_numpy(c).cuda() for c, _ in ins]
    sin = [torch.from_numpy(s.view(np.int16)).cuda() for _, s in ins]
    pin = bc.QParams(bits, B)
    sum_, co, so = bc.unpack_dequant_reduce_requant(cin, sin, n, pin, sum_out=True, p_out=pin)
    s_ref, c_ref, sc_ref = O.unpack_dequant_reduce_requant([c for c, _ in ins], [s for _, s in ins], n,
                                                           O.params(bits, B), True, None, O.params(bits, B))
    assert np.array_equal(sum_.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert co.cpu().numpy().tobytes() == c_ref.tobytes()
    assert np.array_equal(so.cpu().numpy().view(np.uint16), sc_ref)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("block", [8, 128, 4096])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_allgather_decode_matches_oracle(bits, block, out):
    torch, bc = need_gpu()
    rng = np.random.default_rng(bits * 31 + block)
    for n, mul in ((13, 1.0), (3 * 4096 + 40, 0.125), (5 * 4096 + 8, float(np.float32(1 / 3)))):
        codes, scales = _random_codes(rng, n, bits, block)
        cg = Guarded(torch, codes.size, fill=codes)
        sg = Guarded(torch, 2 * scales.size, fill=scales)
        og = Guarded(torch, (4 if out == "f32" else 2) * n)
        dst = og.view(torch.float32 if out == "f32" else torch.bfloat16)
        bc.unpack_dequant(cg.view(torch.uint8), sg.view(torch.int16), n, bc.QParams(bits, block), mul, out=dst)
        torch.cuda.synchronize()
        assert og.guards_intact()
        ref = O.unpack_dequant(codes, scales, n, O.params(bits, block), mul, O.F32 if out == "f32" else O.BF16)
        got = og.host(np.uint32 if out == "f32" else np.uint16)
        assert np.array_equal(got, ref.view(np.uint32 if out == "f32" else np.uint16)), f"n={n} mul={mul}"


# Smallest code-pointer alignment the ABI accepts per width, and the one the
# 16-element all-gather-side decode needs (twice that, 8 bytes for 12 bits);
# 16-bit codes need 16 bytes on both paths.
CODE_ALIGN = {1: 1, 2: 2, 4: 4, 8: 8, 12: 4, 16: 16}


def _dequant_case(torch, bc, rng, n, bits, block, out, mul, code_off=0, out_off=0, hadamard=0):
    """Decode random codes through the ABI with the codes placed code_off bytes
    and the output out_off bytes past an aligned address; compare every output
    element with the oracle and check that nothing outside the output moved."""
    codes, scales = _random_codes(rng, n, bits, block)
    cg = Guarded(torch, code_off + codes.size, fill=np.concatenate([np.zeros(code_off, np.uint8), codes]))
    sg = Guarded(torch, 2 * scales.size, fill=scales)
    esz = 4 if out == "f32" else 2
    og = Guarded(torch, out_off + esz * n)
    dst = og.view(torch.uint8)[out_off:].view(torch.float32 if out == "f32" else torch.bfloat16)
    bc.unpack_dequant(cg.view(torch.uint8)[code_off:], sg.view(torch.int16), n,
                      bc.QParams(bits, block, hadamard=hadamard), mul, out=dst)
    torch.cuda.synchronize()
    assert og.guards_intact()
    raw = og.host(np.uint8)
    assert (raw[:out_off] == 0xA5).all(), "bytes before the output changed"
    ref = O.unpack_dequant(codes, scales, n, O.params(bits, block, hadamard=hadamard), mul,
                           O.F32 if out == "f32" else O.BF16)
    got = raw[out_off:].view(np.uint32 if out == "f32" else np.uint16)
    assert np.array_equal(got, ref.view(np.uint32 if out == "f32" else np.uint16)), \
        f"n={n} bits={bits} block={block} code_off={code_off} out_off={out_off}"


@pytest.mark.parametrize("bits", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("path", ["wide", "narrow"])
def test_allgather_decode_many_rows_per_cta(bits, out, path):
    # 2,600 rows of 4096 elements and a ragged last row.  "wide" takes the
    # 16-element kernel (about three rows per CTA); "narrow" places the output
    # (bf16) or the codes (fp32) off that kernel's alignment, so the persistent
    # 8-element kernel decodes more than eight rows per CTA and the bf16
    # decode's four-row register ring is refilled several times and wraps
    # around the ragged row.
    torch, bc = need_gpu()
    rng = np.random.default_rng(bits + (7 if out == "bf16" else 0) + (100 if path == "narrow" else 0))
    code_off = out_off = 0
    if path == "narrow":
        if out == "bf16":
            out_off = 16
        elif bits != 16:
            code_off = CODE_ALIGN[bits]
        else:
            pytest.skip("16-bit codes into fp32 always meet the 16-element kernel's alignment")
    _dequant_case(torch, bc, rng, 2600 * 4096 + 77, bits, 128, out, float(np.float32(1 / 8)), code_off, out_off)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_allgather_decode_ragged_and_alignment_paths(bits, out):
    # Ragged sizes (inside the first piece, at a piece and a row boundary, one
    # past them), blocks from the smallest the 16-element kernel takes (16) to
    # 4096 and 8 (the 8-element kernel only); codes at the smallest accepted
    # alignment and an output 16 bytes off a 32-byte boundary (bf16) send the
    # call to the 8-element kernel.  Every path gives the oracle's bits.
    torch, bc = need_gpu()
    rng = np.random.default_rng(1000 + bits * 2 + (out == "bf16"))
    mul = float(np.float32(1 / 3))
    layouts = [(0, 0)]
    if bits != 16:
        layouts.append((CODE_ALIGN[bits], 0))
    if out == "bf16":
        layouts.append((0, 16))
    for block in (8, 16, 64, 4096):
        for n in (1, 15, 16, 17, 4096, 4096 + 16 * 5 + 7, 3 * 4096 + 1):
            for code_off, out_off in layouts:
                _dequant_case(torch, bc, rng, n, bits, block, out, mul, code_off, out_off)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("H", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_rotated_decode_paths(bits, H, out):
    # The rotated all-gather-side decode with blocks of >= 32 elements (32
    # elements per thread, the fp32 output staged through shared memory): 41
    # rows of 8192 and a ragged last row (for H = 8 and 16 ending inside a
    # thread's 32 elements), a single transform block, and codes at the
    # smallest accepted alignment or a bf16 output 16 bytes off a 32-byte
    # boundary, which take the 8-element kernel instead.
    torch, bc = need_gpu()
    rng = np.random.default_rng(3000 + bits * 10 + H + (out == "bf16"))
    block = max(H, 128)
    mul = float(np.float32(1 / 3))
    layouts = [(0, 0), (CODE_ALIGN[bits], 0)] + ([(0, 16)] if out == "bf16" else [])
    for n in (41 * 8192 + 3 * H, H):
        for code_off, out_off in layouts:
            _dequant_case(torch, bc, rng, n, bits, block, out, mul, code_off, out_off, hadamard=H)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("H,block", [(8, 8), (32, 128), (128, 128), (128, 512), (256, 4096)])
@pytest.mark.parametrize("mode", ["rtn", "sr_ef"])
def test_hadamard_encoder_and_decode_match_oracle(dt, bits, H, block, mode):
    # Walsh-Hadamard smoothing: rotated encoder (error feedback in the rotated
    # domain) and the all-gather-side decode with the inverse rotation.
    torch, bc = need_gpu()
    sr, ef = mode.startswith("sr"), mode.endswith("ef")
    for k, n in enumerate([block, 3 * 4096 + 2 * block, 6 * 4096]):
        x, e = _inputs(n, dt, seed=bits * 100 + H + k)
        xh = x if dt == "f32" else bf16_bits_of(torch, x)
        p = bc.QParams(bits, block, bc.SR if sr else bc.RTN, seed=5 + k, index_offset=4 * k, hadamard=H)
        po = O.params(bits, block, O.SR if sr else O.RTN, seed=5 + k, index_offset=4 * k, hadamard=H)
        codes, scales, err = _run_encode(torch, bc, xh, dt, n, p, e.copy() if ef else None)
        e_ref = e.copy() if ef else None
        c_ref, s_ref = O.quantize_pack(xh, po, e_ref)
        assert codes.tobytes() == c_ref.tobytes(), f"codes n={n}"
        assert np.array_equal(scales, s_ref), f"scales n={n}"
        if ef:
            assert np.array_equal(err.view(np.uint32), e_ref.view(np.uint32)), f"e' n={n}"
        for out in ("f32", "bf16"):
            dst = torch.empty(n, dtype=torch.float32 if out == "f32" else torch.bfloat16, device="cuda")
            bc.unpack_dequant(torch.from_numpy(codes).cuda(), torch.from_numpy(scales.view(np.int16)).cuda(),
                              n, p, 0.5, out=dst)
            ref = O.unpack_dequant(codes, scales, n, po, 0.5, O.F32 if out == "f32" else O.BF16)
            got = dst.view(torch.int32 if out == "f32" else torch.int16).cpu().numpy()
            assert np.array_equal(got.view(np.uint32 if out == "f32" else np.uint16),
                                  ref.view(np.uint32 if out == "f32" else np.uint16)), f"{out} n={n}"


def test_hadamard_roundtrip_matches_oracle():
    torch, bc = need_gpu()
    n = 8 * 4096
    x, e = _inputs(n, "f32", 3)
    p = bc.QParams(4, 128, hadamard=128)
    eg = torch.from_numpy(e.copy()).cuda()
    deq = bc.roundtrip(torch.from_numpy(x).cuda(), p, err=eg)
    e_ref = e.copy()
    _, _, d_ref = O.roundtrip(x, O.params(4, 128, hadamard=128), e_ref)
    assert np.array_equal(deq.cpu().numpy().view(np.uint32), d_ref.view(np.uint32))
    assert np.array_equal(eg.cpu().numpy().view(np.uint32), e_ref.view(np.uint32))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("block,rounding", [(2048, 0), (128, 1), (8, 0)])
def test_qwd_matches_oracle_over_steps(dt, bits, block, rounding):
    # Weight-difference quantisation: the sender's encoder (ref advances) and a
    # receiver's apply (ref advances, bf16 weights out), three steps in a row.
    torch, bc = need_gpu()
    rng = np.random.default_rng(bits * 10 + block)
    n = 3 * 4096 + 2 * block + 8
    w = rng.standard_normal(n).astype(np.float32)
    ref_s = torch.from_numpy(w.copy()).cuda()
    ref_r = torch.from_numpy(w.copy()).cuda()
    h_ref_s, h_ref_r = w.copy(), w.copy()
    for t in range(3):
        w = (w + np.float32(1e-3) * rng.standard_normal(n).astype(np.float32)).astype(np.float32)
        wh = w if dt == "f32" else bf16_bits_of(torch, w)
        wg = torch.from_numpy(wh if dt == "f32" else wh.view(np.int16)).cuda()
        if dt == "bf16":
            wg = wg.view(torch.bfloat16)
        p = bc.QParams(bits, block, rounding, seed=9, index_offset=t * n)
        po = O.params(bits, block, rounding, seed=9, index_offset=t * n)
        codes, scales = bc.qwd_encode(wg, ref_s, p)
        wout = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        bc.qwd_apply(codes, scales, n, p, ref_r, wout)
        torch.cuda.synchronize()
        c_ref, s_ref = O.qwd_encode(wh, h_ref_s, po)
        w_ref = O.qwd_apply(c_ref, s_ref, n, po, h_ref_r, O.BF16)
        assert codes.cpu().numpy().tobytes() == c_ref.tobytes(), f"step {t}"
        assert np.array_equal(scales.cpu().numpy().view(np.uint16), s_ref), f"step {t}"
        assert np.array_equal(ref_s.cpu().numpy().view(np.uint32), h_ref_s.view(np.uint32)), f"step {t}"
        assert np.array_equal(ref_r.cpu().numpy().view(np.uint32), h_ref_r.view(np.uint32)), f"step {t}"
        assert np.array_equal(wout.view(torch.int16).cpu().numpy().view(np.uint16), w_ref), f"step {t}"


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("wout", ["none", "f32", "bf16"])
def test_qwd_apply_ragged_and_alignment_paths(bits, wout):
    # The receiver's apply on random codes: ragged sizes, blocks 8 (the
    # 8-element kernel only), 16 and 2048, codes at the smallest accepted
    # alignment and bf16 weights 16 bytes off a 32-byte boundary (both send
    # the call to the 8-element kernel), and 2,600 rows (several rows per CTA
    # on either kernel).  The reference and the weights match the oracle bit
    # for bit and nothing outside them is written.
    torch, bc = need_gpu()
    rng = np.random.default_rng(500 + bits * 3 + len(wout))
    layouts = [(0, 0), (CODE_ALIGN[bits], 0)] + ([(0, 16)] if wout == "bf16" else [])
    cases = [(b, n) for b in (8, 16, 2048) for n in (1, 15, 17, 4096 + 16 * 3 + 5)] + [(2048, 2600 * 4096 + 77)]
    for block, n in cases:
        for code_off, out_off in layouts:
            codes, scales = _random_codes(rng, n, bits, block)
            ref0 = rng.standard_normal(n).astype(np.float32)
            cg = Guarded(torch, code_off + codes.size, fill=np.concatenate([np.zeros(code_off, np.uint8), codes]))
            sg = Guarded(torch, 2 * scales.size, fill=scales)
            rg = Guarded(torch, 4 * n, fill=ref0)
            og = None
            dst = None
            if wout != "none":
                esz = 4 if wout == "f32" else 2
                og = Guarded(torch, out_off + esz * n)
                dst = og.view(torch.uint8)[out_off:].view(torch.float32 if wout == "f32" else torch.bfloat16)
            bc.qwd_apply(cg.view(torch.uint8)[code_off:], sg.view(torch.int16), n, bc.QParams(bits, block),
                         rg.view(torch.float32), dst)
            torch.cuda.synchronize()
            h_ref = ref0.copy()
            w_ref = O.qwd_apply(codes, scales, n, O.params(bits, block), h_ref,
                                O.BF16 if wout == "bf16" else O.F32)
            tag = f"n={n} block={block} code_off={code_off} out_off={out_off}"
            assert rg.guards_intact(), tag
            assert np.array_equal(rg.host(np.uint32), h_ref.view(np.uint32)), tag
            if og is not None:
                assert og.guards_intact(), tag
                raw = og.host(np.uint8)
                assert (raw[:out_off] == 0xA5).all(), tag
                got = raw[out_off:].view(np.uint32 if wout == "f32" else np.uint16)
                assert np.array_equal(got, w_ref.view(np.uint32 if wout == "f32" else np.uint16)), tag


@pytest.mark.parametrize("wout", ["none", "f32"])
def test_qwd_apply_weight_outputs(wout):
    # The receiver's apply without a weight copy and with an fp32 one (the
    # bf16 copy is covered above); the reference advances the same way.
    torch, bc = need_gpu()
    rng = np.random.default_rng(7 + len(wout))
    n, bits, block = 2 * 4096 + 136, 4, 128
    w = rng.standard_normal(n).astype(np.float32)
    ref_s = torch.from_numpy(w.copy()).cuda()
    ref_r = torch.from_numpy(w.copy()).cuda()
    h_ref_s, h_ref_r = w.copy(), w.copy()
    w2 = (w + np.float32(1e-3) * rng.standard_normal(n).astype(np.float32)).astype(np.float32)
    p = bc.QParams(bits, block)
    po = O.params(bits, block)
    codes, scales = bc.qwd_encode(torch.from_numpy(w2).cuda(), ref_s, p)
    out = torch.empty(n, dtype=torch.float32, device="cuda") if wout == "f32" else None
    bc.qwd_apply(codes, scales, n, p, ref_r, out)
    torch.cuda.synchronize()
    c_ref, s_ref = O.qwd_encode(w2, h_ref_s, po)
    w_ref = O.qwd_apply(c_ref, s_ref, n, po, h_ref_r, O.F32)
    assert np.array_equal(ref_r.cpu().numpy().view(np.uint32), h_ref_r.view(np.uint32))
    if out is not None:
        assert np.array_equal(out.cpu().numpy().view(np.uint32), w_ref.view(np.uint32))


@pytest.mark.parametrize("bits", [2, 4, 16])
def test_decoder_maximum_ranks(bits):
    # W = 64, the largest rank count the ABI accepts (eight groups of eight in
    # the many-rank kernel), with requantisation and stage-2 error feedback.
    torch, bc = need_gpu()
    rng = np.random.default_rng(64 + bits)
    n, W, B = 2 * 4096 + 72, 64, 128
    ins = [_random_codes(rng, n, bits, B) for _ in range(W)]
    cin = [torch.from_numpy(c).cuda() for c, _ in ins]
    sin = [torch.from_numpy(s.view(np.int16)).cuda() for _, s in ins]
    e2 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    e2g = torch.from_numpy(e2.copy()).cuda()
    p = bc.QParams(bits, B, bc.SR, seed=3, philox_stream=1)
    sum_, co, so = bc.unpack_dequant_reduce_requant(cin, sin, n, bc.QParams(bits, B), sum_out=True, err2=e2g,
                                                    p_out=p)
    torch.cuda.synchronize()
    e2_ref = e2.copy()
    s_ref, c_ref, sc_ref = O.unpack_dequant_reduce_requant(
        [c for c, _ in ins], [s for _, s in ins], n, O.params(bits, B), True, e2_ref,
        O.params(bits, B, O.SR, seed=3, philox_stream=1))
    assert np.array_equal(sum_.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert co.cpu().numpy().tobytes() == c_ref.tobytes()
    assert np.array_equal(so.cpu().numpy().view(np.uint16), sc_ref)
    assert np.array_equal(e2g.cpu().numpy().view(np.uint32), e2_ref.view(np.uint32))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("W", [1, 2, 3, 4, 8, 64])
def test_sum_ranks_matches_oracle(dt, W):
    # The full-precision local reduce: rank-ordered fp32 sum, bit for bit,
    # with values that tie (2^24 + 1) and zeros of both signs mixed in.
    torch, bc = need_gpu()
    rng = np.random.default_rng(W * 7 + (dt == "bf16"))
    for n in (1, 13, 8 * 4096 + 5):
        xs = []
        for w in range(W):
            x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
            x[rng.integers(0, n, max(1, n // 50))] = np.float32(2.0 ** 24)
            x[rng.integers(0, n, max(1, n // 50))] = 1.0
            x[rng.integers(0, n, max(1, n // 50))] = -0.0
            xs.append(x if dt == "f32" else bf16_bits_of(torch, x))
        ref = O.sum_ranks(xs)
        dev = [torch.from_numpy(x if dt == "f32" else x.view(np.int16)).cuda() for x in xs]
        if dt == "bf16":
            dev = [d.view(torch.bfloat16) for d in dev]
        out = Guarded(torch, 4 * n)
        bc.sum_ranks(dev, out=out.view(torch.float32))
        torch.cuda.synchronize()
        assert out.guards_intact()
        assert np.array_equal(out.host(np.float32).view(np.uint32), ref.view(np.uint32)), f"n={n}"
