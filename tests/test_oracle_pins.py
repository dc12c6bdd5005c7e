"""Pins of the CPU oracle to facts that do not come from the oracle itself.

The pages print no worked numeric example, so the pins are: blocks worked by
hand from the definitions (derivations inline), library routines (numpy's
binary16 casts and packbits, cuRAND's host Philox4x32-10 generator), closed
forms and invariants (the round-to-nearest error bound, exact error feedback,
the telescoping error-feedback sum, unbiased stochastic rounding), and special
cases (zero blocks, saturation, subnormal scales, rank order of the sum).

Definitions come from the bitscom README (Aerithy/bitscom), "Implemented
Features" (bitwidths 1/2/4/8/12/16, quantize/dequantize, bit-packing,
stochastic rounding, blockwise quantisation with per-block FP16 scales,
all-to-all -> local reduce -> all-gather, first-stage error feedback) and
"Backend Registration Options" (stage2_error_feedback / ef21_plus).
"""
import ctypes
import os

import numpy as np
import pytest

from codec_util import codes_to_q, pack_codes, qmax, scales_f64, unpack_codes

HAND_X = np.array([0.5, -1.0, 0.25, 2.0, -0.75, 0.0, 1.5, -2.0], dtype=np.float32)

# Hand-worked 8-element blocks (B = 8, round half to even, no error feedback).
#   b=4 : Qmax 7, absmax 2, 2/7 = 0.2857142...; fp16 spacing in [0.25, 0.5) is
#         2^-12, 0.2857142/2^-12 = 1170.29 -> 1170*2^-12 = 0.28564453125,
#         exponent field 13, mantissa 146 -> 0x3492.  v/s = 1.7504, -3.5009,
#         0.8752, 7.0017, -2.6256, 0, 5.2513, -7.0017 -> q = 2,-4,1,7,-3,0,5,-7,
#         u = q+8 = 10,4,9,15,5,8,13,1, nibbles LSB first -> 4a f9 85 1d.
#   b=2 : Qmax 1, s = 2.0 (0x4000); v/s = .25,-.5,.125,1,-.375,0,.75,-1; -0.5 is
#         a tie -> even 0; q = 0,0,0,1,0,0,1,-1, u = 2,2,2,3,2,2,3,1 -> ea 7a.
#   b=8 : 2/127 = 0.015748 lies in [2^-6, 2^-5), spacing 2^-16 -> 1032*2^-16 =
#         0.0157470703125 = 0x2408; q = 32,-64,16,127,-48,0,95,-127,
#         u = q+128 -> a0 40 90 ff 50 80 df 01.
#   b=12: 2/2047 = 9.7704e-4 -> 1025*2^-20 = 0x1401; v/s = 511.5004 -> 512,
#         -1023.0009, 255.75 -> 256, 2046.0018, -767.25, 0, 1534.5014 -> 1535,
#         -2046 ; u = q+2048 = a00 401 900 ffe 501 800 dff 002 (hex), 12 bits
#         each LSB first -> 00 1a 40 00 e9 ff 01 05 80 ff 2d 00.
#   b=16: 2/32767 = 6.1037e-5 rounds down to 2^-14 = 0x0400; 2/s = 32768 is
#         clamped to 32767 (the clamp case): u = a000 4000 9000 ffff 5000 8000
#         e000 0001 -> little-endian bytes below.
#   b=1 : sum|v| = 8 (exact in any order), mean 1 -> s = 1.0 = 0x3c00; signs
#         (v >= 0) = 1,0,1,1,0,1,1,0 -> 0x6d.
HAND = {
    1: (0x3C00, "6d"),
    2: (0x4000, "ea7a"),
    4: (0x3492, "4af9851d"),
    8: (0x2408, "a04090ff5080df01"),
    12: (0x1401, "001a4000e9ff010580ff2d00"),
    16: (0x0400, "00a000400090ffff0050008000e00100"),
}
# Error feedback e' = v - s*q of the same blocks (b=4: s = 0.28564453125).
HAND_ERR = {
    1: [-0.5, 0.0, -0.75, 1.0, 0.25, -1.0, 0.5, -1.0],
    4: [0.5 - 2 * 0.28564453125, -1.0 + 4 * 0.28564453125, 0.25 - 0.28564453125,
        2.0 - 7 * 0.28564453125, -0.75 + 3 * 0.28564453125, 0.0,
        1.5 - 5 * 0.28564453125, -2.0 + 7 * 0.28564453125],
    16: [0, 0, 0, 2.0 - 32767 * 2.0 ** -14, 0, 0, 0, -2.0 + 32767 * 2.0 ** -14],
}


@pytest.mark.parametrize("bits", [1, 2, 4, 8, 12, 16])
def test_hand_blocks(orc, bits):
    codes, scales = orc.quantize_pack(HAND_X, orc.params(bits, 8))
    assert int(scales[0]) == HAND[bits][0]
    assert codes.tobytes().hex() == HAND[bits][1]


@pytest.mark.parametrize("bits", sorted(HAND_ERR))
def test_hand_block_error_feedback(orc, bits):
    err = np.zeros(8, np.float32)
    orc.quantize_pack(HAND_X, orc.params(bits, 8), err)
    np.testing.assert_array_equal(err.astype(np.float64), np.array(HAND_ERR[bits]))


def test_hand_block_with_incoming_error(orc):
    # v = g + e: g = 0 and e = HAND_X gives the b=4 hand block again, and the new
    # error replaces the old one.
    err = HAND_X.copy()
    codes, scales = orc.quantize_pack(np.zeros(8, np.float32), orc.params(4, 8), err)
    assert int(scales[0]) == 0x3492 and codes.tobytes().hex() == "4af9851d"
    np.testing.assert_array_equal(err.astype(np.float64), np.array(HAND_ERR[4]))


def test_feedback_rounds_the_product_separately(orc):
    # b = 16: v = 32798.998046875 (fp32), absmax/32767 = 1.0009765 -> s = 1 +
    # 2^-10 (0x3c01), t = 32766.99999 -> q = 32767.  s*q = 32798.9990234375 needs
    # 25 bits, so fl(s*q) = 32798.998046875 = v and e' = fl(v - fl(s*q)) = 0; a
    # fused multiply-add would give v - s*q = -2^-10 instead.
    x = np.zeros(8, np.float32)
    x[0] = 32798.998046875
    err = np.zeros(8, np.float32)
    codes, scales = orc.quantize_pack(x, orc.params(16, 8), err)
    assert int(scales[0]) == 0x3C01
    assert codes_to_q(unpack_codes(codes, 16, 8), 16)[0] == 32767
    assert err[0] == 0.0


def test_ties_round_to_even(orc):
    # absmax 7, b=4 -> s = 7/7 = 1 exactly, so v/s = v; halves go to the even
    # neighbour: 0.5->0, 1.5->2, 2.5->2, -0.5->0, -1.5->-2, -2.5->-2, 3.5->4.
    x = np.array([7, .5, 1.5, 2.5, -.5, -1.5, -2.5, 3.5], dtype=np.float32)
    codes, scales = orc.quantize_pack(x, orc.params(4, 8))
    assert int(scales[0]) == 0x3C00
    q = codes_to_q(unpack_codes(codes, 4, 8), 4)
    assert q.tolist() == [7, 0, 2, 2, 0, -2, -2, 4]


@pytest.mark.parametrize("bits", [2, 4, 8, 12, 16])
def test_zero_block(orc, bits):
    # absmax 0 -> s = +0, every q = 0, code 2^(b-1), e' = v = g + e.
    # (-0) + (-0) = -0 keeps the sign; (-0) + (+0) = +0 under round to nearest.
    x = np.zeros(8, np.float32)
    x[3] = -0.0
    x[4] = -0.0
    err = np.zeros(8, np.float32)
    err[3] = -0.0
    codes, scales = orc.quantize_pack(x, orc.params(bits, 8), err)
    assert int(scales[0]) == 0
    assert (unpack_codes(codes, bits, 8) == (1 << (bits - 1))).all()
    assert np.signbit(err).tolist() == [False, False, False, True, False, False, False, False]
    assert (err == 0).all()


def test_underflowing_scale_is_zero(orc):
    # absmax/Qmax below half the smallest fp16 subnormal (2^-25) -> s = 0 -> q = 0.
    x = np.full(8, 2.0 ** -26 * 7, dtype=np.float32)
    codes, scales = orc.quantize_pack(x, orc.params(4, 8))
    assert int(scales[0]) == 0
    assert (unpack_codes(codes, 4, 8) == 8).all()


def test_subnormal_scale_kept(orc):
    # absmax/Qmax = 3 * 2^-24 -> fp16 subnormal 0x0003, no flush to zero.
    x = np.zeros(8, np.float32)
    x[0] = 3 * 2.0 ** -24 * 7
    x[1] = -2 * 2.0 ** -24
    codes, scales = orc.quantize_pack(x, orc.params(4, 8))
    assert int(scales[0]) == 0x0003
    q = codes_to_q(unpack_codes(codes, 4, 8), 4)
    assert q[0] == 7 and q[1] == -1          # -2/3 -> -0.667 -> -1


def test_scale_saturates(orc):
    # absmax/Qmax = 1e6/7 > 65504 -> s clamped to 65504 (0x7bff); q clamps too.
    x = np.array([1e6, -1e6, 65504 * 3.4, 0, 0, 0, 0, 65504.0], dtype=np.float32)
    codes, scales = orc.quantize_pack(x, orc.params(4, 8))
    assert int(scales[0]) == 0x7BFF
    q = codes_to_q(unpack_codes(codes, 4, 8), 4)
    assert q.tolist() == [7, -7, 3, 0, 0, 0, 0, 1]


def test_one_bit_signed_zero_and_mean(orc):
    # +0 and -0 both code as +1; the scale is the mean over the block.
    x = np.array([-0.0, 0.0, -3.0, 1.0, 0.0, 0.0, 0.0, 0.0], dtype=np.float32)
    codes, scales = orc.quantize_pack(x, orc.params(1, 8))
    assert int(scales[0]) == 0x3800          # 4/8 = 0.5: exponent field 14
    assert unpack_codes(codes, 1, 8).tolist() == [1, 1, 0, 1, 1, 1, 1, 1]


def test_one_bit_tree_order(orc):
    # B = 4096, b = 1: x[0] = 1 + 2^-11 - 2^-23 (odd last mantissa bit) and
    # 4095 copies of 2^-24 (half an ulp of x[0]).
    # Contiguous-halves tree: the first pair rounds x[0] + 2^-24 up to the even
    # neighbour 1 + 2^-11; every other partial sum is an exact multiple of
    # 2^-23, so the total is 1 + 2^-11 + 2047*2^-23 and the mean (/4096) is
    # 2^-12 * (1 + 0.000732), above the fp16 midpoint 2^-12 * (1 + 2^-11):
    # s rounds up to 2^-12 * (1 + 2^-10) = 0x0c01.
    # A left-to-right fold would stop at 1 + 2^-11 (each later + 2^-24 is a tie
    # that keeps the even value), land exactly on the midpoint and give 0x0c00.
    x = np.full(4096, 2.0 ** -24, dtype=np.float32)
    x[0] = 1 + 2.0 ** -11 - 2.0 ** -23
    codes, scales = orc.quantize_pack(x, orc.params(1, 4096))
    assert int(scales[0]) == 0x0C01
    assert (unpack_codes(codes, 1, 4096) == 1).all()


def test_one_bit_tail_mean_divides_by_valid(orc):
    # n = 3 in a block of 8: the mean divides by 3, not 8.
    x = np.array([3.0, -3.0, 3.0], dtype=np.float32)
    codes, scales = orc.quantize_pack(x, orc.params(1, 8))
    assert int(scales[0]) == 0x4200          # 3.0
    assert unpack_codes(codes, 1, 8).tolist() == [1, 0, 1, 1, 1, 1, 1, 1]


def test_tail_block_hand_worked(orc):
    # n = 5 in a block of 8 (b = 4): the first five values of the hand-worked
    # 4-bit block.  The tail is zero-padded: absmax 2 -> s = fp16(2/7) (0x3492),
    # q = [2, -4, 1, 7, -3] and three padding codes of q = 0 (offset code 8):
    # u = [10, 4, 9, 15, 5, 8, 8, 8] -> bytes 4a f9 85 88.
    x = np.array([0.5, -1.0, 0.25, 2.0, -0.75], dtype=np.float32)
    e = np.zeros(5, np.float32)
    codes, scales = orc.quantize_pack(x, orc.params(4, 8), e)
    assert scales.tolist() == [0x3492]
    assert codes.tobytes() == bytes([0x4A, 0xF9, 0x85, 0x88])
    assert e.tolist() == [-0.0712890625, 0.142578125, -0.03564453125, 0.00048828125, 0.10693359375]


@pytest.mark.parametrize("bits", [2, 4, 8, 12, 16])
@pytest.mark.parametrize("rounding", [0, 1])
def test_tail_block_equals_zero_padded_block(orc, bits, rounding):
    # The reading for n mod B != 0: the last block behaves as if zero-padded
    # to B elements (b >= 2).  So encoding n elements must give the same codes,
    # scales and error as encoding the padded array, for every element < n.
    rng = np.random.default_rng(bits + 10 * rounding)
    B, n = 64, 5 * 64 + 23
    x = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    xp = np.concatenate([x, np.zeros(64 - 23, np.float32)])
    p = orc.params(bits, B, rounding, seed=3)
    e, ep = np.zeros(n, np.float32), np.zeros(xp.size, np.float32)
    c, sc = orc.quantize_pack(x, p, e)
    cp, scp = orc.quantize_pack(xp, p, ep)
    assert c.tobytes() == cp.tobytes() and np.array_equal(sc, scp)
    assert np.array_equal(e.view(np.uint32), ep[:n].view(np.uint32))


def test_one_bit_ignores_stochastic_rounding(orc):
    # The reading for b = 1 with stochastic rounding: plain sign, as without it.
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(1000) * 1e-3).astype(np.float32)
    a = orc.quantize_pack(x, orc.params(1, 128, orc.RTN), np.zeros(1000, np.float32))
    b = orc.quantize_pack(x, orc.params(1, 128, orc.SR, seed=5), np.zeros(1000, np.float32))
    assert a[0].tobytes() == b[0].tobytes() and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("bits", [1, 2, 4, 8, 12, 16])
def test_packing_matches_numpy_packbits(orc, bits):
    # Build blocks whose codes are known without the oracle: s = 2^-3 (exact in
    # fp16), v = s*q with max |q| = Qmax, so absmax/Qmax = s exactly and v/s = q.
    rng = np.random.default_rng(bits)
    B, nb = 32, 16
    if bits == 1:
        q = rng.choice([-1, 1], size=(nb, B))
        mag = np.full((nb, B), 0.125)
        v = (q * mag).astype(np.float32)
        u = (q + 1) // 2
    else:
        Q = qmax(bits)
        q = rng.integers(-Q, Q + 1, size=(nb, B))
        q[:, 0] = Q
        v = (q * 0.125).astype(np.float32)
        u = q + (1 << (bits - 1))
    codes, scales = orc.quantize_pack(v.reshape(-1), orc.params(bits, B))
    assert (scales == 0x3000).all()          # 0.125
    expect = pack_codes(u.reshape(-1), bits)
    assert codes.tobytes() == expect.tobytes()


def test_f16_to_f32_exhaustive(orc):
    L = orc.lib()
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = np.array([L.orc_f16_to_f32(int(v)) for v in h], dtype=np.float32)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_bf16_to_f32_exhaustive(orc):
    torch = pytest.importorskip("torch")
    L = orc.lib()
    h = np.arange(65536, dtype=np.int64)
    ref = torch.tensor(h.astype(np.int32).astype(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([L.orc_bf16_to_f32(int(v)) for v in h], dtype=np.float32)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32))


def test_f32_to_f16_random_and_boundaries(orc):
    # Random bit patterns plus every pattern near the subnormal, normal and
    # overflow boundaries of binary16; the exhaustive sweep is a separate test.
    rng = np.random.default_rng(0)
    pats = [rng.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)]
    for e in (102, 103, 112, 113, 142, 143):
        base = np.uint32(e << 23)
        pats.append(base + np.arange(0, 1 << 23, 97, dtype=np.uint32))
    u = np.concatenate(pats)
    u = np.concatenate([u, u | np.uint32(0x80000000)])
    x = u.view(np.float32)
    x = x[~np.isnan(x)]
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16_bits(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [hex(int(x.view(np.uint32)[i])) for i in bad[:5]]


def test_host_division_is_correctly_rounded():
    # The oracle divides in IEEE binary32.  Pin that the host's single division
    # is correctly rounded: a binary64 quotient rounded to binary32 is the
    # correctly rounded binary32 quotient (double rounding is innocuous for
    # division when 53 >= 2*24 + 2, Figueroa 1995).
    rng = np.random.default_rng(1)
    a = (rng.standard_normal(1 << 20) * 10.0 ** rng.uniform(-30, 30, 1 << 20)).astype(np.float32)
    b = np.float32(2.0) ** rng.integers(-24, 16, 1 << 20).astype(np.float32)
    b = (b * rng.integers(1024, 2048, 1 << 20).astype(np.float32) / np.float32(1024)).astype(np.float32)
    with np.errstate(all="ignore"):
        got = a / b
        ref = (a.astype(np.float64) / b.astype(np.float64)).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def _curand_words(seed: int, n: int) -> np.ndarray:
    path = None
    for d in (os.environ.get("CUDA_HOME", "/usr/local/cuda"), "/usr/local/cuda"):
        for name in ("libcurand.so", "libcurand.so.10"):
            p = os.path.join(d, "lib64", name)
            if os.path.exists(p):
                path = p
                break
        if path:
            break
    if path is None:
        pytest.skip("cuRAND host library not found")
    lib = ctypes.CDLL(path)
    gen = ctypes.c_void_p()
    CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out


@pytest.mark.parametrize("seed", [0, 42, 0x123456789ABCDEF0])
def test_philox_matches_curand_host_generator(orc, seed):
    # cuRAND's host Philox4x32-10 generator, asked for 2^17 words, returns word
    # k = Philox(counter = (0, 0, k/4, 0), key = (seed low, seed high))[k mod 4]
    # (layout fitted once by matching outputs; a library run, not its code).
    n = 1 << 17
    ref = _curand_words(seed, n)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for g in list(range(0, 64)) + list(range(4090, 4100)) + [n // 4 - 1]:
        got = orc.philox4x32_10([0, 0, g, 0], key)
        assert got.tolist() == ref[4 * g: 4 * g + 4].tolist(), g


def test_random_word_uses_counter_layout(orc):
    # Element i takes word i mod 4 of Philox(counter = (i/4 low, i/4 high,
    # stream, 0)); checked through the Philox function pinned above.
    for seed, stream, i in [(5, 0, 0), (5, 0, 7), (5, 1, 12345), (2 ** 40 + 3, 1, 2 ** 35 + 2)]:
        g = i >> 2
        out = orc.philox4x32_10([g & 0xFFFFFFFF, g >> 32, stream, 0],
                                [seed & 0xFFFFFFFF, seed >> 32])
        assert orc.random_word(seed, stream, i) == int(out[i & 3])


def test_stochastic_rounding_words_are_uniform(orc):
    # Chi-square over 256 bins of 10^7 consecutive elements' words, for two
    # seeds and both Philox streams: the top 8 of the 23 bits that form u and
    # the lowest 8 bits.  255 degrees of freedom (mean 255, sd 22.6); the bound
    # is 6 sd above the mean.
    bound = 255 + 6 * np.sqrt(2 * 255)
    for seed, stream in ((42, 0), (7, 1)):
        w = orc.random_words(seed, stream, 12345, 10_000_000)
        for bins in ((w & 0x7FFFFF) >> 15, w & 0xFF):
            counts = np.bincount(bins.astype(np.int64), minlength=256)
            e = w.size / 256
            chi2 = float(((counts - e) ** 2 / e).sum())
            assert chi2 < bound, (seed, stream, chi2)


def _blocks(rng, kind, n):
    if kind == "normal":
        return rng.standard_normal(n).astype(np.float32)
    if kind == "student":
        return (rng.standard_t(3, n) * 1e-3).astype(np.float32)
    if kind == "laplace":
        return rng.laplace(0, 1e-3, n).astype(np.float32)
    x = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    m = rng.random(n) < 0.01
    x[m] *= 100
    return x


@pytest.mark.parametrize("bits", [2, 4, 8, 12, 16])
@pytest.mark.parametrize("block", [8, 32, 128, 4096])
@pytest.mark.parametrize("kind", ["normal", "student", "laplace", "outliers"])
def test_rtn_error_bound_and_exact_feedback(orc, bits, block, kind):
    # |v - s*q| <= s/2 + 2^-24 |v| for every element whose level is not clamped
    # (the second term is the fp32 rounding of t = v/s before rint); for b <= 8
    # with a normal fp16 scale clamping never breaks it (Qmax*(1 + 2^-11) <
    # Qmax + 1/2), but a subnormal scale can be far below absmax/Qmax and then
    # the clamp binds even at b = 8.  With error feedback, e' + s*q == v exactly for
    # b <= 8 (s*q is exact and v - s*q is exact by Sterbenz when q != 0; when
    # q == 0, e' = v).
    rng = np.random.default_rng(bits * 7 + block)
    n = 8192
    v = _blocks(rng, kind, n)
    err = np.zeros(n, np.float32)
    codes, scales = orc.quantize_pack(v, orc.params(bits, block), err)
    q = codes_to_q(unpack_codes(codes, bits, n), bits).astype(np.float64)
    s = np.repeat(scales_f64(scales), block)[:n]
    resid = np.abs(v.astype(np.float64) - s * q)
    inside = np.abs(q) < qmax(bits)
    if bits <= 8:
        inside |= s >= 2.0 ** -14
    # a block whose absmax/Qmax underflows fp16 has s = 0 and every q = 0
    assert (q[s == 0] == 0).all()
    inside &= s > 0
    bound = s / 2 + 2.0 ** -24 * np.abs(v.astype(np.float64))
    assert (resid[inside] <= bound[inside]).all()
    assert (np.abs(q) <= qmax(bits)).all()
    if bits <= 8:
        np.testing.assert_array_equal(err.astype(np.float64) + s * q, v.astype(np.float64))


def test_sr_unbiased_over_seeds(orc):
    # Mean of the stochastic level over 10^5 seeds equals t = v/s (bias below
    # 2^-23 of a quantum), within 5 sigma / sqrt(10^5).
    x = np.array([0.3, -1.1, 2.0, 0.05, -0.77, 1.234, -2.0, 0.5], dtype=np.float32)
    N = 100_000
    acc = np.zeros(8, np.float64)
    sq = np.zeros(8, np.float64)
    L = orc.lib()
    codes = np.zeros(4, np.uint8)
    scales = np.zeros(1, np.uint16)
    p = orc.params(4, 8, orc.SR)
    for seed in range(N):
        p.seed = seed
        L.orc_quantize_pack(x.ctypes.data, 0, 8, None, ctypes.byref(p),
                            codes.ctypes.data, scales.ctypes.data)
        q = codes_to_q(unpack_codes(codes, 4, 8), 4)
        acc += q
        sq += q * q
    s = float(scales_f64(scales)[0])
    t = (x / np.float32(s)).astype(np.float64)
    mean = acc / N
    frac = t - np.floor(t)
    sigma = np.sqrt(frac * (1 - frac) / N) + 1e-12
    free = np.abs(t) <= 7                      # |t| > Qmax is clamped to +-Qmax
    assert (free.sum() == 6) and (mean[~free] == np.sign(t[~free]) * 7).all()
    assert (np.abs(mean - t)[free] <= 5 * sigma[free] + 2.0 ** -23).all(), (mean, t)
    # every level is floor(t) or floor(t) + 1: the second moment matches
    m2 = np.floor(t) ** 2 * (1 - frac) + (np.floor(t) + 1) ** 2 * frac
    assert (np.abs(sq / N - m2)[free] <= 10 * np.sqrt(1.0 / N) * (np.abs(t[free]) + 1) ** 2).all()


def test_sr_levels_are_neighbours_and_seed_dependent(orc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(4096).astype(np.float32)
    c1, s1 = orc.quantize_pack(x, orc.params(4, 128, orc.SR, seed=1))
    c2, s2 = orc.quantize_pack(x, orc.params(4, 128, orc.SR, seed=2))
    assert (s1 == s2).all()
    assert c1.tobytes() != c2.tobytes()
    s = np.repeat(scales_f64(s1), 128)
    t = x.astype(np.float64) / s
    q = codes_to_q(unpack_codes(c1, 4, 4096), 4)
    lo = np.clip(np.floor(t), -7, 7)
    hi = np.clip(np.floor(t) + 1, -7, 7)
    assert ((q == lo) | (q == hi)).all()


@pytest.mark.parametrize("absmax,tiny,q_expected", [
    (7.0, 2.0 ** -149, 1),      # s = 1: t = 2^-149 > 0 = u
    (7.0, -2.0 ** -149, 0),     # floor(t) = -1, t - floor(t) = 1 - 2^-149 > 0 = u
    (7.0, 0.0, 0),
    (7.0, -0.0, 0),
    (10.5, 2.0 ** -149, 1),     # s = 1.5: 2^-149 / 1.5 rounds up to 2^-149
    (14.0, 2.0 ** -149, 0),     # s = 2: exactly 2^-150, a tie, rounds to even 0
    (21.0, 2.0 ** -149, 0),     # s = 3: a third of the smallest subnormal rounds to 0
])
def test_sr_tiny_quotient_where_u_is_zero(orc, absmax, tiny, q_expected):
    # u = 0 exactly where the low 23 bits of the element's Philox word are 0;
    # there stochastic rounding sends t to floor(t) + 1 iff t - floor(t) > 0,
    # so the sign and zeroness of the correctly rounded quotient decide q.
    words = orc.random_words(11, 0, 0, 1 << 24)
    h = int(np.nonzero((words & 0x7FFFFF) == 0)[0][0])
    x = np.array([absmax, tiny, 0, 0, 0, 0, 0, 0], np.float32)
    codes, scales = orc.quantize_pack(x, orc.params(4, 8, orc.SR, seed=11, index_offset=h - 1))
    assert scales[0] == np.float16(absmax / 7).view(np.uint16)
    q = codes_to_q(unpack_codes(codes, 4, 8), 4)
    assert q[0] == 7 and q[1] == q_expected


def test_sr_compares_the_exact_fraction(orc):
    # For -1/2 < t < 0 the fraction t - floor(t) = 1 + t can need more bits
    # than fp32 holds; stochastic rounding compares u with the exact fraction.
    # With u in (1/2, 3/4) and t = u + 2^-25 - 1 (in (-1/2, -1/4), a multiple
    # of 2^-25), u < 1 + t, so t rounds up to 0 -- although 1 + t rounded to
    # fp32 is a tie that goes to the even neighbour u itself.  t = u - 1 and
    # t = u - 2^-25 - 1 stay at -1.  Scale 1 (absmax 1, 2-bit: Qmax = 1).
    words = orc.random_words(5, 0, 0, 256)
    m = words & 0x7FFFFF
    idx = [int(i) for i in np.nonzero((m > 1 << 22) & (m < 3 << 21))[0][:3]]
    assert len(idx) == 3
    for h in idx:
        u = float(words[h] & 0x7FFFFF) * 2.0 ** -23
        for delta, q_expected in ((2.0 ** -25, 0), (0.0, -1), (-2.0 ** -25, -1)):
            t = u + delta - 1.0
            assert float(np.float32(t)) == t
            x = np.array([1.0, t, 0, 0, 0, 0, 0, 0], np.float32)
            codes, scales = orc.quantize_pack(x, orc.params(2, 8, orc.SR, seed=5, index_offset=h - 1))
            assert scales[0] == np.float16(1.0).view(np.uint16)
            q = codes_to_q(unpack_codes(codes, 2, 8), 2)
            assert q[1] == q_expected, (h, u, delta)


@pytest.mark.parametrize("bits,rounding", [(2, 1), (4, 0), (8, 1), (1, 0)])
def test_error_feedback_telescopes(orc, bits, rounding):
    # Over T steps with error feedback, sum_t s_t*q_t = sum_t g_t - e_T + (the
    # fp32 roundings of g_t + e_t), so the transmitted running sum stays within
    # one quantum of the true running sum.
    # Slack: the roundings of fl(g + e) and of fl(v - s*q), each measured in
    # binary64 (s*q is exact there).  The identity sent = true - e_T (+ slack)
    # holds for every bit width; the one-quantum bound |e_T| <= s_T/2 (round to
    # nearest) or s_T (stochastic) holds for b >= 2.
    rng = np.random.default_rng(bits)
    n, B, T = 4096, 64, 20
    err = np.zeros(n, np.float32)
    sent = np.zeros(n, np.float64)
    true = np.zeros(n, np.float64)
    slack = np.zeros(n, np.float64)
    for t in range(T):
        g = (rng.standard_t(3, n) * 1e-3).astype(np.float32)
        v32 = (g + err).astype(np.float32)
        slack += np.abs(g.astype(np.float64) + err.astype(np.float64) - v32.astype(np.float64))
        codes, scales = orc.quantize_pack(g, orc.params(bits, B, rounding, seed=42, index_offset=t * n), err)
        q = codes_to_q(unpack_codes(codes, bits, n), bits).astype(np.float64)
        s = np.repeat(scales_f64(scales), B)
        d = s * q
        slack += np.abs(v32.astype(np.float64) - d - err.astype(np.float64))
        sent += d
        true += g.astype(np.float64)
    e_T = err.astype(np.float64)
    assert (np.abs(sent - (true - e_T)) <= slack * (1 + 1e-9) + 1e-30).all()
    if bits >= 2:
        assert (np.abs(e_T) <= s * (0.5 if rounding == 0 else 1.0)).all()
        assert (np.abs(sent - true) <= s * (0.5 if rounding == 0 else 1.0) + slack * (1 + 1e-9)).all()


# ---- decoder --------------------------------------------------------------

def test_single_rank_decoder_is_dequantisation(orc):
    codes, scales = orc.quantize_pack(HAND_X, orc.params(4, 8))
    s = 0.28564453125
    deq, _, _ = orc.unpack_dequant_reduce_requant([codes], [scales], 8, orc.params(4, 8))
    np.testing.assert_array_equal(deq.astype(np.float64), np.array([2, -4, 1, 7, -3, 0, 5, -7]) * s)


def _one_element_block(orc, absmax, value, bits=8):
    x = np.zeros(8, np.float32)
    x[1] = absmax
    x[0] = value
    return orc.quantize_pack(x, orc.params(bits, 8))


def test_reduce_is_in_rank_order(orc):
    # Rank 0 sends d = 1.0 (s = 0.125 from absmax 15.875 = 127 * 0.125, q = 8),
    # ranks 1 and 2 send d = 2^-24 (s = 2^-24, the smallest fp16 subnormal, q=1).
    # In rank order (1 + 2^-24) + 2^-24 = 1.0 (each add is a tie to even); the
    # reverse order would give 2^-23 + 1 = 1 + 2^-23.
    c0, s0 = _one_element_block(orc, 15.875, 1.0)
    c1, s1 = _one_element_block(orc, 127 * 2.0 ** -24, 2.0 ** -24)
    assert int(s0[0]) == 0x3000 and int(s1[0]) == 0x0001
    p = orc.params(8, 8)
    fwd, _, _ = orc.unpack_dequant_reduce_requant([c0, c1, c1], [s0, s1, s1], 8, p)
    rev, _, _ = orc.unpack_dequant_reduce_requant([c1, c1, c0], [s1, s1, s0], 8, p)
    assert fwd[0] == np.float32(1.0)
    assert rev[0] == np.float32(1.0 + 2.0 ** -23)


def test_reduce_keeps_negative_zero(orc):
    # b = 1 with an underflowing mean: s = 0 and q = -1 -> d = -0.  The sum of
    # two such ranks is -0, which a sum seeded with +0 would turn into +0.
    x = np.full(8, -1e-10, np.float32)
    c, s = orc.quantize_pack(x, orc.params(1, 8))
    assert int(s[0]) == 0
    out, _, _ = orc.unpack_dequant_reduce_requant([c, c], [s, s], 8, orc.params(1, 8))
    assert np.signbit(out).all()


def test_two_rank_sum_is_symmetric(orc):
    rng = np.random.default_rng(5)
    a = rng.standard_normal(1024).astype(np.float32)
    b = rng.standard_normal(1024).astype(np.float32)
    p = orc.params(4, 128)
    ca, sa = orc.quantize_pack(a, p)
    cb, sb = orc.quantize_pack(b, p)
    ab, _, _ = orc.unpack_dequant_reduce_requant([ca, cb], [sa, sb], 1024, p)
    ba, _, _ = orc.unpack_dequant_reduce_requant([cb, ca], [sb, sa], 1024, p)
    np.testing.assert_array_equal(ab.view(np.uint32), ba.view(np.uint32))


@pytest.mark.parametrize("bin_,bout,Bin,Bout", [(4, 4, 128, 128), (8, 4, 512, 128), (2, 2, 64, 64), (4, 8, 32, 256)])
def test_requant_equals_encoder_on_the_sum(orc, bin_, bout, Bin, Bout):
    # Stage 2 = the encoder's stage applied to v2 = sum + e2, with e2' = v2 - s2*q2.
    rng = np.random.default_rng(bin_ * 100 + bout)
    n, W = 3000, 3
    pin = orc.params(bin_, Bin)
    pout = orc.params(bout, Bout, orc.SR, seed=9, index_offset=123, philox_stream=1)
    cs, ss = zip(*[orc.quantize_pack(rng.standard_normal(n).astype(np.float32), pin) for _ in range(W)])
    e2 = (rng.standard_normal(n) * 0.01).astype(np.float32)
    e2_copy = e2.copy()
    sum_, co, so = orc.unpack_dequant_reduce_requant(list(cs), list(ss), n, pin, True, e2, pout)
    v2 = (sum_ + e2_copy).astype(np.float32)
    e_ref = np.zeros(n, np.float32)
    c_ref, s_ref = orc.quantize_pack(v2, pout, e_ref)
    # quantize_pack adds its err input (zeros) to v2: identical values
    assert co.tobytes() == c_ref.tobytes() and (so == s_ref).all()
    np.testing.assert_array_equal(e2.view(np.uint32), e_ref.view(np.uint32))


# ---- all-gather-side decode ------------------------------------------------

def test_f32_to_bf16_matches_torch(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    u = np.concatenate([rng.integers(0, 2 ** 32, 200_000, dtype=np.uint64).astype(np.uint32),
                        np.arange(0x7F7F0000, 0x7F800000, 7, dtype=np.uint32),     # overflow boundary
                        np.arange(0x00000000, 0x00030000, 3, dtype=np.uint32),     # subnormals
                        (np.arange(0, 65536, dtype=np.uint32) << 16) | 0x8000])   # exact ties
    x = u.view(np.float32)
    x = x[~np.isnan(x)]
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    L = orc.lib()
    got = np.fromiter((L.orc_f32_to_bf16(float(v)) for v in x), dtype=np.uint16, count=x.size)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [hex(int(x.view(np.uint32)[i])) for i in bad[:5]]


@pytest.mark.parametrize("bits", [1, 2, 4, 8, 12, 16])
def test_unpack_dequant_equals_single_rank_sum(orc, bits):
    # With mul = 1 and fp32 output the all-gather-side decode is the W=1
    # decoder's sum; with mul = 1/4 every value is that sum times 2^-2 exactly.
    rng = np.random.default_rng(bits)
    n = 3000
    x = rng.standard_normal(n).astype(np.float32)
    p = orc.params(bits, 128)
    c, s = orc.quantize_pack(x, p)
    ref, _, _ = orc.unpack_dequant_reduce_requant([c], [s], n, p)
    np.testing.assert_array_equal(orc.unpack_dequant(c, s, n, p).view(np.uint32), ref.view(np.uint32))
    np.testing.assert_array_equal(orc.unpack_dequant(c, s, n, p, mul=0.25), ref * np.float32(0.25))
    # a multiplier that rounds: the product s*q is rounded first, then scaled
    third = np.float32(1.0 / 3.0)
    np.testing.assert_array_equal(orc.unpack_dequant(c, s, n, p, mul=float(third)).view(np.uint32),
                                  (ref * third).astype(np.float32).view(np.uint32))
    bf = orc.unpack_dequant(c, s, n, p, mul=0.25, out_dtype=orc.BF16)
    torch = pytest.importorskip("torch")
    exp = torch.from_numpy(ref * np.float32(0.25)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bf, exp)


# ---- Hadamard smoothing (SDP4Bit README, "--hadamard-transform") -----------

@pytest.mark.parametrize("H", [8, 16, 32, 64, 128, 256])
def test_fwht_is_the_sylvester_hadamard_matrix(orc, H):
    sla = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(H)
    x = rng.integers(-1000, 1001, size=4 * H).astype(np.float32)   # sums stay exact in fp32
    got = orc.fwht(x, H)
    Hm = sla.hadamard(H).astype(np.float64)
    ref = (x.reshape(4, H).astype(np.float64) @ Hm.T).reshape(-1)
    np.testing.assert_array_equal(got.astype(np.float64), ref)
    np.testing.assert_array_equal(orc.fwht(got, H) / np.float32(H), x)      # H H = H I


def test_hadamard_hand_block(orc):
    # x = e_0 in one block of 8: the transform is all ones, absmax 1, s =
    # fp16(1/7) = 1170 * 2^-13 = 0.142822265625 (0x3092), every q = rint(7.0017)
    # = 7 (code 15).  Decoding: d = 7s everywhere, the inverse transform puts
    # 8 * 7s / 8 = 0.999755859375 at index 0 and exact zeros elsewhere.
    x = np.zeros(8, np.float32)
    x[0] = 1.0
    p = orc.params(4, 8, hadamard=8)
    codes, scales, deq = orc.roundtrip(x, p)
    assert int(scales[0]) == 0x3092
    assert codes.tobytes().hex() == "ffffffff"
    assert deq.tolist() == [0.999755859375] + [0.0] * 7


def test_decoder_does_not_transform(orc):
    # The rank sum and the requantisation stay in the transformed domain:
    # requantising one rank's own dequantised values with the same parameters
    # reproduces its codes and scales exactly.
    rng = np.random.default_rng(2)
    x = rng.standard_normal(4096).astype(np.float32)
    p = orc.params(4, 128, hadamard=128)
    c, s = orc.quantize_pack(x, p)
    _, co, so = orc.unpack_dequant_reduce_requant([c], [s], 4096, p, False, None, p)
    assert co.tobytes() == c.tobytes() and np.array_equal(so, s)
    with pytest.raises(ValueError):   # stages must share the transform
        orc.unpack_dequant_reduce_requant([c], [s], 4096, p, False, None, orc.params(4, 128))


def test_hadamard_reduces_error_on_outlier_blocks(orc):
    # The page's stated purpose: the rotation spreads an outlier over its block,
    # so the 4-bit roundtrip error of outlier-heavy gradients drops.
    rng = np.random.default_rng(3)
    n = 1 << 16
    x = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    x[rng.integers(0, n, n // 128)] *= 100.0
    plain = orc.roundtrip(x, orc.params(4, 128))[2]
    rot = orc.roundtrip(x, orc.params(4, 128, hadamard=128))[2]
    e_plain = np.linalg.norm(plain.astype(np.float64) - x)
    e_rot = np.linalg.norm(rot.astype(np.float64) - x)
    assert e_rot < 0.7 * e_plain, (e_rot, e_plain)


def test_hadamard_rejects_bad_sizes(orc):
    with pytest.raises(ValueError):
        orc.quantize_pack(np.zeros(100, np.float32), orc.params(4, 128, hadamard=128))   # n % H
    with pytest.raises(ValueError):
        orc.quantize_pack(np.zeros(128, np.float32), orc.params(4, 64, hadamard=128))    # H > B


# ---- weight-difference quantisation (SDP4Bit README, weight quantisation) ---

def test_qwd_hand_block(orc):
    # ref = 1.0 everywhere, w = ref + HAND_X: the difference is the hand block,
    # so codes and scale are the b=4 hand values and ref advances by s*q.
    ref = np.ones(8, np.float32)
    w = (ref + HAND_X).astype(np.float32)
    codes, scales = orc.qwd_encode(w, ref, orc.params(4, 8))
    assert int(scales[0]) == 0x3492 and codes.tobytes().hex() == "4af9851d"
    s = 0.28564453125
    np.testing.assert_array_equal(ref.astype(np.float64), 1.0 + np.array([2, -4, 1, 7, -3, 0, 5, -7]) * s)


def test_qwd_receivers_track_the_sender(orc):
    # Every receiver applying the gathered codes to its reference copy ends with
    # the sender's reference, bit for bit, over many steps; the gap w - ref
    # stays within half a quantum of the last step's scale (round to nearest).
    rng = np.random.default_rng(6)
    n, B = 8192, 2048
    w = rng.standard_normal(n).astype(np.float32)
    ref_send = w.copy()
    ref_recv = w.copy()
    p = orc.params(4, B)
    for t in range(12):
        w = (w - np.float32(1e-3) * rng.standard_normal(n).astype(np.float32)).astype(np.float32)
        codes, scales = orc.qwd_encode(w, ref_send, p)
        wout = orc.qwd_apply(codes, scales, n, p, ref_recv, w_dtype=orc.BF16)
        np.testing.assert_array_equal(ref_send.view(np.uint32), ref_recv.view(np.uint32))
        s = np.repeat(scales_f64(scales), B)
        gap = np.abs(w.astype(np.float64) - ref_send.astype(np.float64))
        assert (gap <= s / 2 + 2.0 ** -23 * np.abs(w) + 1e-30).all()
        torch = pytest.importorskip("torch")
        exp = torch.from_numpy(ref_recv.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(wout, exp)


def test_sum_ranks_order_and_zeros(orc):
    # The full-precision local reduce adds the ranks in order, rank 0 first, in
    # fp32.  Worked by hand: 2^24 + 1 is a tie between 2^24 and 2^24 + 2 that
    # goes to the even 2^24, so ((2^24 + 1) + 1) - 2^24 = 0 in rank order,
    # while any order that adds the two ones first gives 2; and (-2^24 + 2^24)
    # + 1 = 1 where ((1 + 2^24) - 2^24) would give 0.  Rank 0's -0 stays -0
    # (a sum seeded with +0 would turn it into +0); +0 + -0 = +0.
    big = np.float32(2.0 ** 24)
    xs = [np.array([big, -big, 1.0, -0.0, 0.0], np.float32),
          np.array([1.0, big, big, -0.0, -0.0], np.float32),
          np.array([1.0, 1.0, -big, -0.0, -0.0], np.float32),
          np.array([-big, 0.0, 0.0, -0.0, -0.0], np.float32)]
    out = orc.sum_ranks(xs)
    assert out.tolist()[:3] == [0.0, 1.0, 0.0]
    assert np.signbit(out[3]) and not np.signbit(out[4])
    # reversing the rank order changes both sums: (((-2^24 + 1) + 1) + 2^24) = 2
    # exactly, and (0 + 1) + 2^24 is the tie that goes to 2^24, leaving 0
    rev = orc.sum_ranks(xs[::-1])
    assert rev.tolist()[:2] == [2.0, 0.0]


def test_sum_ranks_exact_on_small_integers_and_bf16(orc):
    # Sums of small integers are exact in any order: the closed form is the
    # integer sum.  bf16 inputs widen exactly (bf16 bits << 16); integers up to
    # 256 in magnitude are exact in bf16's 8 significant bits.
    rng = np.random.default_rng(3)
    xs = [rng.integers(-256, 257, 257).astype(np.float32) for _ in range(9)]
    assert np.array_equal(orc.sum_ranks(xs), np.sum(np.array(xs, np.int64), axis=0).astype(np.float32))
    bf = [(x.view(np.uint32) >> 16).astype(np.uint16) for x in xs]
    assert np.array_equal(orc.sum_ranks(bf), orc.sum_ranks(xs))
