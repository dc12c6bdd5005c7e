"""The five workloads at their full sizes on the GPU, checked against the CPU
oracle on every element.  The small ones are compared in one piece; the large
ones are streamed through the oracle in block-aligned slices on every host
core (tests/whole_check.py): every block is independent given its global
element index, so a slice is a complete oracle problem of its own.  The
oracle always starts from its own state (zero error buffers) -- no oracle
input comes from the CUDA path."""
import numpy as np
import pytest
import torch

import oracle as O
import whole_check
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu


def _bits16(x):
    return x.view(torch.int16).cpu().numpy().view(np.uint16)


def _host(x):
    return x.cpu().numpy() if x.dtype == torch.float32 else _bits16(x)


def test_roundtrip_1m_full():
    _, bc = need_gpu()
    from bit_gradient_communication_gb300 import synth
    wl = synth.WORKLOADS["roundtrip_1m"]
    x = synth.gradients(wl.kind, wl.n, wl.seed, **wl.params)
    p = bc.QParams(wl.bits, wl.block)
    codes, scales = bc.alloc_codes(wl.n, p)
    deq = bc.roundtrip(x, p, codes_tmp=codes, scales_tmp=scales)
    torch.cuda.synchronize()
    c_ref, s_ref, d_ref = O.roundtrip(x.cpu().numpy(), O.params(wl.bits, wl.block))
    assert codes.cpu().numpy().tobytes() == c_ref.tobytes()
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), s_ref)
    assert np.array_equal(deq.cpu().numpy().view(np.uint32), d_ref.view(np.uint32))


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_bucket25mb_ten_steps_full(bits):
    _, bc = need_gpu()
    from bit_gradient_communication_gb300 import synth
    wl = synth.WORKLOADS["bucket25mb_f32"]
    n = wl.n
    sched = bc.Scheduler(n_streams=2, bucket_bytes=wl.bucket_bytes)
    err = torch.zeros(n, device="cuda")
    err_ref = np.zeros(n, np.float32)
    for t in range(10):
        x = synth.gradients(wl.kind, n, t, **wl.params)
        p = bc.QParams(bits, wl.block, wl.rounding, seed=wl.sr_seed, index_offset=t * n)
        codes, scales = sched.quantize_pack(x, p, err)
        sched.wait()
        c_ref, s_ref = O.quantize_pack(x.cpu().numpy(),
                                       O.params(bits, wl.block, wl.rounding, seed=wl.sr_seed,
                                                index_offset=t * n), err_ref)
        assert codes.cpu().numpy().tobytes() == c_ref.tobytes(), f"step {t}"
        assert np.array_equal(scales.cpu().numpy().view(np.uint16), s_ref), f"step {t}"
        assert np.array_equal(err.cpu().numpy().view(np.uint32), err_ref.view(np.uint32)), f"step {t}"
    sched.close()


def _f32(t):
    return t.cpu().numpy()


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _u8(t):
    return t.cpu().numpy()


def test_allreduce_w8_gpt1p3b_whole_two_steps():
    """Config 3 whole: 8 ranks x 1.3e9 bf16, two steps of the simulated
    all-reduce with the bench's launches (8 encoders, 8 chunk decoders).  Every
    element's codes, scale, error e' and stage-2 error e2' and every output code
    and scale of both steps is compared with the oracle (step 2 starts from the
    errors step 1 left, on both sides)."""
    _, bc = need_gpu()
    import bench
    from bit_gradient_communication_gb300 import synth
    W, n, B, b = 8, bench.N_PER_RANK, bench.BLOCK, bench.BITS
    ar = bench.AllReduceW8(torch, bc, synth, n, W, torch.device("cuda"))
    ar.encode()
    ar.decode()
    first = {"err": [e.clone() for e in ar.err], "codes": [c.clone() for c in ar.codes],
             "scales": [s.clone() for s in ar.scales], "err2": ar.err2.clone(),
             "codes_out": ar.codes_out.clone(), "scales_out": ar.scales_out.clone()}
    ar.encode()
    ar.decode()
    torch.cuda.synchronize()
    second = {"err": ar.err, "codes": list(ar.codes), "scales": list(ar.scales), "err2": ar.err2,
              "codes_out": ar.codes_out, "scales_out": ar.scales_out}
    assert n % B == 0

    def state(st, lo, hi):
        return {"err": [_f32(e[lo:hi]) for e in st["err"]],
                "codes": [_u8(c[lo * b // 8: hi * b // 8]) for c in st["codes"]],
                "scales": [_u16(s[lo // B: hi // B]) for s in st["scales"]],
                "err2": _f32(st["err2"][lo:hi]), "codes_out": _u8(st["codes_out"][lo * b // 8: hi * b // 8]),
                "scales_out": _u16(st["scales_out"][lo // B: hi // B])}

    def fetch(lo, hi):
        return {"x": [_u16(x[lo:hi]) for x in ar.x], 1: state(first, lo, hi), 2: state(second, lo, hi)}

    def check(lo, hi, d):
        m = hi - lo
        e = [np.zeros(m, np.float32) for _ in range(W)]
        e2 = np.zeros(m, np.float32)
        for step in (1, 2):
            g = d[step]
            enc = []
            for w in range(W):
                c, s = O.quantize_pack(d["x"][w], O.params(b, B, seed=1000 + w, index_offset=lo), e[w])
                assert whole_check.same_bits(c, g["codes"][w]), f"step {step} rank {w} codes at {lo}"
                assert whole_check.same_bits(s, g["scales"][w]), f"step {step} rank {w} scales at {lo}"
                assert whole_check.same_bits(e[w], g["err"][w]), f"step {step} rank {w} e' at {lo}"
                enc.append((c, s))
            _, co, so = O.unpack_dequant_reduce_requant([c for c, _ in enc], [s for _, s in enc], m,
                                                        O.params(b, B), False, e2,
                                                        O.params(b, B, index_offset=lo, philox_stream=1))
            assert whole_check.same_bits(co, g["codes_out"]), f"step {step} output codes at {lo}"
            assert whole_check.same_bits(so, g["scales_out"]), f"step {step} output scales at {lo}"
            assert whole_check.same_bits(e2, g["err2"]), f"step {step} e2' at {lo}"

    checked = whole_check.run(whole_check.slices(n, 1 << 21), fetch, check)
    assert checked == n
    del ar, first, second
    torch.cuda.empty_cache()


def test_gpt6p7b_2bit_buckets_whole_two_steps():
    """Config 4 whole: 6.7e9 bf16, 2-bit block-64 stochastic rounding with
    error feedback, 512 buckets of 25 MiB on two streams, two steps (step t
    draws Philox words at global index t*n + i).  Every element's codes,
    scale and e' of both steps is compared with the oracle."""
    _, bc = need_gpu()
    from bit_gradient_communication_gb300 import synth
    wl = synth.WORKLOADS["gpt6p7b_2bit_buckets"]
    n, b, B = wl.n, wl.bits, wl.block
    x = synth.gradients(wl.kind, n, wl.seed, dtype=torch.bfloat16, **wl.params)
    err = torch.zeros(n, device="cuda")
    codes, scales = bc.alloc_codes(n, bc.QParams(b, B))
    sched = bc.Scheduler(n_streams=2, bucket_bytes=wl.bucket_bytes)
    assert len(bc.plan_buckets(n, 2, B, wl.bucket_bytes)) - 1 == 512
    p = lambda t: bc.QParams(b, B, wl.rounding, seed=wl.sr_seed, index_offset=t * n)
    sched.quantize_pack(x, p(0), err, codes, scales)
    sched.wait(timeout_s=120)
    first = (err.clone(), codes.clone(), scales.clone())
    sched.quantize_pack(x, p(1), err, codes, scales)
    sched.wait(timeout_s=120)
    torch.cuda.synchronize()
    sched.close()
    assert n % B == 0

    def fetch(lo, hi):
        out = {"x": _u16(x[lo:hi])}
        for step, (e, c, s) in ((0, first), (1, (err, codes, scales))):
            out[step] = (_f32(e[lo:hi]), _u8(c[lo * b // 8: hi * b // 8]), _u16(s[lo // B: hi // B]))
        return out

    def check(lo, hi, d):
        e = np.zeros(hi - lo, np.float32)
        for step in (0, 1):
            c, s = O.quantize_pack(d["x"], O.params(b, B, wl.rounding, seed=wl.sr_seed,
                                                    index_offset=step * n + lo), e)
            ge, gc, gs = d[step]
            assert whole_check.same_bits(c, gc), f"step {step} codes at {lo}"
            assert whole_check.same_bits(s, gs), f"step {step} scales at {lo}"
            assert whole_check.same_bits(e, ge), f"step {step} e' at {lo}"

    checked = whole_check.run(whole_check.slices(n, 1 << 22), fetch, check)
    assert checked == n
    del x, err, codes, scales, first
    torch.cuda.empty_cache()


SWEEP_BITS = (1, 2, 4, 8, 12, 16)
SWEEP_BLOCKS = (32, 64, 128, 256, 1024, 4096)


def test_sweep_laplace_256m_whole():
    """Config 5 whole: 268,435,456 fp32 Laplace(0, 1e-3), every bits x block x
    {RTN, SR} cell (72).  Per cell the encoder (codes, scales) and the W=1
    decoder the sweep times (fl(s*q) as the rank sum) are compared with the
    oracle on every element; the one-pass roundtrip entry point must give the
    same codes, scales and values bit for bit."""
    _, bc = need_gpu()
    from bit_gradient_communication_gb300 import synth
    wl = synth.WORKLOADS["sweep_laplace_256m"]
    n = wl.n
    x = synth.gradients(wl.kind, n, wl.seed, **wl.params)
    xh = x.cpu().numpy()
    deq = torch.empty(n, device="cuda")
    rt = torch.empty(n, device="cuda")
    total = 0
    for bits in SWEEP_BITS:
        for block in SWEEP_BLOCKS:
            for rounding in (bc.RTN, bc.SR):
                p = bc.QParams(bits, block, rounding, seed=wl.sr_seed)
                codes, scales = bc.quantize_pack(x, p)
                bc.unpack_dequant_reduce_requant([codes], [scales], n, p, sum_out=deq)
                c2, s2 = bc.alloc_codes(n, p)
                bc.roundtrip(x, p, codes_tmp=c2, scales_tmp=s2, deq_out=rt)
                torch.cuda.synchronize()
                tag = f"b={bits} B={block} r={rounding}"
                assert torch.equal(c2, codes) and torch.equal(s2, scales), tag
                assert torch.equal(rt.view(torch.int32), deq.view(torch.int32)), tag
                del c2, s2

                def fetch(lo, hi):
                    return (_u8(codes[lo * bits // 8: hi * bits // 8]), _u16(scales[lo // block: hi // block]),
                            _f32(deq[lo:hi]))

                def check(lo, hi, d):
                    op = O.params(bits, block, rounding, seed=wl.sr_seed, index_offset=lo)
                    c, s = O.quantize_pack(xh[lo:hi], op)
                    assert whole_check.same_bits(c, d[0]), f"{tag} codes at {lo}"
                    assert whole_check.same_bits(s, d[1]), f"{tag} scales at {lo}"
                    assert whole_check.same_bits(O.unpack_dequant(c, s, hi - lo, op), d[2]), f"{tag} values at {lo}"

                total += whole_check.run(whole_check.slices(n, 1 << 22), fetch, check)
                del codes, scales
    assert total == n * len(SWEEP_BITS) * len(SWEEP_BLOCKS) * 2
    del x, deq, rt
    torch.cuda.empty_cache()


def test_local_sum_w8_gpt1p3b_whole():
    """Pipeline-A's full-precision local reduce at the bench's size: the fp32
    rank-ordered sum of 8 local ranks' 1.3e9-element bf16 gradients, compared
    with the oracle's sum on every element."""
    _, bc = need_gpu()
    from bit_gradient_communication_gb300 import synth
    wl = synth.WORKLOADS["local_sum_w8_gpt1p3b"]
    n = wl.n
    xs = [synth.gradients(wl.kind, n, wl.seed + w, dtype=torch.bfloat16, **wl.params) for w in range(wl.ranks)]
    out = torch.empty(n, device="cuda")
    bc.sum_ranks(xs, out=out)
    torch.cuda.synchronize()

    def fetch(lo, hi):
        return [_bits16(x[lo:hi]) for x in xs], _f32(out[lo:hi])

    def check(lo, hi, d):
        assert whole_check.same_bits(O.sum_ranks(d[0]), d[1]), f"sum at {lo}"

    assert whole_check.run(whole_check.slices(n, 1 << 22), fetch, check) == n
    del xs, out
    torch.cuda.empty_cache()


def test_local_decode_w8_gpt1p3b_whole():
    """Pipeline-A's local stage with local quantisation at the bench's size: 8
    local ranks' 1.3e9-element bf16 gradients encoded to 4-bit block-128 codes
    and decoded by the leader into their rank-ordered fp32 sum.  Per slice the
    oracle encodes every rank's gradient itself and sums the decoded values;
    codes, scales and the sum are compared on every element."""
    _, bc = need_gpu()
    from bit_gradient_communication_gb300 import synth
    wl = synth.WORKLOADS["local_decode_w8_gpt1p3b"]
    n, b, B = wl.n, wl.bits, wl.block
    p = bc.QParams(b, B)
    xs, cs, ss = [], [], []
    for w in range(wl.ranks):
        x = synth.gradients(wl.kind, n, wl.seed + w, dtype=torch.bfloat16, **wl.params)
        c, s = bc.quantize_pack(x, p)
        xs.append(x)
        cs.append(c)
        ss.append(s)
    out = torch.empty(n, device="cuda")
    bc.unpack_dequant_reduce_requant(cs, ss, n, p, sum_out=out)
    torch.cuda.synchronize()

    def fetch(lo, hi):
        return ([_bits16(x[lo:hi]) for x in xs], [_u8(c[lo * b // 8: hi * b // 8]) for c in cs],
                [_u16(s[lo // B: hi // B]) for s in ss], _f32(out[lo:hi]))

    def check(lo, hi, d):
        op = O.params(b, B)
        enc = [O.quantize_pack(x, op) for x in d[0]]
        for w, (c, s) in enumerate(enc):
            assert whole_check.same_bits(c, d[1][w]), f"rank {w} codes at {lo}"
            assert whole_check.same_bits(s, d[2][w]), f"rank {w} scales at {lo}"
        total, _, _ = O.unpack_dequant_reduce_requant([c for c, _ in enc], [s for _, s in enc], hi - lo, op,
                                                      True, None, None)
        assert whole_check.same_bits(total, d[3]), f"sum at {lo}"

    assert whole_check.run(whole_check.slices(n, 1 << 22), fetch, check) == n
    del xs, cs, ss, out
    torch.cuda.empty_cache()
