"""Bucket scheduler on the GPU: bucketed results equal one unbucketed call and
the oracle; the simulated W-rank all-reduce equals the oracle's W-array
simulation; the bench's launch sequence equals the scheduler's; resuming from
saved error buffers equals an uninterrupted run; the host wait is bounded."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import bf16_bits_of, need_gpu

pytestmark = pytest.mark.gpu


def _x(n, seed, dt):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn(n, generator=g, device="cuda") * 1e-3
    return x if dt == "f32" else x.to(torch.bfloat16)


def _host_bits(x):
    if x.dtype == torch.float32:
        return x.cpu().numpy()
    return x.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("sr", [False, True])
@pytest.mark.parametrize("ef", [True, False])
def test_bucketed_encoder_equals_unbucketed_and_oracle(dt, sr, ef):
    # with and without error feedback (the two take different thread layouts)
    _, bc = need_gpu()
    n = 20 * 4096 + 77
    x = _x(n, 1, dt)
    p = bc.QParams(2, 64, bc.SR if sr else bc.RTN, seed=4242, index_offset=12345)
    sched = bc.Scheduler(n_streams=3, bucket_bytes=16 * 1024)
    assert len(bc.plan_buckets(n, x.element_size(), 64, 16 * 1024)) - 1 > 4
    e1 = torch.zeros(n, device="cuda") if ef else None
    e2 = torch.zeros(n, device="cuda") if ef else None
    for _ in range(2):                       # two calls: error feedback carried
        c1, s1 = sched.quantize_pack(x, p, e1)
        c2, s2 = bc.quantize_pack(x, p, e2)
    sched.wait()
    torch.cuda.synchronize()
    assert torch.equal(c1, c2) and torch.equal(s1, s2)
    if ef:
        assert torch.equal(e1.view(torch.int32), e2.view(torch.int32))
    e_ref = np.zeros(n, np.float32) if ef else None
    po = O.params(2, 64, O.SR if sr else O.RTN, seed=4242, index_offset=12345)
    for _ in range(2):
        c_ref, s_ref = O.quantize_pack(_host_bits(x), po, e_ref)
    assert c1.cpu().numpy().tobytes() == c_ref.tobytes()
    assert np.array_equal(s1.cpu().numpy().view(np.uint16), s_ref)
    if ef:
        assert np.array_equal(e1.cpu().numpy().view(np.uint32), e_ref.view(np.uint32))
    sched.close()


def _oracle_allreduce(xs_host, n, W, p1s, p2, errs, e2):
    enc = [O.quantize_pack(xs_host[w], p1s[w], errs[w]) for w in range(W)]
    s, co, so = O.unpack_dequant_reduce_requant([c for c, _ in enc], [s for _, s in enc], n, p1s[0],
                                                True, e2, p2)
    return enc, s, co, so


@pytest.mark.parametrize("W,bucket", [(3, 48 * 1024), (8, 0), (2, 8 * 1024)])
def test_scheduled_allreduce_matches_oracle(W, bucket):
    _, bc = need_gpu()
    n = 30 * 4096 + 200
    sched = bc.Scheduler(n_streams=2, bucket_bytes=bucket)
    xs = [_x(n, 10 + w, "bf16") for w in range(W)]
    errs = [torch.zeros(n, device="cuda") for _ in range(W)]
    codes, scales = zip(*[bc.alloc_codes(n, bc.QParams(4, 128)) for _ in range(W)])
    err2 = torch.zeros(n, device="cuda")
    co, so = bc.alloc_codes(n, bc.QParams(4, 128))
    sum_out = torch.empty(n, device="cuda")
    h_err = [np.zeros(n, np.float32) for _ in range(W)]
    h_e2 = np.zeros(n, np.float32)
    for step in range(2):
        p1 = [bc.QParams(4, 128, bc.SR, seed=1000 + w, index_offset=step * n) for w in range(W)]
        p2 = bc.QParams(4, 128, bc.SR, seed=7, index_offset=step * n, philox_stream=1)
        sched.allreduce(xs, p1, codes, scales, errs, p2, err2, co, so, sum_out)
        sched.wait()
        enc, s_ref, c_ref, sc_ref = _oracle_allreduce(
            [_host_bits(x) for x in xs], n, W,
            [O.params(4, 128, O.SR, seed=1000 + w, index_offset=step * n) for w in range(W)],
            O.params(4, 128, O.SR, seed=7, index_offset=step * n, philox_stream=1), h_err, h_e2)
        for w in range(W):
            assert codes[w].cpu().numpy().tobytes() == enc[w][0].tobytes()
            assert np.array_equal(errs[w].cpu().numpy().view(np.uint32), h_err[w].view(np.uint32))
        assert np.array_equal(sum_out.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
        assert co.cpu().numpy().tobytes() == c_ref.tobytes()
        assert np.array_equal(so.cpu().numpy().view(np.uint16), sc_ref)
        assert np.array_equal(err2.cpu().numpy().view(np.uint32), h_e2.view(np.uint32))
    sched.close()


def test_bench_sequence_equals_scheduler():
    torch_, bc = need_gpu()
    import bench
    from bit_gradient_communication_gb300 import synth
    n = 50 * 4096 + 128
    ar = bench.AllReduceW8(torch, bc, synth, n, 8, torch.device("cuda"))
    xs = [x.clone() for x in ar.x]
    ar.encode()
    ar.decode()
    sched = bc.Scheduler(n_streams=2, bucket_bytes=0)
    errs = [torch.zeros(n, device="cuda") for _ in range(8)]
    codes, scales = zip(*[bc.alloc_codes(n, ar.p1[0]) for _ in range(8)])
    err2 = torch.zeros(n, device="cuda")
    co, so = bc.alloc_codes(n, ar.p2)
    sched.allreduce(xs, ar.p1, codes, scales, errs, ar.p2, err2, co, so)
    sched.wait()
    torch.cuda.synchronize()
    assert torch.equal(co, ar.codes_out) and torch.equal(so, ar.scales_out)
    assert torch.equal(err2.view(torch.int32), ar.err2.view(torch.int32))
    for w in range(8):
        assert torch.equal(codes[w], ar.codes[w])
    sched.close()


def test_checkpoint_resume_equals_uninterrupted():
    # The library is stateless: state = the caller's error buffer + the Philox
    # index offset.  Ten steps straight == five, save, restore into fresh
    # buffers, five more.
    _, bc = need_gpu()
    n = 8 * 4096 + 16
    grads = [_x(n, 100 + t, "f32") for t in range(10)]

    def run(steps, err):
        out = None
        for t in steps:
            out = bc.quantize_pack(grads[t], bc.QParams(2, 256, bc.SR, seed=42, index_offset=t * n), err)
        return out

    e_a = torch.zeros(n, device="cuda")
    ca, sa = run(range(10), e_a)
    e_b = torch.zeros(n, device="cuda")
    run(range(5), e_b)
    saved = e_b.cpu().numpy().copy()
    e_c = torch.from_numpy(saved).cuda()
    cb, sb = run(range(5, 10), e_c)
    torch.cuda.synchronize()
    assert torch.equal(ca, cb) and torch.equal(sa, sb) and torch.equal(e_a.view(torch.int32), e_c.view(torch.int32))


def test_host_wait_times_out_then_completes():
    _, bc = need_gpu()
    sched = bc.Scheduler(n_streams=1, bucket_bytes=0)
    torch.cuda._sleep(int(1.5e9))            # a bounded busy kernel (~0.7 s)
    with pytest.raises(bc.BitscomError) as ei:
        sched.wait(timeout_s=0.01)
    assert ei.value.status == 5
    sched.wait(timeout_s=60.0)
    sched.close()


def test_allreduce_then_allgather_decode_matches_oracle():
    # The whole low-bit all-reduce: encoders, chunk decoders, and every rank's
    # decode of the all-gathered requantised codes into its mean gradient (bf16).
    _, bc = need_gpu()
    W, n = 4, 20 * 4096 + 64
    sched = bc.Scheduler(n_streams=2, bucket_bytes=64 * 1024)
    xs = [_x(n, 40 + w, "bf16") for w in range(W)]
    errs = [torch.zeros(n, device="cuda") for _ in range(W)]
    p1 = [bc.QParams(4, 128, bc.RTN) for _ in range(W)]
    p2 = bc.QParams(4, 128, bc.RTN, philox_stream=1)
    codes, scales = zip(*[bc.alloc_codes(n, p1[0]) for _ in range(W)])
    err2 = torch.zeros(n, device="cuda")
    co, so = bc.alloc_codes(n, p2)
    sched.allreduce(xs, p1, codes, scales, errs, p2, err2, co, so)
    mean = bc.unpack_dequant(co, so, n, p2, mul=1.0 / W, out_dtype=torch.bfloat16)
    sched.wait()
    torch.cuda.synchronize()
    h_err = [np.zeros(n, np.float32) for _ in range(W)]
    _, _, c_ref, s_ref = _oracle_allreduce([_host_bits(x) for x in xs], n, W,
                                           [O.params(4, 128) for _ in range(W)],
                                           O.params(4, 128, philox_stream=1), h_err, np.zeros(n, np.float32))
    ref = O.unpack_dequant(c_ref, s_ref, n, O.params(4, 128), float(np.float32(1.0 / W)), O.BF16)
    assert np.array_equal(_host_bits(mean), ref)
    sched.close()


def test_two_level_hadamard_allreduce_matches_oracle():
    # SDP4Bit-style two-level quantisation with Hadamard smoothing: stage 1
    # 8-bit groups of 512, stage 2 4-bit groups of 128, both rotated by H = 128;
    # then the all-gather-side decode back to the bf16 mean gradient.
    _, bc = need_gpu()
    W, n = 8, 16 * 4096
    sched = bc.Scheduler(n_streams=2, bucket_bytes=0)
    xs = [_x(n, 70 + w, "bf16") for w in range(W)]
    errs = [torch.zeros(n, device="cuda") for _ in range(W)]
    p1 = [bc.QParams(8, 512, bc.RTN, hadamard=128) for _ in range(W)]
    p2 = bc.QParams(4, 128, bc.SR, seed=11, philox_stream=1, hadamard=128)
    codes, scales = zip(*[bc.alloc_codes(n, p1[0]) for _ in range(W)])
    err2 = torch.zeros(n, device="cuda")
    co, so = bc.alloc_codes(n, p2)
    sched.allreduce(xs, p1, codes, scales, errs, p2, err2, co, so)
    mean = bc.unpack_dequant(co, so, n, p2, mul=1.0 / W, out_dtype=torch.bfloat16)
    sched.wait()
    torch.cuda.synchronize()
    h_err = [np.zeros(n, np.float32) for _ in range(W)]
    h_e2 = np.zeros(n, np.float32)
    o1 = [O.params(8, 512, hadamard=128) for _ in range(W)]
    o2 = O.params(4, 128, O.SR, seed=11, philox_stream=1, hadamard=128)
    _, _, c_ref, s_ref = _oracle_allreduce([_host_bits(x) for x in xs], n, W, o1, o2, h_err, h_e2)
    assert co.cpu().numpy().tobytes() == c_ref.tobytes()
    assert np.array_equal(err2.cpu().numpy().view(np.uint32), h_e2.view(np.uint32))
    ref = O.unpack_dequant(c_ref, s_ref, n, o2, float(np.float32(1.0 / W)), O.BF16)
    assert np.array_equal(_host_bits(mean), ref)
    sched.close()
