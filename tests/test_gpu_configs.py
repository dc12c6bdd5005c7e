"""The five workloads at their full sizes on the GPU, checked against the CPU
oracle.  Workloads the oracle finishes in seconds are compared whole; the
large ones on block-aligned windows (first and last blocks, chunk and bucket
boundaries, random positions): every block is independent given its global
element index, so a window is a complete oracle problem of its own.
The oracle always starts from its own state (zero error buffers) -- no
oracle input comes from the CUDA path."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu


def _bits16(x):
    return x.view(torch.int16).cpu().numpy().view(np.uint16)


def _host(x):
    return x.cpu().numpy() if x.dtype == torch.float32 else _bits16(x)


def _windows(n, block, count, length_blocks, seed, must_blocks=()):
    nb = (n + block - 1) // block
    rng = np.random.default_rng(seed)
    starts = {0, max(0, nb - length_blocks)}
    for b in must_blocks:
        for d in (-1, 0):
            starts.add(min(max(0, b + d * length_blocks // 2), max(0, nb - length_blocks)))
    starts |= set(int(v) for v in rng.integers(0, max(1, nb - length_blocks), count))
    return [(b * block, min((b + length_blocks) * block, n), b) for b in sorted(starts)]


def _codes_window(codes, bits, lo, hi, block):
    b0 = lo // block
    b1 = (hi + block - 1) // block
    return codes[b0 * block * bits // 8: b1 * block * bits // 8]


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


def test_allreduce_w8_gpt1p3b_windows():
    _, bc = need_gpu()
    import bench
    from bit_gradient_communication_gb300 import synth
    W, n = 8, bench.N_PER_RANK
    ar = bench.AllReduceW8(torch, bc, synth, n, W, torch.device("cuda"))
    ar.encode()
    ar.decode()
    torch.cuda.synchronize()
    B = bench.BLOCK
    bounds = [lo // B for (lo, _) in ar.chunks]
    for lo, hi, b0 in _windows(n, B, 48, 64, 3, bounds):
        m = hi - lo
        enc = []
        for w in range(W):
            e = np.zeros(m, np.float32)
            c_ref, s_ref = O.quantize_pack(_bits16(ar.x[w][lo:hi]), O.params(4, B), e)
            enc.append((c_ref, s_ref))
            assert _codes_window(ar.codes[w], 4, lo, hi, B).cpu().numpy().tobytes() == c_ref.tobytes()
            assert np.array_equal(ar.scales[w][b0:b0 + len(s_ref)].cpu().numpy().view(np.uint16), s_ref)
            assert np.array_equal(ar.err[w][lo:hi].cpu().numpy().view(np.uint32), e.view(np.uint32))
        e2 = np.zeros(m, np.float32)
        _, co, so = O.unpack_dequant_reduce_requant([c for c, _ in enc], [s for _, s in enc], m,
                                                    O.params(4, B), False, e2,
                                                    O.params(4, B, index_offset=lo, philox_stream=1))
        assert _codes_window(ar.codes_out, 4, lo, hi, B).cpu().numpy().tobytes() == co.tobytes()
        assert np.array_equal(ar.scales_out[b0:b0 + len(so)].cpu().numpy().view(np.uint16), so)
        assert np.array_equal(ar.err2[lo:hi].cpu().numpy().view(np.uint32), e2.view(np.uint32))
    del ar
    torch.cuda.empty_cache()


def test_gpt6p7b_2bit_buckets_windows():
    _, bc = need_gpu()
    from bit_gradient_communication_gb300 import synth
    wl = synth.WORKLOADS["gpt6p7b_2bit_buckets"]
    n = wl.n
    x = synth.gradients(wl.kind, n, wl.seed, dtype=torch.bfloat16, **wl.params)
    err = torch.zeros(n, device="cuda")
    p = bc.QParams(wl.bits, wl.block, wl.rounding, seed=wl.sr_seed)
    codes, scales = bc.alloc_codes(n, p)
    sched = bc.Scheduler(n_streams=2, bucket_bytes=wl.bucket_bytes)
    sched.quantize_pack(x, p, err, codes, scales)
    sched.wait(timeout_s=120)
    starts = bc.plan_buckets(n, 2, wl.block, wl.bucket_bytes)
    assert len(starts) - 1 == 512
    bounds = [s // wl.block for s in starts[1:-1:37]] + [starts[-2] // wl.block]
    for lo, hi, b0 in _windows(n, wl.block, 48, 128, 4, bounds):
        e = np.zeros(hi - lo, np.float32)
        c_ref, s_ref = O.quantize_pack(_bits16(x[lo:hi]),
                                       O.params(wl.bits, wl.block, wl.rounding, seed=wl.sr_seed,
                                                index_offset=lo), e)
        assert _codes_window(codes, wl.bits, lo, hi, wl.block).cpu().numpy().tobytes() == c_ref.tobytes()
        assert np.array_equal(scales[b0:b0 + len(s_ref)].cpu().numpy().view(np.uint16), s_ref)
        assert np.array_equal(err[lo:hi].cpu().numpy().view(np.uint32), e.view(np.uint32))
    sched.close()
    del x, err, codes, scales
    torch.cuda.empty_cache()


def test_sweep_laplace_256m_windows():
    _, bc = need_gpu()
    from bit_gradient_communication_gb300 import synth
    wl = synth.WORKLOADS["sweep_laplace_256m"]
    n = wl.n
    x = synth.gradients(wl.kind, n, wl.seed, **wl.params)
    deq = torch.empty(n, device="cuda")
    for bits in (1, 2, 4, 8, 12, 16):
        for block in (32, 64, 128, 256, 1024, 4096):
            for rounding in (bc.RTN, bc.SR):
                p = bc.QParams(bits, block, rounding, seed=wl.sr_seed)
                codes, scales = bc.alloc_codes(n, p)
                bc.roundtrip(x, p, codes_tmp=codes, scales_tmp=scales, deq_out=deq)
                torch.cuda.synchronize()
                for lo, hi, b0 in _windows(n, block, 6, max(1, 4096 // block), bits * 100 + block):
                    c_ref, s_ref, d_ref = O.roundtrip(
                        x[lo:hi].cpu().numpy(), O.params(bits, block, rounding, seed=wl.sr_seed, index_offset=lo))
                    tag = f"b={bits} B={block} r={rounding} lo={lo}"
                    assert _codes_window(codes, bits, lo, hi, block).cpu().numpy().tobytes() == c_ref.tobytes(), tag
                    assert np.array_equal(scales[b0:b0 + len(s_ref)].cpu().numpy().view(np.uint16), s_ref), tag
                    assert np.array_equal(deq[lo:hi].cpu().numpy().view(np.uint32), d_ref.view(np.uint32)), tag
                del codes, scales
    del x, deq
    torch.cuda.empty_cache()
