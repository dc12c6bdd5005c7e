"""One launch over more than 2^31 elements: the encoder (stochastic rounding,
error feedback), the decoder (two ranks, stage-2 feedback, stochastic
requantisation) and the all-gather-side decode to bf16, each over
n = 2^31 + 2^20 + 37 elements (a ragged last block), checked against the CPU
oracle on block-aligned windows on both sides of element 2^31 and at the
tail.  Every block is an independent problem given its global element index,
so a window is a complete oracle problem of its own; the oracle starts from
zero error buffers like the GPU run.  Guard bands around every output must
survive."""
import numpy as np
import pytest

import oracle as O
from gpu_util import GUARD, SENTINEL, need_gpu

pytestmark = pytest.mark.gpu

N = 2 ** 31 + 2 ** 20 + 37
B = 128
SEED_1, SEED_2 = 77, 99


def _guarded(torch, nbytes, fill=None):
    raw = torch.full((nbytes + 2 * GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
    if fill is not None:
        raw[GUARD:GUARD + nbytes].fill_(fill)
    return raw


def _payload(raw, nbytes, dtype):
    return raw[GUARD:GUARD + nbytes].view(dtype)


def _bands_intact(raw, nbytes):
    return bool((raw[:GUARD] == SENTINEL).all().item() and (raw[GUARD + nbytes:] == SENTINEL).all().item())


@pytest.fixture(scope="module")
def run():
    torch, bc = need_gpu()
    from bit_gradient_communication_gb300 import synth
    free, _ = torch.cuda.mem_get_info()
    if free < 40 * 2 ** 30:
        pytest.skip("needs about 30 GB of device memory")
    x = synth.gradients("normal", N, 2024, dtype=torch.bfloat16, sigma=1e-3)
    p1 = bc.QParams(4, B, bc.SR, seed=SEED_1)
    p2 = bc.QParams(4, B, bc.SR, seed=SEED_2, philox_stream=1)
    nc, ns = bc.packed_bytes(N, 4, B), 2 * bc.num_blocks(N, B)
    codes, scales, err = _guarded(torch, nc), _guarded(torch, ns), _guarded(torch, 4 * N, 0)
    bc.quantize_pack(x, p1, _payload(err, 4 * N, torch.float32), _payload(codes, nc, torch.uint8),
                     _payload(scales, ns, torch.int16))
    c_in, s_in = _payload(codes, nc, torch.uint8), _payload(scales, ns, torch.int16)
    e2, co, so = _guarded(torch, 4 * N, 0), _guarded(torch, nc), _guarded(torch, ns)
    bc.unpack_dequant_reduce_requant([c_in, c_in], [s_in, s_in], N, bc.QParams(4, B), None,
                                     _payload(e2, 4 * N, torch.float32), p2,
                                     _payload(co, nc, torch.uint8), _payload(so, ns, torch.int16))
    deq = _guarded(torch, 2 * N)
    bc.unpack_dequant(_payload(co, nc, torch.uint8), _payload(so, ns, torch.int16), N, p2, 0.5,
                      _payload(deq, 2 * N, torch.bfloat16))
    torch.cuda.synchronize()
    out = dict(x=x, codes=codes, scales=scales, err=err, e2=e2, co=co, so=so, deq=deq, nc=nc, ns=ns)
    yield out
    out.clear()
    del x, codes, scales, err, e2, co, so, deq
    torch.cuda.empty_cache()


def _windows():
    nb = (N + B - 1) // B
    rng = np.random.default_rng(5)
    starts = {0, 2 ** 31 // B - 8, 2 ** 31 // B - 1, 2 ** 31 // B + 3, nb - 16}
    starts |= set(int(v) for v in rng.integers(0, nb - 16, 6))
    return [(b * B, min((b + 16) * B, N), b) for b in sorted(starts)]


def test_guard_bands_survive(run):
    for k in ("codes", "scales", "err", "e2", "co", "so", "deq"):
        nbytes = {"codes": run["nc"], "co": run["nc"], "scales": run["ns"], "so": run["ns"]}.get(k)
        if nbytes is None:
            nbytes = 4 * N if k in ("err", "e2") else 2 * N
        assert _bands_intact(run[k], nbytes), k


@pytest.mark.parametrize("lo,hi,b0", _windows())
def test_window_matches_oracle(run, lo, hi, b0):
    import torch
    m = hi - lo
    c0, c1 = lo * 4 // 8, (b0 + (m + B - 1) // B) * B * 4 // 8
    nbw = (m + B - 1) // B

    def codes_of(raw):
        return raw[GUARD + c0:GUARD + c1].cpu().numpy()

    def scales_of(raw):
        return raw[GUARD + 2 * b0:GUARD + 2 * (b0 + nbw)].cpu().numpy().view(np.uint16)

    def f32_of(raw):
        return raw[GUARD + 4 * lo:GUARD + 4 * hi].cpu().numpy().view(np.float32)

    xw = run["x"][lo:hi].view(torch.int16).cpu().numpy().view(np.uint16)
    e = np.zeros(m, np.float32)
    c_ref, s_ref = O.quantize_pack(xw, O.params(4, B, O.SR, seed=SEED_1, index_offset=lo), e)
    assert codes_of(run["codes"]).tobytes() == c_ref.tobytes()
    assert np.array_equal(scales_of(run["scales"]), s_ref)
    assert np.array_equal(f32_of(run["err"]).view(np.uint32), e.view(np.uint32))

    e2 = np.zeros(m, np.float32)
    p_out = O.params(4, B, O.SR, seed=SEED_2, index_offset=lo, philox_stream=1)
    _, co, so = O.unpack_dequant_reduce_requant([c_ref, c_ref], [s_ref, s_ref], m, O.params(4, B), False,
                                                e2, p_out)
    assert codes_of(run["co"]).tobytes() == co.tobytes()
    assert np.array_equal(scales_of(run["so"]), so)
    assert np.array_equal(f32_of(run["e2"]).view(np.uint32), e2.view(np.uint32))

    d_ref = O.unpack_dequant(co, so, m, p_out, 0.5, O.BF16)
    d = run["deq"][GUARD + 2 * lo:GUARD + 2 * hi].cpu().numpy().view(np.uint16)
    assert np.array_equal(d, d_ref)
