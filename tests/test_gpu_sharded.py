"""The multi-rank low-bit all-reduce with libbitscom doing every codec step.

W processes share cuda:0 (one GPU per box here): each runs the package's
orchestration (sharded.LowBitAllReduce) with the default codec -- the CUDA
kernels behind the C ABI -- and exchanges codes and scales over gloo through
host memory (no kernel waits on another process).  Over two steps, every
rank's gathered codes, scales, decoded mean, error buffer and stage-2 error
shard must equal, bit for bit,
  * the single-process oracle simulation of W ranks (tests/sharded_sim.py), and
  * the library's own single-GPU simulation (bitscom_sched_allreduce through
    Scheduler.allreduce), which pins the multi-rank chunking to the C
    scheduler's.
"""
import os
import socket

import numpy as np
import pytest

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N, STEPS, BUCKET_BYTES = 3 * 4096 + 640, 2, 16 * 1024


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _grad_f32(rank, step):
    import sys
    sys.path.insert(0, ROOT)
    from bit_gradient_communication_gb300 import synth
    return synth.np_gradients("student_t3", N, 100 * rank + step, scale=1e-3)


def _grad(torch, rank, step, bf16):
    g = torch.from_numpy(_grad_f32(rank, step))
    return g.to(torch.bfloat16) if bf16 else g


# (bits1, block1, bits2, block2, hadamard): one format, and the two-level 8 -> 4-bit
# format with Hadamard smoothing
FORMATS = {"b4": (4, 128, 4, 128, 0), "tlq_hs": (8, 512, 4, 128, 128)}


def _params(bc, rounding, rank, fmt, index_offset=0):
    b1, B1, b2, B2, H = FORMATS[fmt]
    return (bc.QParams(b1, B1, rounding, seed=1000 + rank, hadamard=H, index_offset=index_offset),
            bc.QParams(b2, B2, rounding, seed=77, philox_stream=1, hadamard=H, index_offset=index_offset))


def _worker(rank, W, port, outdir, bf16, rounding, fmt):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bit_gradient_communication_gb300 as bc
    from bit_gradient_communication_gb300 import sharded
    bc.lib()
    torch.cuda.set_device(0)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=W)
    dt = torch.bfloat16 if bf16 else torch.float32
    p1, p2 = _params(bc, rounding, rank, fmt)
    ar = sharded.LowBitAllReduce(N, dt, p1, p2, device="cuda:0", bucket_bytes=BUCKET_BYTES,
                                 exchange=sharded.Exchange(host_staging=True))
    for step in range(STEPS):
        g = _grad(torch, rank, step, bf16).cuda()
        codes = torch.zeros(bc.packed_bytes(N, p2.bits, p2.block), dtype=torch.uint8, device="cuda")
        scales = torch.zeros(bc.num_blocks(N, p2.block), dtype=torch.int16, device="cuda")
        out = torch.empty(N, device="cuda")
        ar(g, out=out, mul=1.0 / W, out_codes=codes, out_scales=scales)
        torch.cuda.synchronize()
        np.savez(os.path.join(outdir, f"step{step}_rank{rank}.npz"), codes=codes.cpu().numpy(),
                 scales=scales.cpu().numpy().view(np.uint16), out=out.cpu().numpy())
    np.save(os.path.join(outdir, f"err{rank}.npy"), ar.err.cpu().numpy())
    np.save(os.path.join(outdir, f"e2_{rank}.npy"), ar.err2[:ar.shard].cpu().numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("W,bf16,rounding,fmt", [(2, True, 0, "b4"), (3, False, 1, "b4"), (3, False, 1, "tlq_hs")])
def test_ranks_on_libbitscom_equal_oracle_and_single_gpu_simulation(orc, tmp_path, W, bf16, rounding, fmt):
    torch, bc = need_gpu()
    import torch.multiprocessing as mp

    import sharded_sim
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, W, port, str(tmp_path), bf16, rounding, fmt)) for r in range(W)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]

    esz = 2 if bf16 else 4
    host = [[_grad(torch, w, t, bf16) for w in range(W)] for t in range(STEPS)]
    grads = [[(g.view(torch.int16).numpy().view(np.uint16) if bf16 else g.numpy()) for g in gw] for gw in host]
    b1, B1, b2, B2, H = FORMATS[fmt]
    results, errs, e2 = sharded_sim.simulate(grads, N, b1, B1, rounding, [1000 + w for w in range(W)], 77,
                                             BUCKET_BYTES, elem_bytes=esz, mul=1.0 / W, bits2=b2, block2=B2,
                                             hadamard=H)
    # the library's single-GPU simulation of the same W ranks
    sched = bc.Scheduler(n_streams=2, bucket_bytes=BUCKET_BYTES)
    d_err = [torch.zeros(N, device="cuda") for _ in range(W)]
    d_e2 = torch.zeros(N, device="cuda")
    sim = []
    for t in range(STEPS):
        xs = [g.cuda() for g in host[t]]
        p1 = [_params(bc, rounding, w, fmt, t * N)[0] for w in range(W)]
        p2 = _params(bc, rounding, 0, fmt, t * N)[1]
        cs, ss = zip(*[bc.alloc_codes(N, p1[0]) for _ in range(W)])
        co, so = bc.alloc_codes(N, p2)
        sched.allreduce(xs, p1, cs, ss, d_err, p2, d_e2, co, so)
        sched.wait()
        sim.append((co.cpu().numpy(), so.cpu().numpy().view(np.uint16)))
    sched.close()

    for step in range(STEPS):
        codes, scales, out = results[step]
        assert sim[step][0].tobytes() == codes.tobytes() and np.array_equal(sim[step][1], scales), step
        for w in range(W):
            got = np.load(tmp_path / f"step{step}_rank{w}.npz")
            assert got["codes"].tobytes() == codes.tobytes(), (step, w)
            assert np.array_equal(got["scales"], scales), (step, w)
            assert np.array_equal(got["out"].view(np.uint32), out.view(np.uint32)), (step, w)
    for w in range(W):
        assert np.array_equal(np.load(tmp_path / f"err{w}.npy").view(np.uint32), errs[w].view(np.uint32))
        assert np.array_equal(d_err[w].cpu().numpy().view(np.uint32), errs[w].view(np.uint32))
        shard = sharded_sim.shard_of(e2, N, W, w, B1, BUCKET_BYTES, elem_bytes=esz, block2=B2)
        assert np.array_equal(np.load(tmp_path / f"e2_{w}.npy").view(np.uint32), shard.view(np.uint32))
    assert np.array_equal(d_e2.cpu().numpy().view(np.uint32), e2.view(np.uint32))
