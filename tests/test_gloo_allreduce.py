"""The sharded low-bit all-reduce across real ranks, on the CPU (gloo).

Each of W processes runs the package's multi-rank orchestration
(bit_gradient_communication_gb300.sharded.LowBitAllReduce): it encodes its own
gradient bucket by bucket (first-stage error feedback, per-rank
stochastic-rounding seed), sends chunk c of its codes and scales to rank c
(all_to_all_single), decodes the W chunks it received in rank order,
requantises with its shard of the stage-2 error, all-gathers the requantised
chunks and decodes the mean (bitscom README, "Implemented Features":
all-to-all -> local reduce -> all-gather; DeAR README: reduce-scatter +
all-gather).  The codec steps run in the CPU oracle here (tests/oracle_codec.py;
the GPU version of this test, tests/test_gpu_sharded.py, runs libbitscom).  The
gathered codes, scales, decoded mean and every error buffer must equal the
single-process simulation of W ranks (tests/sharded_sim.py) over two steps.
"""
import os
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N, BITS, BLOCK, STEPS = 3 * 4096 + 640, 4, 128, 2
BUCKET_BYTES = 16 * 1024          # 4096 fp32 elements: four buckets, the last one ragged


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _grad(rank, step):
    import sys
    sys.path.insert(0, ROOT)
    from bit_gradient_communication_gb300 import synth
    return synth.np_gradients("student_t3", N, 100 * rank + step, scale=1e-3)


# (bits1, block1, bits2, block2, hadamard): one format, and the two-level 8 -> 4-bit
# format with Hadamard smoothing (chunks are then whole 512-element blocks)
FORMATS = {"b4": (4, 128, 4, 128, 0), "tlq_hs": (8, 512, 4, 128, 128)}


def _worker(rank, W, port, outdir, drop=None, timeout_s=None, fmt="b4"):
    """One rank.  drop = (rank, step): that rank leaves at the start of that
    step without a word (a crashed process); the others must notice on the
    host, through an error from the exchange, and leave that step cleanly."""
    import sys
    from datetime import timedelta
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist

    import bit_gradient_communication_gb300 as bc
    from bit_gradient_communication_gb300 import sharded
    from oracle_codec import OracleCodec
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    kw = {"timeout": timedelta(seconds=timeout_s)} if timeout_s else {}
    dist.init_process_group("gloo", rank=rank, world_size=W, **kw)
    b1, B1, b2, B2, H = FORMATS[fmt]
    ar = sharded.LowBitAllReduce(N, torch.float32, bc.QParams(b1, B1, bc.SR, seed=1000 + rank, hadamard=H),
                                 bc.QParams(b2, B2, bc.SR, seed=77, philox_stream=1, hadamard=H), device="cpu",
                                 bucket_bytes=BUCKET_BYTES, codec=OracleCodec(),
                                 exchange=sharded.Exchange(host_staging=(W == 3)))
    for step in range(STEPS):
        if drop is not None and drop == (rank, step):
            os._exit(0)
        g = torch.from_numpy(_grad(rank, step))
        codes = torch.zeros(bc.packed_bytes(N, b2, B2), dtype=torch.uint8)
        scales = torch.zeros(bc.num_blocks(N, B2), dtype=torch.int16)
        out = torch.empty(N)
        try:
            ar(g, out=out, mul=1.0 / W, out_codes=codes, out_scales=scales)
        except RuntimeError as exc:
            if drop is None:
                raise
            with open(os.path.join(outdir, f"failed{rank}.txt"), "w") as f:
                f.write(f"{step}\n{type(exc).__name__}: {exc}\n")
            os._exit(0)
        np.savez(os.path.join(outdir, f"step{step}_rank{rank}.npz"), codes=codes.numpy(),
                 scales=scales.numpy().view(np.uint16), out=out.numpy())
    np.save(os.path.join(outdir, f"err{rank}.npy"), ar.err.numpy())
    np.save(os.path.join(outdir, f"e2_{rank}.npy"), ar.err2[:ar.shard].numpy())
    dist.barrier()
    dist.destroy_process_group()


def _run_ranks(W, tmp_path, drop=None, timeout_s=None, join_s=300, fmt="b4"):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, W, port, str(tmp_path), drop, timeout_s, fmt)) for r in range(W)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=join_s)
    return procs


@pytest.mark.parametrize("W,fmt", [(2, "b4"), (3, "b4"), (3, "tlq_hs")])
def test_gloo_ranks_equal_single_process_simulation(orc, tmp_path, W, fmt):
    pytest.importorskip("torch")
    import sharded_sim
    procs = _run_ranks(W, tmp_path, fmt=fmt)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    grads = [[_grad(w, t) for w in range(W)] for t in range(STEPS)]
    b1, B1, b2, B2, H = FORMATS[fmt]
    results, errs, e2 = sharded_sim.simulate(grads, N, b1, B1, 1, [1000 + w for w in range(W)], 77,
                                             BUCKET_BYTES, mul=1.0 / W, bits2=b2, block2=B2, hadamard=H)
    for step in range(STEPS):
        codes, scales, out = results[step]
        for w in range(W):
            got = np.load(tmp_path / f"step{step}_rank{w}.npz")
            assert got["codes"].tobytes() == codes.tobytes(), (step, w)
            assert np.array_equal(got["scales"], scales), (step, w)
            assert np.array_equal(got["out"].view(np.uint32), out.view(np.uint32)), (step, w)
    for w in range(W):
        assert np.array_equal(np.load(tmp_path / f"err{w}.npy").view(np.uint32), errs[w].view(np.uint32))
        shard = sharded_sim.shard_of(e2, N, W, w, B1, BUCKET_BYTES, block2=B2)
        assert np.array_equal(np.load(tmp_path / f"e2_{w}.npy").view(np.uint32), shard.view(np.uint32))


def test_bench_reference_arm_under_torchrun(tmp_path):
    # The multi-rank launch of bench.py: rank 0 prints one JSON line, the other
    # ranks exit 0 without work (the reference arm needs no GPU).
    import json
    import subprocess
    import sys
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
                        "--ref-sample", "4096"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["cpu_baseline"]["cores"] == 1


def test_rank_that_leaves_is_detected_on_the_host(tmp_path):
    # Rank 1 of 2 crashes at the start of step 1 (no goodbye); rank 0 must get
    # an error from that step's exchange within the process-group timeout,
    # record it and exit, instead of waiting for ever.
    pytest.importorskip("torch")
    import time
    t0 = time.monotonic()
    procs = _run_ranks(2, tmp_path, drop=(1, 1), timeout_s=20, join_s=240)
    alive = [p.is_alive() for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert not any(alive), "a rank hung after its peer left"
    assert time.monotonic() - t0 < 240
    failed = tmp_path / "failed0.txt"
    assert failed.exists(), "rank 0 did not notice that rank 1 left"
    step, what = failed.read_text().split("\n", 1)
    assert step == "1" and what.strip()
    # step 0 completed on both ranks before the drop
    assert (tmp_path / "step0_rank0.npz").exists() and (tmp_path / "step0_rank1.npz").exists()


BENCH_N, BENCH_BUCKET = 2 * 4096 + 256, 8 * 1024      # bf16: three buckets of 4096, 4096, 256


def _bench_grad(rank):
    import torch
    return torch.from_numpy(_grad(rank, 0)[:BENCH_N].copy()).to(torch.bfloat16)


def _bench_worker(rank, W, port, outdir):
    """One rank of bench.py's multi-GPU mode (its setup, parameters and call),
    with the oracle codec on host tensors in place of the GPU."""
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist

    import bench
    import bit_gradient_communication_gb300 as bc
    from bit_gradient_communication_gb300 import sharded, synth
    from oracle_codec import OracleCodec
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=W)
    ar, grad = bench.sharded_rank(torch, bc, synth, sharded, BENCH_N, rank, W, "cpu", BENCH_BUCKET,
                                  codec=OracleCodec(), exchange=sharded.Exchange(), grad=_bench_grad(rank))
    codes = torch.zeros(bc.packed_bytes(BENCH_N, 4, 128), dtype=torch.uint8)
    scales = torch.zeros(bc.num_blocks(BENCH_N, 128), dtype=torch.int16)
    ar.finish(ar.reduce(ar.send(grad)), out_codes=codes, out_scales=scales)
    np.savez(os.path.join(outdir, f"bench{rank}.npz"), codes=codes.numpy(), scales=scales.numpy().view(np.uint16),
             err=ar.err.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_bench_multi_gpu_mode_is_the_simulated_all_reduce(orc, tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    import sharded_sim
    W = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_bench_worker, args=(r, W, port, str(tmp_path))) for r in range(W)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    grads = [[_bench_grad(w).view(torch.int16).numpy().view(np.uint16) for w in range(W)]]
    results, errs, _ = sharded_sim.simulate(grads, BENCH_N, 4, 128, 0, [1000 + w for w in range(W)], 0,
                                            BENCH_BUCKET, elem_bytes=2)
    codes, scales, _ = results[0]
    for w in range(W):
        got = np.load(tmp_path / f"bench{w}.npz")
        assert got["codes"].tobytes() == codes.tobytes()
        assert np.array_equal(got["scales"], scales)
        assert np.array_equal(got["err"].view(np.uint32), errs[w].view(np.uint32))
