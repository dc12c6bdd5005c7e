"""The sharded low-bit all-reduce across real ranks, on the CPU (gloo).

Each of W ranks encodes its own gradient (oracle codec, first-stage error
feedback, per-rank stochastic-rounding seed), sends chunk c of its codes and
scales to rank c (the all-to-all, done with point-to-point messages because
gloo has no all-to-all), decodes the W chunks it received in rank order,
requantises with its shard of the stage-2 error and all-gathers the
requantised chunks (bitscom README, "Implemented Features": all-to-all ->
local reduce -> all-gather; DeAR README: reduce-scatter + all-gather).  The
gathered result and every error buffer must equal the single-process
simulation with W arrays, which is what the GPU path computes.
"""
import os
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N, BITS, BLOCK, STEPS = 3 * 4096 + 640, 4, 128, 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _chunks(n, W, B):
    nb = (n + B - 1) // B
    cb = (nb + W - 1) // W
    out = []
    for c in range(W):
        b0, b1 = c * cb, min((c + 1) * cb, nb)
        out.append((b0 * B, min(b1 * B, n), b0, b1))
    return out


def _grad(rank, step):
    import sys
    sys.path.insert(0, ROOT)
    from bit_gradient_communication_gb300 import synth
    return synth.np_gradients("student_t3", N, 100 * rank + step, scale=1e-3)


def _worker(rank, W, port, outdir, drop=None, timeout_s=None):
    """One rank.  drop = (rank, step): that rank leaves at the start of that
    step without a word (a crashed process); the others must notice on the
    host, through an error from the exchange, and leave that step cleanly."""
    import sys
    from datetime import timedelta
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    kw = {"timeout": timedelta(seconds=timeout_s)} if timeout_s else {}
    dist.init_process_group("gloo", rank=rank, world_size=W, **kw)
    chunks = _chunks(N, W, BLOCK)
    lo, hi, b0, b1 = chunks[rank]
    err = np.zeros(N, np.float32)
    e2_shard = np.zeros(hi - lo, np.float32)
    for step in range(STEPS):
        if drop is not None and drop == (rank, step):
            os._exit(0)
        if drop is not None:
            try:
                _step(rank, W, step, chunks, err, e2_shard, outdir, O, torch, dist)
            except RuntimeError as exc:
                with open(os.path.join(outdir, f"failed{rank}.txt"), "w") as f:
                    f.write(f"{step}\n{type(exc).__name__}: {exc}\n")
                os._exit(0)
            continue
        _step(rank, W, step, chunks, err, e2_shard, outdir, O, torch, dist)
    np.save(os.path.join(outdir, f"err{rank}.npy"), err)
    dist.barrier()
    dist.destroy_process_group()


def _step(rank, W, step, chunks, err, e2_shard, outdir, O, torch, dist):
    """One all-reduce step of one rank: encode, all-to-all, reduce, all-gather."""
    lo, hi, b0, b1 = chunks[rank]
    g = _grad(rank, step)
    p1 = O.params(BITS, BLOCK, O.SR, seed=1000 + rank, index_offset=step * N)
    codes, scales = O.quantize_pack(g, p1, err)
    # all-to-all: rank c receives chunk c from every rank
    recv_c, recv_s = [None] * W, [None] * W
    reqs = []
    for c in range(W):
        clo, chi, cb0, cb1 = chunks[c]
        cc = codes[clo * BITS // 8: cb1 * BLOCK * BITS // 8]
        cs = scales[cb0:cb1]
        if c == rank:
            recv_c[rank], recv_s[rank] = cc.copy(), cs.copy()
            continue
        reqs.append(dist.isend(torch.from_numpy(cc.copy()), dst=c))
        reqs.append(dist.isend(torch.from_numpy(cs.view(np.int16).copy()), dst=c))
    for w in range(W):
        if w == rank:
            continue
        tc = torch.empty((b1 - b0) * BLOCK * BITS // 8, dtype=torch.uint8)
        ts = torch.empty(b1 - b0, dtype=torch.int16)
        dist.recv(tc, src=w)
        dist.recv(ts, src=w)
        recv_c[w], recv_s[w] = tc.numpy(), ts.numpy().view(np.uint16)
    for r in reqs:
        r.wait()
    # local reduce + stage-2 requantisation of this rank's chunk
    p2 = O.params(BITS, BLOCK, O.SR, seed=77, index_offset=step * N + lo, philox_stream=1)
    _, co, so = O.unpack_dequant_reduce_requant(recv_c, recv_s, hi - lo, O.params(BITS, BLOCK),
                                                False, e2_shard, p2)
    gathered = [None] * W
    dist.all_gather_object(gathered, (co, so, e2_shard.copy()))
    if rank == 0:
        np.savez(os.path.join(outdir, f"step{step}.npz"),
                 codes=np.concatenate([x[0] for x in gathered]),
                 scales=np.concatenate([x[1] for x in gathered]),
                 e2=np.concatenate([x[2] for x in gathered]))


def _simulate(O, W):
    errs = [np.zeros(N, np.float32) for _ in range(W)]
    e2 = np.zeros(N, np.float32)
    outs = []
    for step in range(STEPS):
        enc = []
        for w in range(W):
            p1 = O.params(BITS, BLOCK, O.SR, seed=1000 + w, index_offset=step * N)
            enc.append(O.quantize_pack(_grad(w, step), p1, errs[w]))
        p2 = O.params(BITS, BLOCK, O.SR, seed=77, index_offset=step * N, philox_stream=1)
        _, co, so = O.unpack_dequant_reduce_requant([c for c, _ in enc], [s for _, s in enc], N,
                                                    O.params(BITS, BLOCK), False, e2, p2)
        outs.append((co, so, e2.copy()))
    return outs, errs


@pytest.mark.parametrize("W", [2, 3])
def test_gloo_ranks_equal_single_process_simulation(orc, tmp_path, W):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, W, port, str(tmp_path))) for r in range(W)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    outs, errs = _simulate(orc, W)
    for step in range(STEPS):
        got = np.load(tmp_path / f"step{step}.npz")
        co, so, e2 = outs[step]
        assert got["codes"].tobytes() == co.tobytes()
        assert np.array_equal(got["scales"], so)
        assert np.array_equal(got["e2"].view(np.uint32), e2.view(np.uint32))
    for w in range(W):
        assert np.array_equal(np.load(tmp_path / f"err{w}.npy").view(np.uint32), errs[w].view(np.uint32))
    del torch


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
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    port = _free_port()
    W = 2
    procs = [ctx.Process(target=_worker, args=(r, W, port, str(tmp_path), (1, 1), 20)) for r in range(W)]
    t0 = time.monotonic()
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
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
    assert (tmp_path / "step0.npz").exists()
