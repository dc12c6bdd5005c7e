"""Hierarchical pipeline-A across real ranks on the CPU (gloo): 4 ranks in 2
local groups of 2 (leaders 0 and 2 form the inter group) run the package's
orchestration (hierarchical.PipelineA) with the codec steps in the CPU oracle
(tests/oracle_codec.py), for both settings of local_quantize, over two steps
and several pipeline chunks (the last one ragged).  Every rank's output and
every error buffer must equal a single-process restatement written with the
oracle: per chunk, the local reduce (full-precision rank-ordered sum, or the
local ranks' encoders + the rank-ordered decode), the leaders' low-bit
all-reduce (encoders, chunking, decode + stage-2 requantisation, all-gather)
and the decode (bitscom README, "Implemented Features": hierarchical pipeline-A
local reduce -> inter lowbit all-reduce -> local broadcast; "Hierarchical
All-Reduce Options": local_quantize)."""
import os
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N, CHUNK, STEPS, L, G = 3 * 1024 + 256, 1024, 2, 2, 2
B1 = B2 = BL = 128
BITS, ROUNDING = 4, 1


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
    return synth.np_gradients("student_t3", N, 31 * rank + step, scale=1e-3)


def _worker(rank, port, outdir, local_quantize):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist

    import bit_gradient_communication_gb300 as bc
    from bit_gradient_communication_gb300 import hierarchical, sharded
    from oracle_codec import OracleCodec
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=L * G)
    local_groups = [dist.new_group([g * L + l for l in range(L)]) for g in range(G)]
    inter_group = dist.new_group([g * L for g in range(G)])
    node, lrank = divmod(rank, L)
    local = sharded.Exchange(local_groups[node], host_staging=(node == 1))
    inter = sharded.Exchange(inter_group) if lrank == 0 else None
    pa = hierarchical.PipelineA(N, torch.float32, local, inter,
                                bc.QParams(BITS, B1, ROUNDING, seed=500 + node),
                                bc.QParams(BITS, B2, ROUNDING, seed=77, philox_stream=1), chunk_size=CHUNK,
                                local_quantize=local_quantize,
                                p_local=bc.QParams(BITS, BL, ROUNDING, seed=900 + rank), device="cpu",
                                codec=OracleCodec())
    for step in range(STEPS):
        out = torch.empty(N)
        pa(torch.from_numpy(_grad(rank, step)), out, mul=1.0 / (L * G))
        np.save(os.path.join(outdir, f"out{step}_{rank}.npy"), out.numpy())
    if pa.err_local is not None:
        np.save(os.path.join(outdir, f"elocal{rank}.npy"), pa.err_local.numpy())
    if pa.ar is not None:
        np.save(os.path.join(outdir, f"einter{node}.npy"), pa.ar.err.numpy())
        np.save(os.path.join(outdir, f"e2_{node}.npy"), pa.ar.err2[:pa.ar.shard].numpy())
    dist.barrier()
    dist.destroy_process_group()


def _restate(O, local_quantize):
    """The single-process oracle restatement of the four ranks, chunk by chunk."""
    from bit_gradient_communication_gb300 import sharded
    e_local = [np.zeros(N, np.float32) for _ in range(L * G)]
    e_inter = [np.zeros(N, np.float32) for _ in range(G)]
    e2 = np.zeros(N, np.float32)
    outs = []
    for step in range(STEPS):
        base = step * N
        g = [_grad(r, step) for r in range(L * G)]
        out = np.zeros(N, np.float32)
        for c0 in range(0, N, CHUNK):
            c1 = min(c0 + CHUNK, N)
            m = c1 - c0
            # local reduce to each leader
            sums = []
            for node in range(G):
                ranks = [node * L + l for l in range(L)]
                if not local_quantize:
                    sums.append(O.sum_ranks([g[r][c0:c1] for r in ranks]))
                else:
                    enc = [O.quantize_pack(g[r][c0:c1], O.params(BITS, BL, ROUNDING, seed=900 + r,
                                                                 index_offset=base + c0, philox_stream=2),
                                           e_local[r][c0:c1]) for r in ranks]
                    s, _, _ = O.unpack_dequant_reduce_requant([c for c, _ in enc], [q for _, q in enc], m,
                                                              O.params(BITS, BL), True)
                    sums.append(s)
            # the leaders' low-bit all-reduce of the chunk (one bucket)
            enc = [O.quantize_pack(sums[node], O.params(BITS, B1, ROUNDING, seed=500 + node, index_offset=base + c0),
                                   e_inter[node][c0:c1]) for node in range(G)]
            codes = np.zeros(O.packed_bytes(m, BITS, B2), np.uint8)
            scales = np.zeros(O.num_blocks(m, B2), np.uint16)
            bk = sharded.plan(m, 4, B1, B2, G, 0)[0]
            for lo, hi in bk.chunks:
                if hi <= lo:
                    continue
                cs = slice(lo * BITS // 8, lo * BITS // 8 + sharded.code_bytes(lo, hi, BITS, B1))
                ss = slice(lo // B1, lo // B1 + sharded.scale_count(lo, hi, B1))
                _, co, so = O.unpack_dequant_reduce_requant(
                    [c[cs] for c, _ in enc], [q[ss] for _, q in enc], hi - lo, O.params(BITS, B1), False,
                    e2[c0 + lo:c0 + hi], O.params(BITS, B2, ROUNDING, seed=77, philox_stream=1,
                                                  index_offset=base + c0 + lo))
                codes[lo * BITS // 8: lo * BITS // 8 + co.size] = co
                scales[lo // B2: lo // B2 + so.size] = so
            out[c0:c1] = O.unpack_dequant(codes, scales, m, O.params(BITS, B2), 1.0 / (L * G))
        outs.append(out)
    return outs, e_local, e_inter, e2


@pytest.mark.parametrize("local_quantize", [False, True])
def test_pipeline_a_equals_oracle_restatement(orc, tmp_path, local_quantize):
    pytest.importorskip("torch")
    import torch.multiprocessing as mp

    from bit_gradient_communication_gb300 import sharded
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, str(tmp_path), local_quantize)) for r in range(L * G)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    outs, e_local, e_inter, e2 = _restate(orc, local_quantize)
    for step in range(STEPS):
        for r in range(L * G):
            got = np.load(tmp_path / f"out{step}_{r}.npy")
            assert np.array_equal(got.view(np.uint32), outs[step].view(np.uint32)), (step, r)
    if local_quantize:
        for r in range(L * G):
            assert np.array_equal(np.load(tmp_path / f"elocal{r}.npy").view(np.uint32), e_local[r].view(np.uint32))
    for node in range(G):
        assert np.array_equal(np.load(tmp_path / f"einter{node}.npy").view(np.uint32), e_inter[node].view(np.uint32))
        # the leader's stage-2 shard: its chunks of every pipeline chunk, in order
        shard = np.concatenate([e2[c0 + bk.chunks[node][0]:c0 + bk.chunks[node][1]]
                                for c0 in range(0, N, CHUNK)
                                for bk in [sharded.plan(min(CHUNK, N - c0), 4, B1, B2, G, 0)[0]]])
        assert np.array_equal(np.load(tmp_path / f"e2_{node}.npy").view(np.uint32), shard.view(np.uint32))
