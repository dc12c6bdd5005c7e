"""Hierarchical pipeline-A with libbitscom doing every codec step: 4 processes
share cuda:0, in 2 local groups of 2, exchanging over gloo through host
memory (no kernel waits on another process).  Every rank's output and error
buffers must equal the oracle restatement of tests/test_gloo_hierarchical.py,
for both settings of local_quantize, over two steps."""
import os
import socket

import numpy as np
import pytest

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, port, outdir, local_quantize):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist

    import bit_gradient_communication_gb300 as bc
    import test_gloo_hierarchical as T
    from bit_gradient_communication_gb300 import hierarchical, sharded
    bc.lib()
    torch.cuda.set_device(0)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=T.L * T.G)
    local_groups = [dist.new_group([g * T.L + l for l in range(T.L)]) for g in range(T.G)]
    inter_group = dist.new_group([g * T.L for g in range(T.G)])
    node, lrank = divmod(rank, T.L)
    local = sharded.Exchange(local_groups[node], host_staging=True)
    inter = sharded.Exchange(inter_group, host_staging=True) if lrank == 0 else None
    pa = hierarchical.PipelineA(T.N, torch.float32, local, inter,
                                bc.QParams(T.BITS, T.B1, T.ROUNDING, seed=500 + node),
                                bc.QParams(T.BITS, T.B2, T.ROUNDING, seed=77, philox_stream=1),
                                chunk_size=T.CHUNK, local_quantize=local_quantize,
                                p_local=bc.QParams(T.BITS, T.BL, T.ROUNDING, seed=900 + rank), device="cuda:0")
    for step in range(T.STEPS):
        out = torch.empty(T.N, device="cuda:0")
        pa(torch.from_numpy(T._grad(rank, step)).cuda(), out, mul=1.0 / (T.L * T.G))
        torch.cuda.synchronize()
        np.save(os.path.join(outdir, f"out{step}_{rank}.npy"), out.cpu().numpy())
    if pa.err_local is not None:
        np.save(os.path.join(outdir, f"elocal{rank}.npy"), pa.err_local.cpu().numpy())
    if pa.ar is not None:
        np.save(os.path.join(outdir, f"einter{node}.npy"), pa.ar.err.cpu().numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("local_quantize", [False, True])
def test_pipeline_a_on_libbitscom_equals_oracle_restatement(orc, tmp_path, local_quantize):
    torch, bc = need_gpu()
    import torch.multiprocessing as mp

    import test_gloo_hierarchical as T
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, str(tmp_path), local_quantize)) for r in range(T.L * T.G)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    outs, e_local, e_inter, _ = T._restate(orc, local_quantize)
    for step in range(T.STEPS):
        for r in range(T.L * T.G):
            got = np.load(tmp_path / f"out{step}_{r}.npy")
            assert np.array_equal(got.view(np.uint32), outs[step].view(np.uint32)), (step, r)
    if local_quantize:
        for r in range(T.L * T.G):
            assert np.array_equal(np.load(tmp_path / f"elocal{r}.npy").view(np.uint32), e_local[r].view(np.uint32))
    for node in range(T.G):
        assert np.array_equal(np.load(tmp_path / f"einter{node}.npy").view(np.uint32), e_inter[node].view(np.uint32))
