"""Host-side partition of the multi-rank all-reduce (no GPU).

The buckets of bit_gradient_communication_gb300.sharded.plan must be those
of the C bucket scheduler (bitscom_sched_plan, with the chunk unit max(B1, B2)
as its block), and its chunks must tile every bucket with whole units in rank
order, ceil(units / W) units each (the rule the simulated all-reduce applies).
"""
import ctypes

import pytest

from bit_gradient_communication_gb300 import sharded


@pytest.fixture(scope="module")
def bc():
    from bit_gradient_communication_gb300 import _build
    _build.build()
    import bit_gradient_communication_gb300 as bc
    bc.lib()
    return bc


CASES = [(1, 4, 128, 128, 2, 0), (4096 * 3 + 640, 4, 128, 128, 3, 16 * 1024), (10 ** 6 + 17, 2, 64, 64, 8, 1 << 20),
         (5000, 4, 8, 8, 64, 1024), (1 << 20, 2, 512, 128, 8, 25 * 1024 * 1024), (123457, 4, 4096, 32, 5, 1 << 16),
         (0, 4, 128, 128, 4, 1 << 20), (640, 4, 128, 128, 8, 0)]


@pytest.mark.parametrize("n,esz,B1,B2,W,bucket_bytes", CASES)
def test_buckets_are_the_schedulers(bc, n, esz, B1, B2, W, bucket_bytes):
    U = max(B1, B2)
    count = bc.lib().bitscom_sched_plan(n, esz, U, bucket_bytes, None, 0)
    starts = (ctypes.c_int64 * (count + 1))()
    bc.lib().bitscom_sched_plan(n, esz, U, bucket_bytes, starts, count)
    buckets = sharded.plan(n, esz, B1, B2, W, bucket_bytes)
    if n == 0:
        assert count == 0
        return
    assert [bk.b0 for bk in buckets] + [n] == list(starts)
    assert [bk.n for bk in buckets] == [starts[k + 1] - starts[k] for k in range(count)]


@pytest.mark.parametrize("n,esz,B1,B2,W,bucket_bytes", CASES)
def test_chunks_tile_each_bucket_in_rank_order(n, esz, B1, B2, W, bucket_bytes):
    U = max(B1, B2)
    for bk in sharded.plan(n, esz, B1, B2, W, bucket_bytes):
        assert len(bk.chunks) == W
        units = -(-bk.n // U)
        cu = -(-units // W)
        at = bk.b0
        for c, (lo, hi) in enumerate(bk.chunks):
            if lo == hi:
                assert c * cu >= units and lo == bk.b0 + bk.n
                continue
            assert lo == at and (lo - bk.b0) == c * cu * U
            assert hi - lo == min(cu * U, bk.n - (lo - bk.b0))
            at = hi
        assert at == bk.b0 + bk.n


def test_chunk_byte_counts():
    # codes of [lo, hi) start on a block boundary and cover whole blocks
    assert sharded.code_bytes(0, 0, 4, 128) == 0
    assert sharded.code_bytes(128, 256, 4, 128) == 64
    assert sharded.code_bytes(128, 257, 4, 128) == 128
    assert sharded.code_bytes(0, 1, 16, 8) == 16
    assert sharded.scale_count(128, 257, 128) == 2
    assert sharded.scale_count(5, 5, 128) == 0
